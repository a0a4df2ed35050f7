// One-token step in a single cooperative kernel: routing, gate/up + SwiGLU, down and the
// gate-weighted combine into the residual.
//
// "DwarfStar" README, "运行大于 RAM 的模型": every new token is routed through the experts
// again, so each decode step streams the selected experts' packed rows once. At one token the
// step is a pure stream of bytes, so the kernel is built to keep HBM busy:
//   * every CTA (one per SM) routes the token itself -- top-k of the router logits, ties to the
//     lower index -- so no launch or barrier separates routing from the experts;
//   * one producer warp streams weight rows into a 3-stage shared-memory ring with 1-D TMA
//     bulk copies (up to ~110 KB in flight per SM), sixteen compute warps decode from shared
//     memory; the phase-2 (down) rows are fetched before the grid barrier that waits for h;
//   * dot products of packed rows are exact integer sums: x (per 2048 columns) and h (per
//     routed pair) are held as int16 with a power-of-two scale (2^14 over the absolute
//     maximum: error ~2^-15 of that maximum), IQ2-style groups become signed int8 vectors
//     (grid magnitudes, signs applied through a 128-entry table of byte masks) and Q2_K-style
//     codes become int8 bytes through a 256-entry table; dp2a accumulates int16 x int8 pairs
//     into int32 without rounding, and each 16- or 32-weight sub-block's integer sum is
//     scaled into fp32 once; the bf16 shared expert runs in fp32;
//   * the down phase owns whole output rows, so each row's 8 routed contributions and the
//     shared one are summed in a fixed order and added to the residual once: deterministic.
// Every wait is bounded (~2 s): a timeout sets DS4MOE_ETIMEOUT in the status word and the CTA
// finishes without waiting further. The kernel is launched cooperatively, so all CTAs are
// resident together when they meet at the grid barrier.
#include <cuda_runtime.h>

#include <cfloat>
#include <climits>

#include "common.cuh"
#include "ptx.cuh"

namespace ds4moe {
namespace {

constexpr int kCompute = 16;                   // compute warps
constexpr int kThreads = (kCompute + 1) * 32;  // + one producer warp
constexpr int kStages = 3;
constexpr int kStageBytes = 38912;
constexpr int kTabEntries = 256 * 16;  // lookup table replicated per half-warp lane
constexpr int kSignEntries = 128 * 8;  // sign masks, replicated per quarter-warp lane (16-byte reads)
constexpr int kActBytes = 44 * 1024;
constexpr int kRows2 = 4;  // output rows per down-phase unit

// Swizzled 16-byte chunk index: lanes reading 64 or 128 contiguous bytes each hit distinct banks.
__device__ __forceinline__ int swz(int q) { return q ^ ((q >> 3) & 7); }

__device__ __forceinline__ uint64_t now_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void named_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kCompute * 32) : "memory"); }

// Barrier of the 4 warps that share output row r of a down-phase unit (ids 2..5).
__device__ __forceinline__ void row_sync(int r) { asm volatile("bar.sync %0, 128;" ::"r"(2 + r) : "memory"); }

struct StepParams {
    DeviceWeights w;
    const uint16_t *x;     // bf16 [D]
    const float *logits;   // [E]
    float *out;            // [D], += delta
    int k, mode;
    const uint8_t *grid;   // grid magnitudes [256][8]
    int32_t *topk_idx;     // [k] (written by CTA 0)
    float *topk_w;         // [k]
    float *h;              // [k+1][F] fp32, row k = shared expert
    unsigned *bar;         // grid barrier: count, generation
    float *hmax;           // [gridDim][8] per-CTA max |h| of each routed pair
    uint64_t *trace;       // null, or [gridDim][6] timestamps (ns)
    int *status;
    int r1, rs;            // rows per phase-1 routed / shared unit
};

// Geometry of the units of one call, identical in every CTA.
struct Units {
    int per1;   // routed units per expert (F / r1)
    int n1r;    // routed phase-1 units
    int n1;     // all phase-1 units
    int n2;     // phase-2 units (D / kRows2)
};

__device__ __forceinline__ Units units_of(const StepParams &p) {
    Units u;
    u.per1 = p.w.F / p.r1;
    u.n1r = p.k * u.per1;
    u.n1 = u.n1r + (p.w.has_shared ? p.w.F / p.rs : 0);
    u.n2 = p.w.D / kRows2;
    return u;
}

// Issues the bulk copies of one unit into a stage (one thread).
__device__ void issue_unit(const StepParams &p, const Units &U, const int *idx, int phase, int unit, uint32_t dst,
                           uint32_t bar) {
    const DeviceWeights &w = p.w;
    if (phase == 1) {
        if (unit < U.n1r) {
            const int e = idx[unit / U.per1];
            const int row0 = (unit % U.per1) * p.r1;
            const size_t rb = (static_cast<size_t>(e) * w.F + row0) * w.nbD;  // first block
            const uint32_t qs = static_cast<uint32_t>(p.r1 * w.nbD * 64), ds = static_cast<uint32_t>(p.r1 * w.nbD * 2);
            mbar_expect_tx(bar, 2 * qs + 2 * ds);
            bulk_load(dst, w.gate_qs + rb * 64, qs, bar);
            bulk_load(dst + qs, w.up_qs + rb * 64, qs, bar);
            bulk_load(dst + 2 * qs, w.gate_d + rb, ds, bar);
            bulk_load(dst + 2 * qs + ds, w.up_d + rb, ds, bar);
        } else {
            const int row0 = (unit - U.n1r) * p.rs;
            const uint32_t b = static_cast<uint32_t>(p.rs * w.D * 2);
            mbar_expect_tx(bar, 2 * b);
            bulk_load(dst, w.sh_gate + static_cast<size_t>(row0) * w.D, b, bar);
            bulk_load(dst + b, w.sh_up + static_cast<size_t>(row0) * w.D, b, bar);
        }
    } else {
        const int d0 = unit * kRows2;
        const uint32_t sqb = static_cast<uint32_t>(kRows2 * w.nbF * 80), ddb = static_cast<uint32_t>(kRows2 * w.nbF * 4);
        const uint32_t shb = w.has_shared ? static_cast<uint32_t>(kRows2 * w.F * 2) : 0u;
        mbar_expect_tx(bar, p.k * (sqb + ddb) + shb);
        for (int s = 0; s < p.k; s++) {
            const size_t rb = (static_cast<size_t>(idx[s]) * w.D + d0) * w.nbF;
            bulk_load(dst + s * sqb, w.down_sq + rb * 80, sqb, bar);
            bulk_load(dst + p.k * sqb + s * ddb, w.down_dd + rb, ddb, bar);
        }
        if (w.has_shared) bulk_load(dst + p.k * (sqb + ddb), w.sh_down + static_cast<size_t>(d0) * w.F, shb, bar);
    }
}

// One group of 8 IQ2-style weights dotted with 8 int16 x (4 registers of pairs), exactly:
// grid magnitudes (int8 x 8) with the group's signs applied through the sign masks.
__device__ __forceinline__ int iq2_group_idot(uint2 mag, uint4 sm, const uint32_t *xv, int acc) {
    const int lo = static_cast<int>((mag.x ^ sm.x) + sm.z);
    const int hi = static_cast<int>((mag.y ^ sm.y) + sm.w);
    acc = __dp2a_lo(static_cast<int>(xv[0]), lo, acc);
    acc = __dp2a_hi(static_cast<int>(xv[1]), lo, acc);
    acc = __dp2a_lo(static_cast<int>(xv[2]), hi, acc);
    acc = __dp2a_hi(static_cast<int>(xv[3]), hi, acc);
    return acc;
}

// Bounded grid barrier, one thread per CTA. Generation counting: the barrier words never need
// resetting between calls.
__device__ bool grid_barrier(unsigned *bar, int *status) {
    volatile unsigned *gen = bar + 1;
    const unsigned g = *gen;
    __threadfence();
    const unsigned ticket = atomicAdd(bar, 1u);
    if (ticket == gridDim.x - 1) {
        atomicExch(bar, 0u);
        __threadfence();
        atomicAdd(bar + 1, 1u);
        return true;
    }
    const long long t0 = clock64();
    while (*gen == g) {
        if (clock64() - t0 > kWaitCycles) {
            report(status, ST_TIMEOUT);
            return false;
        }
        __nanosleep(64);
    }
    __threadfence();
    return true;
}

__global__ void __launch_bounds__(kThreads, 1) decode_step_kernel(StepParams p) {
    extern __shared__ uint8_t smem_raw[];
    // align by an integer offset so that every pointer below stays a shared-memory pointer
    uint8_t *smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
    uint8_t *ring = smem;                                                     // kStages x kStageBytes
    uint2 *tab = reinterpret_cast<uint2 *>(smem + kStages * kStageBytes);    // [256][16]
    uint4 *stab = reinterpret_cast<uint4 *>(smem + kStages * kStageBytes + kTabEntries * 8);  // [128][8]
    uint8_t *act = smem + kStages * kStageBytes + kTabEntries * 8 + kSignEntries * 16;        // kActBytes
    uint64_t *bars = reinterpret_cast<uint64_t *>(act + kActBytes);          // full[S], empty[S]
    int *sidx = reinterpret_cast<int *>(bars + 2 * kStages);                 // [8]
    float *sgw = reinterpret_cast<float *>(sidx + 8);                         // [8]
    float *scal = sgw + 8;                                                    // [8] x scales / [9] h scales
    float *red = scal + 16;                                                   // [8 warps][16]
    volatile int *abort_flag = reinterpret_cast<volatile int *>(red + kCompute * 16);
    unsigned *hmax_cta = reinterpret_cast<unsigned *>(red + kCompute * 16 + 4);  // [8] max |h| per pair, this CTA

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const DeviceWeights &w = p.w;
    const int D = w.D, F = w.F, nbD = w.nbD, nbF = w.nbF;
    const Units U = units_of(p);
    const int nph = (D + 2047) / 2048;  // x phases of 2048 columns
    uint64_t *tr = (p.trace && threadIdx.x == 0) ? p.trace + 6 * static_cast<size_t>(blockIdx.x) : nullptr;
    if (tr) tr[0] = now_ns();

    // ---------------------------------------------------------------- prologue
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; s++) {
            mbar_init(smem_u32(bars + s), 1);
            mbar_init(smem_u32(bars + kStages + s), kCompute);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {  // route: top-k of the logits, ties to the lower expert index
        const int E = w.E;
        float key[32];  // lane holds experts lane, lane+32, ... (E <= 1024)
#pragma unroll
        for (int j = 0; j < 32; j++) {
            const int e = lane + 32 * j;
            float v = (e < E) ? __ldg(p.logits + e) : -INFINITY;
            key[j] = (v != v) ? -INFINITY : v;
        }
        uint32_t taken = 0;
        float my_v = -INFINITY;
        int my_i = 0;
        for (int r = 0; r < p.k; r++) {
            float bv = -INFINITY;
            int bi = INT_MAX;
#pragma unroll
            for (int j = 0; j < 32; j++) {
                const int e = lane + 32 * j;
                if (e < E && !((taken >> j) & 1u) && (key[j] > bv || (key[j] == bv && e < bi))) {
                    bv = key[j];
                    bi = e;
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                if (ov > bv || (ov == bv && oi < bi)) {
                    bv = ov;
                    bi = oi;
                }
            }
            if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
            if (lane == r) {
                my_v = bv;
                my_i = bi;
            }
        }
        const float top = __shfl_sync(0xffffffffu, my_v, 0);
        float num = 0.0f;
        if (lane < p.k) num = (p.mode == DS4MOE_GATE_SOFTMAX) ? expf(my_v - top) : 1.0f / (1.0f + expf(-my_v));
        const float den = warp_sum(num);
        if (lane < p.k) {
            sidx[lane] = my_i;
            sgw[lane] = num / den;
            if (blockIdx.x == 0) {
                p.topk_idx[lane] = my_i;
                p.topk_w[lane] = num / den;
            }
        }
    }
    // x: per 2048-column phase, a power-of-two scale and the fp16 values (swizzled chunks)
    if (warp < kCompute) {
        uint16_t *x16 = reinterpret_cast<uint16_t *>(act);
        unsigned *xmax = reinterpret_cast<unsigned *>(scal);
        if (threadIdx.x < 16) xmax[threadIdx.x] = 0u;
        if (threadIdx.x < 8) hmax_cta[threadIdx.x] = 0u;
        named_sync();
        constexpr int kXq = 2;  // 16-byte chunks of x per thread (D <= 8192)
        uint4 xr[kXq];
#pragma unroll
        for (int j = 0; j < kXq; j++) {
            const int q = threadIdx.x + j * kCompute * 32;
            xr[j] = q < D / 8 ? __ldg(reinterpret_cast<const uint4 *>(p.x) + q) : make_uint4(0, 0, 0, 0);
            const uint32_t u4[4] = {xr[j].x, xr[j].y, xr[j].z, xr[j].w};
            float m = 0.0f;
#pragma unroll
            for (int i = 0; i < 4; i++) m = fmaxf(m, fmaxf(fabsf(bf16_lo(u4[i])), fabsf(bf16_hi(u4[i]))));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));  // a warp's 32 chunks share one phase
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
            if (lane == 0 && q < D / 8) atomicMax(xmax + q / 256, __float_as_uint(m));
        }
        named_sync();
        if (threadIdx.x < nph) {
            const float m = __uint_as_float(xmax[threadIdx.x]);
            int e = 0;
            frexpf(m, &e);
            e = m > 0.0f ? e : 0;
            scal[threadIdx.x] = ldexpf(1.0f, e);  // 1/scale, multiplies results back
        }
        named_sync();
#pragma unroll
        for (int j = 0; j < kXq; j++) {  // 16-byte chunks -> int16 with the phase's scale 2^(14-e)
            const int q = threadIdx.x + j * kCompute * 32;
            if (q >= D / 8) continue;
            const float sc = 16384.0f / scal[q / 256];
            const uint32_t u4[4] = {xr[j].x, xr[j].y, xr[j].z, xr[j].w};
            uint32_t o[4];
#pragma unroll
            for (int i = 0; i < 4; i++)
                o[i] = (static_cast<uint32_t>(__float2int_rn(bf16_lo(u4[i]) * sc)) & 0xffffu) |
                       (static_cast<uint32_t>(__float2int_rn(bf16_hi(u4[i]) * sc)) << 16);
            reinterpret_cast<uint4 *>(x16)[swz(q)] = make_uint4(o[0], o[1], o[2], o[3]);
        }
        for (int i = threadIdx.x; i < kTabEntries; i += kCompute * 32)  // grid magnitudes (int8)
            tab[i] = __ldg(reinterpret_cast<const uint2 *>(p.grid) + (i >> 4));
        for (int i = threadIdx.x; i < kSignEntries; i += kCompute * 32) {
            // 7 stored signs + parity -> byte masks M (0xFF where negative) and B = M & 0x01:
            // (magnitudes ^ M) + B negates the marked bytes (no carry: magnitudes are <= 7)
            const uint32_t s7 = static_cast<uint32_t>(i >> 3);
            const uint32_t s8 = s7 | ((__popc(s7) & 1u) << 7);
            uint32_t m[2];
#pragma unroll
            for (int h2 = 0; h2 < 2; h2++) {
                uint32_t v = 0;
#pragma unroll
                for (int b = 0; b < 4; b++) v |= ((s8 >> (4 * h2 + b)) & 1u) ? (0xFFu << (8 * b)) : 0u;
                m[h2] = v;
            }
            stab[i] = make_uint4(m[0], m[1], m[0] & 0x01010101u, m[1] & 0x01010101u);
        }
    }
    __syncthreads();
    if (tr) tr[1] = now_ns();

    if (warp == kCompute) {
        // ---------------------------------------------------------------- producer
        if (lane == 0) {
            int stage = 0, issued_parity[kStages];
            uint32_t phase = 0;
            for (int s = 0; s < kStages; s++) issued_parity[s] = -1;
            bool ok = true;
            for (int ph = 1; ph <= 2 && ok; ph++) {
                const int n = ph == 1 ? U.n1 : U.n2;
                for (int u = blockIdx.x; u < n; u += gridDim.x) {
                    if (!mbar_wait(smem_u32(bars + kStages + stage), phase ^ 1u, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    issue_unit(p, U, sidx, ph, u, smem_u32(ring + stage * kStageBytes), smem_u32(bars + stage));
                    issued_parity[stage] = static_cast<int>(phase);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok)
                for (int s = 0; s < kStages; s++)
                    if (issued_parity[s] >= 0) mbar_drain(smem_u32(bars + s), static_cast<uint32_t>(issued_parity[s]));
        }
        return;  // the producer takes no part in the compute warps' barriers
    }

    // -------------------------------------------------------------------- compute warps
    const uint2 *gt = tab + (lane & 15);
    const uint4 *st8 = stab + (lane & 7);
    const uint4 *x16v = reinterpret_cast<const uint4 *>(act);
    int stage = 0;
    uint32_t sphase = 0;
    bool ok = true;
    auto next_stage = [&]() -> const uint8_t * {
        if (!ok || !mbar_wait(smem_u32(bars + stage), sphase, abort_flag, p.status)) {
            ok = false;
            return nullptr;
        }
        return ring + stage * kStageBytes;
    };
    auto release_stage = [&]() {
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(bars + kStages + stage));
        if (++stage == kStages) {
            stage = 0;
            sphase ^= 1u;
        }
    };

    // ---------------------------------------------------------------- phase 1: gate/up, SwiGLU
    const int nchunk = nbD * 4;  // 64-column chunks per row
    for (int u = blockIdx.x; u < U.n1 && ok; u += gridDim.x) {
        const uint8_t *st = next_stage();
        if (!st) break;
        if (u < U.n1r) {
            const int slot = u / U.per1, row0 = (u % U.per1) * p.r1;
            const int wpr = kCompute / p.r1;                      // warps per row (1 or 2)
            const int rl = warp % p.r1, psub = warp / p.r1;       // local row, phase subset
            const uint8_t *gq = st, *uq = st + p.r1 * nbD * 64;
            const uint16_t *gd = reinterpret_cast<const uint16_t *>(st + 2 * p.r1 * nbD * 64);
            const uint16_t *ud = gd + p.r1 * nbD;
            float ag = 0.0f, au = 0.0f;
            for (int ph = psub; ph < nph; ph += wpr) {
                const int c = ph * 32 + lane;
                if (c >= nchunk) continue;
                uint32_t xh[32];
#pragma unroll
                for (int j = 0; j < 8; j++) {
                    const uint4 v = x16v[swz(8 * c + j)];
                    xh[4 * j] = v.x;
                    xh[4 * j + 1] = v.y;
                    xh[4 * j + 2] = v.z;
                    xh[4 * j + 3] = v.w;
                }
                const float xinv = scal[ph] * (1.0f / 16384.0f);
                const uint4 qg = *reinterpret_cast<const uint4 *>(gq + (rl * nbD * 4 + c) * 16);
                const uint4 qu = *reinterpret_cast<const uint4 *>(uq + (rl * nbD * 4 + c) * 16);
                const float dg = f16_to_f32(gd[rl * nbD + (c >> 2)]) * xinv;
                const float du = f16_to_f32(ud[rl * nbD + (c >> 2)]) * xinv;
#pragma unroll
                for (int sb = 0; sb < 2; sb++) {
                    const uint32_t igw = sb ? qg.z : qg.x, sgw2 = sb ? qg.w : qg.y;
                    const uint32_t iuw = sb ? qu.z : qu.x, suw = sb ? qu.w : qu.y;
                    int g0 = 0, g1 = 0, u0 = 0, u1 = 0;  // two accumulators per matrix: shorter chains
#pragma unroll
                    for (int g = 0; g < 4; g += 2) {
                        const uint32_t *xv0 = xh + 16 * sb + 4 * g, *xv1 = xv0 + 4;
                        g0 = iq2_group_idot(gt[((igw >> (8 * g)) & 255u) << 4], st8[((sgw2 >> (7 * g)) & 127u) << 3], xv0, g0);
                        u0 = iq2_group_idot(gt[((iuw >> (8 * g)) & 255u) << 4], st8[((suw >> (7 * g)) & 127u) << 3], xv0, u0);
                        g1 = iq2_group_idot(gt[((igw >> (8 * g + 8)) & 255u) << 4], st8[((sgw2 >> (7 * g + 7)) & 127u) << 3], xv1, g1);
                        u1 = iq2_group_idot(gt[((iuw >> (8 * g + 8)) & 255u) << 4], st8[((suw >> (7 * g + 7)) & 127u) << 3], xv1, u1);
                    }
                    ag = fmaf(iq2_scale(dg, sgw2), static_cast<float>(g0 + g1), ag);
                    au = fmaf(iq2_scale(du, suw), static_cast<float>(u0 + u1), au);
                }
            }
            float g = warp_sum(ag), uu = warp_sum(au);
            release_stage();
            if (wpr > 1) {  // the second warp of a row hands its partial sums over
                if (lane == 0 && psub > 0) {
                    red[warp * 16] = g;
                    red[warp * 16 + 1] = uu;
                }
                named_sync();
                if (psub == 0)
                    for (int o = 1; o < wpr; o++) {
                        g += red[(warp + o * p.r1) * 16];
                        uu += red[(warp + o * p.r1) * 16 + 1];
                    }
                named_sync();
            }
            if (lane == 0 && psub == 0) {
                const float hv = swiglu(g, uu);
                p.h[static_cast<size_t>(slot) * F + row0 + rl] = hv;
                atomicMax(hmax_cta + slot, __float_as_uint(fabsf(hv)));
            }
        } else {
            // shared expert: rs bf16 rows of gate and up; threads split the 16-byte chunks
            const int row0 = (u - U.n1r) * p.rs;
            const uint4 *sg = reinterpret_cast<const uint4 *>(st);
            const uint4 *su = reinterpret_cast<const uint4 *>(st + p.rs * D * 2);
            const int tid = warp * 32 + lane, nq = D / 8;
            float pg[8], pu[8];
#pragma unroll
            for (int r = 0; r < 8; r++) pg[r] = pu[r] = 0.0f;
            for (int q = tid; q < nq; q += kCompute * 32) {
                const uint4 xv = x16v[swz(q)];
                const float xi = scal[q / 256] * (1.0f / 16384.0f);
                const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
                float xf[8];
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    xf[2 * i] = static_cast<float>(static_cast<int16_t>(xw[i] & 0xffffu)) * xi;
                    xf[2 * i + 1] = static_cast<float>(static_cast<int16_t>(xw[i] >> 16)) * xi;
                }
#pragma unroll
                for (int r = 0; r < 8; r++) {
                    if (r < p.rs) {
                        const uint4 gv = sg[r * nq + q], uv = su[r * nq + q];
                        const uint32_t g4[4] = {gv.x, gv.y, gv.z, gv.w}, u4[4] = {uv.x, uv.y, uv.z, uv.w};
#pragma unroll
                        for (int i = 0; i < 4; i++) {
                            pg[r] = fmaf(bf16_lo(g4[i]), xf[2 * i], pg[r]);
                            pg[r] = fmaf(bf16_hi(g4[i]), xf[2 * i + 1], pg[r]);
                            pu[r] = fmaf(bf16_lo(u4[i]), xf[2 * i], pu[r]);
                            pu[r] = fmaf(bf16_hi(u4[i]), xf[2 * i + 1], pu[r]);
                        }
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < 8; r++) {
                if (r < p.rs) {
                    const float g = warp_sum(pg[r]), uu = warp_sum(pu[r]);
                    if (lane == 0) {
                        red[warp * 16 + 2 * r] = g;
                        red[warp * 16 + 2 * r + 1] = uu;
                    }
                }
            }
            release_stage();
            named_sync();
            if (warp == 0 && lane < p.rs) {
                float g = 0.0f, uu = 0.0f;
                for (int ww = 0; ww < kCompute; ww++) {
                    g += red[ww * 16 + 2 * lane];
                    uu += red[ww * 16 + 2 * lane + 1];
                }
                p.h[static_cast<size_t>(p.k) * F + row0 + lane] = swiglu(g, uu);
            }
            named_sync();
        }
    }

    // ---------------------------------------------------------------- grid barrier: all h written
    named_sync();
    if (tr) tr[2] = now_ns();
    uint32_t *ctab = reinterpret_cast<uint32_t *>(tab);  // code byte -> its four codes as int8 [256][16]
    for (int i = threadIdx.x; i < kTabEntries; i += kCompute * 32) {
        const uint32_t b = static_cast<uint32_t>(i >> 4);
        ctab[i] = (b & 3u) | (((b >> 2) & 3u) << 8) | (((b >> 4) & 3u) << 16) | (((b >> 6) & 3u) << 24);
    }
    if (threadIdx.x < p.k) p.hmax[static_cast<size_t>(blockIdx.x) * 8 + threadIdx.x] = __uint_as_float(hmax_cta[threadIdx.x]);
    named_sync();
    if (threadIdx.x == 0 && !grid_barrier(p.bar, p.status)) *abort_flag = 1;
    named_sync();
    if (tr) tr[3] = now_ns();

    // h for the down phase: per routed pair a power-of-two scale (from the CTAs' maxima), fp16
    // values (swizzled chunks) and the fp32 sums of its 16-column sub-blocks; the shared
    // expert's h stays fp32
    uint16_t *h16 = reinterpret_cast<uint16_t *>(act);           // [k][F]
    float *hsum = reinterpret_cast<float *>(act + p.k * F * 2);  // [k][F/16]
    float *hsh = hsum + p.k * (F / 16);                          // [F]
    {
        const int tid = threadIdx.x;
        if (warp < p.k) {  // warp s reduces pair s over the CTAs
            float m = 0.0f;
            for (int c = lane; c < static_cast<int>(gridDim.x); c += 32)
                m = fmaxf(m, __ldcg(p.hmax + static_cast<size_t>(c) * 8 + warp));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
            int e = 0;
            frexpf(m, &e);
            e = m > 0.0f ? e : 0;
            if (lane == 0) scal[warp] = ldexpf(1.0f, e);
        }
        named_sync();
        for (int sb = tid; sb < p.k * F / 16; sb += kCompute * 32) {  // one 16-column sub-block
            const float sc = 16384.0f / scal[sb / (F / 16)];
            const float4 *src = reinterpret_cast<const float4 *>(p.h) + 4 * sb;
            const float4 a = __ldcg(src), b = __ldcg(src + 1), c = __ldcg(src + 2), d = __ldcg(src + 3);
            auto pk = [sc](float x0, float x1) {
                return (static_cast<uint32_t>(__float2int_rn(x0 * sc)) & 0xffffu) |
                       (static_cast<uint32_t>(__float2int_rn(x1 * sc)) << 16);
            };
            uint4 o0, o1;
            o0.x = pk(a.x, a.y);
            o0.y = pk(a.z, a.w);
            o0.z = pk(b.x, b.y);
            o0.w = pk(b.z, b.w);
            o1.x = pk(c.x, c.y);
            o1.y = pk(c.z, c.w);
            o1.z = pk(d.x, d.y);
            o1.w = pk(d.z, d.w);
            reinterpret_cast<uint4 *>(h16)[swz(2 * sb)] = o0;
            reinterpret_cast<uint4 *>(h16)[swz(2 * sb + 1)] = o1;
            hsum[sb] = ((a.x + a.y) + (a.z + a.w)) + ((b.x + b.y) + (b.z + b.w)) + ((c.x + c.y) + (c.z + c.w)) +
                       ((d.x + d.y) + (d.z + d.w));
        }
        if (w.has_shared)
            for (int q = tid; q < F / 4; q += kCompute * 32)
                reinterpret_cast<float4 *>(hsh)[q] = __ldcg(reinterpret_cast<const float4 *>(p.h + static_cast<size_t>(p.k) * F) + q);
        named_sync();
    }
    if (tr) tr[4] = now_ns();

    // ---------------------------------------------------------------- phase 2: down + combine
    const uint4 *h16v = reinterpret_cast<const uint4 *>(h16);
    const int rl2 = warp >> 2;              // local output row of this warp
    const int qt = warp & 3;                // which quarter of F
    const int col = qt * (F / 4) + lane * 16;  // this lane's 16 columns: one sub-block
    const int b2 = col >> 8, part64 = (col >> 6) & 3, sub = (col >> 4) & 3;
    for (int u = blockIdx.x; u < U.n2 && ok; u += gridDim.x) {
        const uint8_t *st = next_stage();
        if (!st) break;
        const int sqb = kRows2 * nbF * 80, ddb = kRows2 * nbF * 4;
        float acc = 0.0f;
        for (int s = 0; s < p.k; s++) {
            const uint8_t *blk = st + s * sqb + (rl2 * nbF + b2) * 80;
            const uint32_t qw = *reinterpret_cast<const uint32_t *>(blk + 16 + 16 * part64 + 4 * sub);
            const uint32_t scb = blk[4 * part64 + sub];
            const uint32_t ddw = *reinterpret_cast<const uint32_t *>(st + p.k * sqb + s * ddb + (rl2 * nbF + b2) * 4);
            const uint4 h0 = h16v[swz((s * F + col) / 8)], h1 = h16v[swz((s * F + col) / 8 + 1)];
            const uint32_t hh[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
            const uint32_t *ct = reinterpret_cast<const uint32_t *>(tab) + (lane & 15);
            int a0 = 0, a1 = 0;
#pragma unroll
            for (int bb = 0; bb < 4; bb += 2) {
                const int c0 = static_cast<int>(ct[((qw >> (8 * bb)) & 255u) << 4]);
                const int c1 = static_cast<int>(ct[((qw >> (8 * bb + 8)) & 255u) << 4]);
                a0 = __dp2a_lo(static_cast<int>(hh[2 * bb]), c0, a0);
                a1 = __dp2a_lo(static_cast<int>(hh[2 * bb + 2]), c1, a1);
                a0 = __dp2a_hi(static_cast<int>(hh[2 * bb + 1]), c0, a0);
                a1 = __dp2a_hi(static_cast<int>(hh[2 * bb + 3]), c1, a1);
            }
            const float d = f16_to_f32(static_cast<uint16_t>(ddw & 0xffffu));
            const float dmin = f16_to_f32(static_cast<uint16_t>(ddw >> 16));
            float part = d * static_cast<float>(scb & 15u) * (scal[s] * (1.0f / 16384.0f)) * static_cast<float>(a0 + a1);
            part = fmaf(-dmin * static_cast<float>(scb >> 4), hsum[s * (F / 16) + (col >> 4)], part);
            acc = fmaf(sgw[s], part, acc);
        }
        if (w.has_shared) {  // this quarter of the row: lanes take interleaved 16-byte chunks
            const uint4 *row = reinterpret_cast<const uint4 *>(st + p.k * (sqb + ddb) + rl2 * F * 2);
            const float4 *hv = reinterpret_cast<const float4 *>(hsh);
            for (int q = qt * (F / 32) + lane; q < (qt + 1) * (F / 32); q += 32) {
                const uint4 v = row[q];
                const float4 x0 = hv[2 * q], x1 = hv[2 * q + 1];
                acc = fmaf(bf16_lo(v.x), x0.x, acc);
                acc = fmaf(bf16_hi(v.x), x0.y, acc);
                acc = fmaf(bf16_lo(v.y), x0.z, acc);
                acc = fmaf(bf16_hi(v.y), x0.w, acc);
                acc = fmaf(bf16_lo(v.z), x1.x, acc);
                acc = fmaf(bf16_hi(v.z), x1.y, acc);
                acc = fmaf(bf16_lo(v.w), x1.z, acc);
                acc = fmaf(bf16_hi(v.w), x1.w, acc);
            }
        }
        acc = warp_sum(acc);
        // the four warps of this output row meet on the row's own barrier; parity-alternating
        // slots let the next unit's partials be written while this one is still read
        float *slot = red + ((u / gridDim.x) & 1) * 64;
        if (lane == 0) slot[warp * 4] = acc;
        release_stage();
        row_sync(rl2);
        if (qt == 0 && lane == 0) {
            const int d = u * kRows2 + rl2;
            p.out[d] += (slot[(4 * rl2) * 4] + slot[(4 * rl2 + 1) * 4]) + (slot[(4 * rl2 + 2) * 4] + slot[(4 * rl2 + 3) * 4]);
        }
    }
    if (tr) tr[5] = now_ns();
}

int n_sms() {
    static int n = 0;
    if (!n) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 148;
    }
    return n;
}

}  // namespace

// Whether the fused single-token kernel covers this shape.
int decode_step_ctas() { return n_sms(); }

bool decode_step_supported(const DeviceWeights &w, int k) {
    if (k < 1 || k > 8 || w.F != 2048 || w.D > 8192) return false;
    const int r1 = (static_cast<size_t>(16) * w.nbD * 132 <= kStageBytes) ? 16 : 8;
    if (static_cast<size_t>(r1) * w.nbD * 132 > kStageBytes) return false;
    if (w.has_shared && static_cast<size_t>(4) * w.D > kStageBytes) return false;
    const size_t down = static_cast<size_t>(k) * kRows2 * w.nbF * 84 + (w.has_shared ? kRows2 * w.F * 2 : 0);
    if (down > kStageBytes) return false;
    const size_t act1 = static_cast<size_t>(w.D) * 2;
    const size_t act2 = static_cast<size_t>(k) * w.F * 2 + static_cast<size_t>(k) * (w.F / 16) * 4 + w.F * 4;
    return act1 <= kActBytes && act2 <= kActBytes;
}

int launch_decode_step(const DeviceWeights &w, const Workspace &ws, const uint16_t *x, const float *logits, int k,
                       int gate_mode, float *out, uint64_t *trace, void *stream) {
    static int seen[64];
    const size_t smem =
        128 + static_cast<size_t>(kStages) * kStageBytes + kTabEntries * 8 + kSignEntries * 16 + kActBytes + 2048;
    int err = ensure_smem(reinterpret_cast<const void *>(decode_step_kernel), static_cast<int>(smem), seen);
    if (err) return err;
    StepParams p;
    p.w = w;
    p.x = x;
    p.logits = logits;
    p.out = out;
    p.k = k;
    p.mode = gate_mode;
    p.grid = ws.grid;
    p.topk_idx = ws.topk_idx;
    p.topk_w = ws.topk_w;
    p.h = ws.h32;
    p.bar = ws.gbar;
    p.hmax = ws.hmax;
    p.trace = trace;
    p.status = ws.status;
    p.r1 = (static_cast<size_t>(16) * w.nbD * 132 <= kStageBytes) ? 16 : 8;
    p.rs = 1;
    while (p.rs < 8 && static_cast<size_t>(p.rs * 2) * w.D * 4 <= kStageBytes && w.F % (p.rs * 2) == 0) p.rs *= 2;
    void *args[] = {&p};
    return static_cast<int>(cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(decode_step_kernel),
                                                        dim3(n_sms()), dim3(kThreads), args, smem,
                                                        static_cast<cudaStream_t>(stream)));
}

}  // namespace ds4moe
