// Small expert groups (a few tokens per expert: decode micro-batches, and the long tail of
// prefill's routing): gate/up + SwiGLU and down on exact dp2a dot products, with every 2-bit
// weight group decoded once for all the tokens of its group.
//
// "DwarfStar" README, "运行大于 RAM 的模型": every token is routed through its experts again, so
// a batch of tokens streams the union of their experts' packed rows; with a few tokens per
// expert the stream is still bound by the per-weight decode work rather than by the tensor
// cores. Design points:
//   * x is quantised once per call (prep_x_kernel): int16 with a power-of-two scale per token,
//     stored per 8-column group as the pairs dp2a reads, plus 8 x the sum of each 32-column
//     sub-block (the offset of the nibble codes);
//   * gate/up (small_up_kernel): a unit is one 16-row tile of one expert (the tile layout of the
//     single-token kernel) for a chunk of up to kTok of its tokens; one producer warp streams
//     tiles into a ring with 1-D bulk copies, and the chunk's x into shared memory; lane l of
//     each compute warp owns row l & 15 (gate and up) and half l >> 4 of the warp's columns, so
//     a lane decodes its rows' groups with the codebook/sign table and reuses them for every
//     token of the chunk (x is read with half-warp broadcasts); a finisher warp sums the warps'
//     partial sums, applies SwiGLU and quantises the unit's 16 h values per token to int16 (one
//     16-column sub-block of the down matrix, in the order the Q2_K-style bit pairs are read);
//   * down (small_down_kernel): a unit is 8 output rows for 8 (token, expert) pairs; each pair's
//     two 4-row down tiles are one bulk copy; thread (slot, j) keeps 32 columns of its pair's h
//     in registers for all units of its slot group;
//   * units are split over the CTAs by cost (decode + tokens), contiguously, so a CTA stages
//     the x of few chunks and its neighbours in time share experts in L2;
//   * every wait is bounded (~2 s): a timeout sets DS4MOE_ETIMEOUT in the status word and the
//     warps keep their hand-shakes without computing, so every CTA finishes.
#include <cuda_runtime.h>

#include <climits>

#include "step_common.cuh"

namespace ds4moe {
namespace {

constexpr int kCompute = 16;             // compute warps
constexpr int kProducer = kCompute;      // warp index of the streamer
constexpr int kFinisher = kCompute + 1;  // warp index of the unit finisher
constexpr int kThreads = (kCompute + 2) * 32;
constexpr int kTok = 6;                  // tokens of a group handled per unit (a chunk)
constexpr int kMaxD = 4096;
constexpr int kMaxF = 2048;

// ---------------------------------------------------------------- x quantisation

// One CTA per token (256 threads, one 8-column group per thread and pass): xq[t][g] = the int16
// pairs (x0,x2), (x4,x6), (x1,x3), (x5,x7) of columns 8g..8g+7 scaled by 2^(14-e) (e: exponent of
// the token's largest |x|), x8[t][c] = 8 x the sum of the 32 int16 values of sub-block c (four
// neighbouring threads), xsc[t][0] = 2^(e-14).
__global__ void __launch_bounds__(256) prep_x_kernel(const uint16_t *__restrict__ x, int T, int D,
                                                     uint4 *__restrict__ xq, int *__restrict__ x8,
                                                     float4 *__restrict__ xsc) {
    pdl_wait();
    __shared__ float wmax[8];
    const int t = blockIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (t >= T) return;
    const uint4 *xr = reinterpret_cast<const uint4 *>(x + static_cast<size_t>(t) * D);
    const int G = D / 8;  // a multiple of 32: whole warps take part in the shuffles below
    float m = 0.0f;
    for (int g = threadIdx.x; g < G; g += 256) {
        const uint4 v = __ldg(xr + g);
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; i++) m = fmaxf(m, fmaxf(fabsf(bf16_lo(u[i])), fabsf(bf16_hi(u[i]))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) wmax[warp] = m;
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 8; i++) m = fmaxf(m, wmax[i]);
    int e = 0;
    frexpf(m, &e);
    e = m > 0.0f ? e : 0;
    const float sc = ldexpf(1.0f, 14 - e);
    uint4 *qo = xq + static_cast<size_t>(t) * G;
    for (int g = threadIdx.x; g < G; g += 256) {
        const uint4 v = __ldg(xr + g);
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
        uint32_t q[8];
#pragma unroll
        for (int i = 0; i < 4; i++) {
            q[2 * i] = round_to_int_bits(bf16_lo(u[i]) * sc);
            q[2 * i + 1] = round_to_int_bits(bf16_hi(u[i]) * sc);
        }
        int s = 0;
#pragma unroll
        for (int i = 0; i < 8; i++) s += static_cast<int>(static_cast<int16_t>(q[i] & 0xffffu));
        qo[g] = make_uint4(__byte_perm(q[0], q[2], 0x5410), __byte_perm(q[4], q[6], 0x5410),
                           __byte_perm(q[1], q[3], 0x5410), __byte_perm(q[5], q[7], 0x5410));
        s += __shfl_xor_sync(0xffffffffu, s, 1);
        s += __shfl_xor_sync(0xffffffffu, s, 2);
        if ((g & 3) == 0) x8[static_cast<size_t>(t) * (D / 32) + (g >> 2)] = 8 * s;
    }
    if (threadIdx.x == 0) xsc[t] = make_float4(ldexpf(1.0f, e - 14), 0.0f, 0.0f, 0.0f);
}

// ---------------------------------------------------------------- gate/up + SwiGLU

constexpr int kUpStages = 2;
constexpr int kUpStageBytes = kIq2TileRows * (kMaxD / 256) * 132;  // one 16-row gate/up tile
constexpr int kUpTabOff = kUpStages * kUpStageBytes;
constexpr int kXTokBytes = kMaxD * 2;                                // int16 x of one token
constexpr int kX8Tok = kMaxD / 32;                                   // sub-block sums of one token
constexpr int kUpXOff = kUpTabOff + 65536;
constexpr int kUpX8Off = kUpXOff + kTok * kXTokBytes;
constexpr int kUpXscOff = kUpX8Off + kTok * kX8Tok * 4;
constexpr int kUpRedOff = kUpXscOff + kTok * 16;
constexpr int kRedUnit = kCompute * kTok * 32;                       // floats of one unit's partial sums
constexpr int kUpMiscOff = kUpRedOff + 2 * kRedUnit * 4;
constexpr int kUpSmem = kUpMiscOff + 256;
static_assert(kUpTabOff % 256 == 0 && kUpXOff % 16 == 0 && kUpX8Off % 16 == 0 && kUpXscOff % 16 == 0,
              "table slots 256-byte aligned, bulk-copy targets 16-byte aligned");
static_assert(kUpSmem <= 232448, "shared memory of one CTA");

struct UpParams {
    DeviceWeights w;
    const int32_t *list;     // experts of the small groups, in expert order (meta->n_gemv of them)
    const int32_t *offsets;  // [E+1] first position of each expert's pairs
    const int32_t *perm;     // [P] pair id at each position
    const GroupMeta *meta;
    const uint8_t *grid;     // codebook magnitudes [256][8]
    const uint4 *xq;         // [T][D/8]
    const int *x8;           // [T][D/32]
    const float4 *xsc;       // [T]
    int16_t *hq;             // [P][F] h per position, int16, each 16-column sub-block in q2k_h_pos order
    float *hsc;              // [P][F/16] dequantisation factor of each sub-block
    float *hsum;             // [P][F/16] fp32 sum of each sub-block's h
    int k;
    int *status;
};

// Position in the unit order (small-group expert i, chunk c of its tokens, tile t) and what a
// chunk needs: expert e, its token count ne, this chunk's n tokens and first position pos0.
struct Walker {
    int i, c, t;
    int e, ne, n, pos0;
    __device__ void load(const UpParams &p, int n_list) {
        if (i >= n_list) {
            e = ne = n = pos0 = 0;
            return;
        }
        e = p.list[i];
        const int o = p.offsets[e];
        ne = p.offsets[e + 1] - o;
        n = min(kTok, ne - kTok * c);
        pos0 = o + kTok * c;
    }
    // advances by one unit; true when that starts a new chunk
    __device__ bool advance(const UpParams &p, int n_list, int nt) {
        if (++t < nt) return false;
        t = 0;
        if (kTok * ++c >= ne) {
            c = 0;
            i++;
        }
        load(p, n_list);
        return true;
    }
};

// Cost of a unit of a chunk with n tokens: its decode (about one token's dot products) plus n.
// Returns the first unit, in unit order, whose start cost is at least target (one whole warp);
// *u = its index among all units (every chunk has nt units).
__device__ Walker locate_unit(const UpParams &p, int n_list, int nt, long long target, int lane, int *u) {
    long long base = 0;
    int base_ch = 0;
    for (int i0 = 0; i0 < n_list; i0 += 32) {
        const int i = i0 + lane;
        int ne = 0;
        if (i < n_list) {
            const int e = p.list[i];
            ne = p.offsets[e + 1] - p.offsets[e];
        }
        const int nch = (ne + kTok - 1) / kTok;
        const long long cost = static_cast<long long>(nt) * (nch + ne);
        long long inc = cost;
        int ich = nch;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long v = __shfl_up_sync(0xffffffffu, inc, o);
            const int vc = __shfl_up_sync(0xffffffffu, ich, o);
            if (lane >= o) {
                inc += v;
                ich += vc;
            }
        }
        const unsigned hit = __ballot_sync(0xffffffffu, i < n_list && base + inc > target);
        if (hit) {
            const int j = __ffs(hit) - 1;
            int wi = 0, wc = 0, wt = 0, wu = 0;
            if (lane == j) {
                long long rem = target - (base + inc - cost);  // 0 <= rem < cost
                int c = 0, n = min(kTok, ne);
                while (true) {
                    n = min(kTok, ne - kTok * c);
                    const long long cc = static_cast<long long>(nt) * (1 + n);
                    if (rem < cc) break;
                    rem -= cc;
                    c++;
                }
                int t = static_cast<int>((rem + n) / (1 + n));  // ceil(rem / (1 + n))
                int chunk = base_ch + ich - nch + c;
                wi = i;
                if (t == nt) {  // the next chunk's first unit
                    t = 0;
                    chunk++;
                    if (kTok * ++c >= ne) {
                        c = 0;
                        wi++;
                    }
                }
                wc = c;
                wt = t;
                wu = chunk * nt + t;
            }
            Walker r;
            r.i = __shfl_sync(0xffffffffu, wi, j);
            r.c = __shfl_sync(0xffffffffu, wc, j);
            r.t = __shfl_sync(0xffffffffu, wt, j);
            *u = __shfl_sync(0xffffffffu, wu, j);
            return r;
        }
        base += __shfl_sync(0xffffffffu, inc, 31);
        base_ch += __shfl_sync(0xffffffffu, ich, 31);
    }
    Walker r;
    r.i = n_list;
    r.c = r.t = 0;
    *u = base_ch * nt;
    return r;
}

// Total cost of all units (one whole warp).
__device__ long long total_cost(const UpParams &p, int n_list, int nt, int lane) {
    long long s = 0;
    for (int i = lane; i < n_list; i += 32) {
        const int e = p.list[i];
        const int ne = p.offsets[e + 1] - p.offsets[e];
        s += static_cast<long long>(nt) * ((ne + kTok - 1) / kTok + ne);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    return s;
}

// This lane's part of one unit for N tokens: rows r = lane & 15 of gate and up, 16-byte chunks
// q = 2 * warp + (lane >> 4) + 32 i (two 32-weight sub-blocks each) of the row; pg/pu get the
// lane's partial sums per token (in units of the token's x scale / 16).
template <int N>
__device__ __forceinline__ void unit_dot(const uint8_t *st, const uint8_t *tab, const uint8_t *xs, const int *x8s,
                                         int nbD, int swm, int warp, int lane, float *pg, float *pu) {
    const int r = lane & 15, h = lane >> 4;
    const uint32_t lane4 = static_cast<uint32_t>(lane) * 4u;
    const int rowb = nbD * 64;
    const uint8_t *rg = st + r * rowb, *ru = st + (kIq2TileRows + r) * rowb;
    const uint16_t *dgp = reinterpret_cast<const uint16_t *>(st + 2 * kIq2TileRows * rowb) + r * nbD;
    const uint16_t *dup = dgp + kIq2TileRows * nbD;
    const int s = r & swm, nq = 4 * nbD;
#pragma unroll 1
    for (int q = 2 * warp + h; q < nq; q += 2 * kCompute) {
        const uint4 qg4 = *reinterpret_cast<const uint4 *>(rg + ((q ^ s) << 4));
        const uint4 qu4 = *reinterpret_cast<const uint4 *>(ru + ((q ^ s) << 4));
        const float dg = f16_to_f32(dgp[q >> 2]), du = f16_to_f32(dup[q >> 2]);
#pragma unroll
        for (int sb = 0; sb < 2; sb++) {
            const int c = 2 * q + sb;
            const uint2 qg = sb ? make_uint2(qg4.z, qg4.w) : make_uint2(qg4.x, qg4.y);
            const uint2 qu = sb ? make_uint2(qu4.z, qu4.w) : make_uint2(qu4.x, qu4.y);
            int ceg[N], cog[N], ceu[N], cou[N];
#pragma unroll
            for (int t = 0; t < N; t++) {
                const int b8 = x8s[t * kX8Tok + c];  // the offset of 8 per weight, removed up front
                ceg[t] = -b8;
                ceu[t] = -b8;
                cog[t] = 0;
                cou[t] = 0;
            }
#pragma unroll
            for (int g = 0; g < 4; g++) {
                const uint32_t gvg = *reinterpret_cast<const uint32_t *>(tab + iq2_cb_off(qg.x, g, lane4));
                const uint32_t svg = *reinterpret_cast<const uint32_t *>(tab + iq2_sg_off(qg.y, g, lane4));
                const uint32_t gvu = *reinterpret_cast<const uint32_t *>(tab + iq2_cb_off(qu.x, g, lane4));
                const uint32_t svu = *reinterpret_cast<const uint32_t *>(tab + iq2_sg_off(qu.y, g, lane4));
                const uint32_t evg = (gvg ^ svg) & 0x0F0F0F0Fu, odg = (gvg ^ svg) & 0xF0F0F0F0u;
                const uint32_t evu = (gvu ^ svu) & 0x0F0F0F0Fu, odu = (gvu ^ svu) & 0xF0F0F0F0u;
#pragma unroll
                for (int t = 0; t < N; t++) {
                    const uint4 xv = *reinterpret_cast<const uint4 *>(xs + t * kXTokBytes + (c * 4 + g) * 16);
                    ceg[t] = dp2a_hi_su(xv.y, evg, dp2a_lo_su(xv.x, evg, ceg[t]));
                    cog[t] = dp2a_hi_su(xv.w, odg, dp2a_lo_su(xv.z, odg, cog[t]));
                    ceu[t] = dp2a_hi_su(xv.y, evu, dp2a_lo_su(xv.x, evu, ceu[t]));
                    cou[t] = dp2a_hi_su(xv.w, odu, dp2a_lo_su(xv.z, odu, cou[t]));
                }
            }
            // (s + 1) of each row's sub-block; the odd sums are multiples of 16, so the shift is exact
            const float sg = dg * small_int_to_float(static_cast<int>((qg.y >> 28) + 1u));
            const float su = du * small_int_to_float(static_cast<int>((qu.y >> 28) + 1u));
#pragma unroll
            for (int t = 0; t < N; t++) {
                pg[t] = fmaf(sg, small_int_to_float(ceg[t] + (cog[t] >> 4)), pg[t]);
                pu[t] = fmaf(su, small_int_to_float(ceu[t] + (cou[t] >> 4)), pu[t]);
            }
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1) small_up_kernel(UpParams p) {
    pdl_wait();
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw;  // fixed offsets from the symbol: the table's base folds into its loads
    uint8_t *ring = smem, *tab = smem + kUpTabOff, *xs = smem + kUpXOff;
    int *x8s = reinterpret_cast<int *>(smem + kUpX8Off);
    float4 *xscs = reinterpret_cast<float4 *>(smem + kUpXscOff);
    float *red = reinterpret_cast<float *>(smem + kUpRedOff);  // [2][kCompute][kTok][32]
    // mbarriers: full[2], empty[2], xfull, xempty, rfull[2], rempty[2]
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kUpMiscOff);
    int *info = reinterpret_cast<int *>(bars + 10);  // first unit (i, c, t), unit count
    volatile int *abort_flag = reinterpret_cast<volatile int *>(info + 4);
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + 2);
    const uint32_t xfull = smem_u32(bars + 4), xempty = smem_u32(bars + 5);
    const uint32_t rfull = smem_u32(bars + 6), rempty = smem_u32(bars + 8);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const DeviceWeights &w = p.w;
    const int D = w.D, F = w.F, nbD = w.nbD, nt = F / kIq2TileRows;
    const int n_list = p.meta->n_gemv;

    if (warp == kProducer) {
        if (lane == 0) {
            for (int s = 0; s < kUpStages; s++) {
                mbar_init(full0 + 8 * s, 1);
                mbar_init(empty0 + 8 * s, kCompute);
            }
            mbar_init(xfull, 1);
            mbar_init(xempty, kCompute + 1);
            for (int b = 0; b < 2; b++) {
                mbar_init(rfull + 8 * b, kCompute);
                mbar_init(rempty + 8 * b, 1);
            }
            *abort_flag = 0;
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        }
        // this CTA's units: those whose start cost lies in [C b / G, C (b + 1) / G)
        const long long C = total_cost(p, n_list, nt, lane);
        const long long G = gridDim.x, b = blockIdx.x;
        int u0 = 0, u1 = 0;
        const Walker s0 = locate_unit(p, n_list, nt, C * b / G, lane, &u0);
        locate_unit(p, n_list, nt, C * (b + 1) / G, lane, &u1);
        if (lane == 0) {
            info[0] = s0.i;
            info[1] = s0.c;
            info[2] = s0.t;
            info[3] = u1 - u0;
        }
    } else if (warp < kCompute) {
        const uint2 gown = __ldg(reinterpret_cast<const uint2 *>(p.grid) + warp + 16 * (lane & 15));
        iq2_table_store(tab, gown, warp, lane);
    }
    __syncthreads();
    Walker wk;
    wk.i = info[0];
    wk.c = info[1];
    wk.t = info[2];
    const int nu = info[3];
    if (nu <= 0) return;
    wk.load(p, n_list);

    // ---------------------------------------------------------------- producer
    if (warp == kProducer) {
        if (lane == 0) {
            int stage = 0, ch = -1, x_parity = -1, issued[kUpStages];
            uint32_t phase = 0;
            for (int s = 0; s < kUpStages; s++) issued[s] = -1;
            bool ok = true;
            const uint32_t tb = static_cast<uint32_t>(iq2_tile_bytes(nbD));
            for (int kk = 0; kk < nu; kk++) {
                const bool first = kk == 0 || wk.t == 0;
                if (!mbar_wait(empty0 + 8 * stage, phase ^ 1u, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                mbar_expect_tx(full0 + 8 * stage, tb);
                bulk_load(smem_u32(ring + stage * kUpStageBytes), w.iq2 + iq2_tile_offset(w, wk.e, wk.t * kIq2TileRows),
                          tb, full0 + 8 * stage);
                issued[stage] = static_cast<int>(phase);
                if (++stage == kUpStages) {
                    stage = 0;
                    phase ^= 1u;
                }
                if (first) {  // first unit of a chunk: stage the x of its tokens once the last chunk is done
                    ch++;
                    if (ch > 0 && !mbar_wait(xempty, static_cast<uint32_t>(ch - 1) & 1u, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(xfull, static_cast<uint32_t>(wk.n * (2 * D + D / 8 + 16)));
                    for (int t = 0; t < wk.n; t++) {
                        const int tok = p.perm[wk.pos0 + t] / p.k;
                        bulk_load(smem_u32(xs + t * kXTokBytes), p.xq + static_cast<size_t>(tok) * (D / 8),
                                  static_cast<uint32_t>(2 * D), xfull);
                        bulk_load(smem_u32(x8s + t * kX8Tok), p.x8 + static_cast<size_t>(tok) * (D / 32),
                                  static_cast<uint32_t>(D / 8), xfull);
                        bulk_load(smem_u32(xscs + t), p.xsc + tok, 16u, xfull);
                    }
                    x_parity = ch & 1;
                }
                wk.advance(p, n_list, nt);
            }
            if (!ok) {  // the copies in flight land before the CTA exits
                for (int s = 0; s < kUpStages; s++)
                    if (issued[s] >= 0) mbar_drain(full0 + 8 * s, static_cast<uint32_t>(issued[s]));
                if (x_parity >= 0) mbar_drain(xfull, static_cast<uint32_t>(x_parity));
            }
        }
        return;
    }

    // ---------------------------------------------------------------- compute warps
    if (warp < kCompute) {
        const int swm = iq2_swz(w, 15);
        bool ok = true;
        int ch = -1;
        for (int kk = 0; kk < nu; kk++) {
            const int n = wk.n;
            if (kk == 0 || wk.t == 0) {
                ch++;
                if (ok && !wait_phase(xfull, static_cast<uint32_t>(ch) & 1u, abort_flag, p.status)) ok = false;
            }
            const int stg = kk % kUpStages;
            if (ok && !wait_phase(full0 + 8 * stg, static_cast<uint32_t>(kk / kUpStages) & 1u, abort_flag, p.status))
                ok = false;
            float pg[kTok], pu[kTok];
#pragma unroll
            for (int t = 0; t < kTok; t++) pg[t] = pu[t] = 0.0f;
            if (ok) {
                const uint8_t *st = ring + stg * kUpStageBytes;
                switch (n) {
                    case 1: unit_dot<1>(st, tab, xs, x8s, nbD, swm, warp, lane, pg, pu); break;
                    case 2: unit_dot<2>(st, tab, xs, x8s, nbD, swm, warp, lane, pg, pu); break;
                    case 3: unit_dot<3>(st, tab, xs, x8s, nbD, swm, warp, lane, pg, pu); break;
                    case 4: unit_dot<4>(st, tab, xs, x8s, nbD, swm, warp, lane, pg, pu); break;
                    case 5: unit_dot<5>(st, tab, xs, x8s, nbD, swm, warp, lane, pg, pu); break;
                    default: unit_dot<6>(st, tab, xs, x8s, nbD, swm, warp, lane, pg, pu); break;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * stg);
#pragma unroll
            for (int t = 0; t < kTok; t++) {  // the two column halves of each row
                pg[t] += __shfl_xor_sync(0xffffffffu, pg[t], 16);
                pu[t] += __shfl_xor_sync(0xffffffffu, pu[t], 16);
            }
            const int buf = kk & 1;
            if (kk >= 2) wait_phase(rempty + 8 * buf, static_cast<uint32_t>((kk >> 1) - 1) & 1u, abort_flag, p.status);
            float *rb = red + buf * kRedUnit + warp * kTok * 32;
#pragma unroll
            for (int t = 0; t < kTok; t++)
                if (t < n) rb[t * 32 + lane] = (lane & 16) ? pu[t] : pg[t];  // lanes 0-15 gate, 16-31 up
            __syncwarp();
            if (lane == 0) mbar_arrive(rfull + 8 * buf);
            const bool next_chunk = wk.advance(p, n_list, nt);
            if (kk == nu - 1 || next_chunk) {  // done with this chunk's x
                __syncwarp();
                if (lane == 0) mbar_arrive(xempty);
            }
        }
        return;
    }

    // ---------------------------------------------------------------- finisher
    // per unit: h = silu(gate) * up for the 16 rows and the chunk's tokens, quantised per token
    // to int16 with a power-of-two scale of the 16 values (one down sub-block) and their sum
    bool ok = true;
    int ch = -1;
    const int r = lane & 15, hh = lane >> 4;
    for (int kk = 0; kk < nu; kk++) {
        const int n = wk.n;
        if (kk == 0 || wk.t == 0) {
            ch++;
            if (ok && !wait_phase(xfull, static_cast<uint32_t>(ch) & 1u, abort_flag, p.status)) ok = false;
        }
        const int buf = kk & 1;
        if (ok && !wait_phase(rfull + 8 * buf, static_cast<uint32_t>(kk >> 1) & 1u, abort_flag, p.status)) ok = false;
        const float *rb = red + buf * kRedUnit;
        const int row0 = wk.t * kIq2TileRows;
        for (int t0 = 0; t0 < n; t0 += 2) {
            const int t = t0 + hh;
            const bool valid = ok && t < n;
            float g = 0.0f, u = 0.0f;
            if (valid) {
#pragma unroll
                for (int ww = 0; ww < kCompute; ww++) {
                    g += rb[(ww * kTok + t) * 32 + r];
                    u += rb[(ww * kTok + t) * 32 + 16 + r];
                }
            }
            const float xf = valid ? xscs[t].x * 0.0625f : 0.0f;  // the token's x scale, and 1/16 of (s + 1)
            const float hv = valid ? swiglu(g * xf, u * xf) : 0.0f;
            float m = fabsf(hv), sum = hv;
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) {
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                sum += __shfl_xor_sync(0xffffffffu, sum, o);
            }
            int e = 0;
            frexpf(m, &e);
            e = m > 0.0f ? e : 0;
            if (valid) {
                const size_t pos = static_cast<size_t>(wk.pos0 + t);
                p.hq[pos * F + row0 + q2k_h_pos(r)] = static_cast<int16_t>(__float2int_rn(hv * ldexpf(1.0f, 14 - e)));
                if (r == 0) {
                    p.hsc[pos * (F / 16) + row0 / 16] = ldexpf(1.0f, e - 14);
                    p.hsum[pos * (F / 16) + row0 / 16] = sum;
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(rempty + 8 * buf);
        const bool next_chunk = wk.advance(p, n_list, nt);
        if (kk == nu - 1 || next_chunk) {
            __syncwarp();
            if (lane == 0) mbar_arrive(xempty);
        }
    }
}

// ---------------------------------------------------------------- down

constexpr int kDnRows = 2 * kQ2kTileRows;  // output rows per unit: two down tiles
constexpr int kDnSlots = 8;                // pairs per unit
constexpr int kDnStages = 4;
constexpr int kDnStageBytes = kDnSlots * kDnRows * (kMaxF / 256) * 84;
constexpr int kDnRedOff = kDnStages * kDnStageBytes;
constexpr int kDnMiscOff = kDnRedOff + 2 * kCompute * 8 * 4;
constexpr int kDnSmem = kDnMiscOff + 256;
static_assert(kDnStageBytes % 16 == 0 && kDnSmem <= 232448, "down stages");

struct DownParams {
    DeviceWeights w;
    const int32_t *small_pos;  // positions of the small groups' pairs, expert order
    const int32_t *perm;       // [P] pair id at each position
    const int32_t *topk_idx;   // [P] expert of each pair
    const GroupMeta *meta;
    const int16_t *hq;
    const float *hsc, *hsum;
    float *y;                  // [P][D] by position
    int *status;
};

// A unit is (slot group g: small-group pairs 8g .. 8g+7, row block rb: output rows 8rb .. 8rb+7).
// Thread (s2 = tid >> 6, j2 = tid & 63) owns slot s2 and columns 32 j2 .. 32 j2 + 31 (two 16-column
// sub-blocks) of its pair's h, kept in registers while the slot group lasts.
__global__ void __launch_bounds__(kThreads, 1) small_down_kernel(DownParams p) {
    pdl_wait();
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *ring = smem_raw;
    float *red = reinterpret_cast<float *>(smem_raw + kDnRedOff);  // [2][kCompute][8]
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem_raw + kDnMiscOff);  // full[4], empty[4], rfull[2], rempty[2]
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 12);
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + kDnStages);
    const uint32_t rfull = smem_u32(bars + 2 * kDnStages), rempty = smem_u32(bars + 2 * kDnStages + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const DeviceWeights &w = p.w;
    const int D = w.D, F = w.F, nbF = w.nbF;
    const int nrb = D / kDnRows;
    const int npairs = p.meta->n_small_pairs;
    const int U = (npairs + kDnSlots - 1) / kDnSlots * nrb;
    const int u0 = static_cast<int>(static_cast<long long>(U) * blockIdx.x / gridDim.x);
    const int u1 = static_cast<int>(static_cast<long long>(U) * (blockIdx.x + 1) / gridDim.x);
    const int tile_b = kQ2kTileRows * nbF * 84, slot_b = 2 * tile_b;

    if (threadIdx.x == kProducer * 32) {
        for (int s = 0; s < kDnStages; s++) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, kCompute);
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(rfull + 8 * b, kCompute);
            mbar_init(rempty + 8 * b, 1);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (u0 >= u1) return;

    // ---------------------------------------------------------------- producer
    if (warp == kProducer) {
        if (lane == 0) {
            int stage = 0, issued[kDnStages];
            uint32_t phase = 0;
            for (int s = 0; s < kDnStages; s++) issued[s] = -1;
            bool ok = true;
            for (int u = u0; u < u1; u++) {
                const int g = u / nrb, rb = u % nrb;
                if (!mbar_wait(empty0 + 8 * stage, phase ^ 1u, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                const int ns = min(kDnSlots, npairs - kDnSlots * g);
                mbar_expect_tx(full0 + 8 * stage, static_cast<uint32_t>(ns * slot_b));
                for (int s = 0; s < ns; s++) {
                    const int e = p.topk_idx[p.perm[p.small_pos[kDnSlots * g + s]]];
                    bulk_load(smem_u32(ring + stage * kDnStageBytes + s * slot_b),
                              w.q2k + q2k_tile_offset(w, e, rb * kDnRows), static_cast<uint32_t>(slot_b),
                              full0 + 8 * stage);
                }
                issued[stage] = static_cast<int>(phase);
                if (++stage == kDnStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok)
                for (int s = 0; s < kDnStages; s++)
                    if (issued[s] >= 0) mbar_drain(full0 + 8 * s, static_cast<uint32_t>(issued[s]));
        }
        return;
    }

    // ---------------------------------------------------------------- finisher
    if (warp == kFinisher) {
        bool ok = true;
        for (int u = u0; u < u1; u++) {
            const int it = u - u0, buf = it & 1, g = u / nrb, rb = u % nrb;
            if (ok && !wait_phase(rfull + 8 * buf, static_cast<uint32_t>(it >> 1) & 1u, abort_flag, p.status)) ok = false;
            const float *rbuf = red + buf * kCompute * 8;
#pragma unroll
            for (int i = 0; i < 2; i++) {
                const int idx = lane + 32 * i, s = idx >> 3, r = idx & 7;  // slot, row of the unit
                const int j = kDnSlots * g + s;
                if (ok && j < npairs) {
                    const size_t pos = static_cast<size_t>(p.small_pos[j]);
                    p.y[pos * D + rb * kDnRows + r] = rbuf[(2 * s) * 8 + r] + rbuf[(2 * s + 1) * 8 + r];
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(rempty + 8 * buf);
        }
        return;
    }

    // ---------------------------------------------------------------- compute warps
    const int tid = threadIdx.x, s2 = tid >> 6, j2 = tid & 63;
    bool ok = true;
    int cur = -1;
    bool sval = false;
    uint32_t hp[16];
    float gh0 = 0.0f, gh1 = 0.0f, gs0 = 0.0f, gs1 = 0.0f;
    for (int u = u0; u < u1; u++) {
        const int it = u - u0, g = u / nrb, stg = it % kDnStages;
        if (g != cur) {  // a new slot group: this thread's 32 columns of its pair's h
            cur = g;
            const int j = kDnSlots * g + s2;
            sval = j < npairs && j2 < F / 32;
#pragma unroll
            for (int i = 0; i < 16; i++) hp[i] = 0u;
            gh0 = gh1 = gs0 = gs1 = 0.0f;
            if (sval) {
                const size_t pos = static_cast<size_t>(p.small_pos[j]);
                const uint4 *src = reinterpret_cast<const uint4 *>(p.hq + pos * F + 32 * j2);
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    const uint4 v = __ldcg(src + i);
                    hp[4 * i] = v.x;
                    hp[4 * i + 1] = v.y;
                    hp[4 * i + 2] = v.z;
                    hp[4 * i + 3] = v.w;
                }
                const float2 sc2 = __ldcg(reinterpret_cast<const float2 *>(p.hsc + pos * (F / 16)) + j2);
                const float2 sm2 = __ldcg(reinterpret_cast<const float2 *>(p.hsum + pos * (F / 16)) + j2);
                gh0 = sc2.x;
                gh1 = sc2.y;
                gs0 = sm2.x;
                gs1 = sm2.y;
            }
        }
        if (ok && !wait_phase(full0 + 8 * stg, static_cast<uint32_t>(it / kDnStages) & 1u, abort_flag, p.status))
            ok = false;
        float acc[kDnRows];
#pragma unroll
        for (int r = 0; r < kDnRows; r++) acc[r] = 0.0f;
        uint2 qw[kDnRows];
        uint32_t scw[kDnRows], dd[kDnRows];
        const bool live = ok && sval;
        if (live) {
            const uint8_t *sb = ring + stg * kDnStageBytes + s2 * slot_b;
#pragma unroll
            for (int r = 0; r < kDnRows; r++) {
                const uint8_t *tb = sb + (r / kQ2kTileRows) * tile_b;
                const int rr = r % kQ2kTileRows;
                const uint8_t *blk = tb + rr * nbF * 80 + (j2 >> 3) * 80;
                qw[r] = *reinterpret_cast<const uint2 *>(blk + 16 + 8 * (j2 & 7));
                scw[r] = *reinterpret_cast<const uint16_t *>(blk + 2 * (j2 & 7));
                dd[r] = *reinterpret_cast<const uint32_t *>(tb + kQ2kTileRows * nbF * 80 + rr * nbF * 4 + (j2 >> 3) * 4);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * stg);
        if (live) {
#pragma unroll
            for (int r = 0; r < kDnRows; r++) {
                const int a0 = q2k_idot(qw[r].x, hp), a1 = q2k_idot(qw[r].y, hp + 8);
                const float d = f16_to_f32(static_cast<uint16_t>(dd[r] & 0xffffu));
                const float dmin = f16_to_f32(static_cast<uint16_t>(dd[r] >> 16));
                const uint32_t sc = scw[r];
                const float t = fmaf(gh0 * small_int_to_float(static_cast<int>(sc & 15u)), small_int_to_float(a0),
                                     gh1 * small_int_to_float(static_cast<int>((sc >> 8) & 15u)) * small_int_to_float(a1));
                const float mt = fmaf(gs0, small_int_to_float(static_cast<int>((sc >> 4) & 15u)),
                                      gs1 * small_int_to_float(static_cast<int>(sc >> 12)));
                acc[r] = fmaf(d, t, -dmin * mt);
            }
        }
        const float v = reduce8(acc, lane);
        const int buf = it & 1;
        if (it >= 2) wait_phase(rempty + 8 * buf, static_cast<uint32_t>((it >> 1) - 1) & 1u, abort_flag, p.status);
        if ((lane & 3) == 0) red[buf * kCompute * 8 + warp * 8 + (lane >> 2)] = v;
        __syncwarp();
        if (lane == 0) mbar_arrive(rfull + 8 * buf);
    }
}

int n_sms_sg() {
    static int n = 0;
    if (!n) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 148;
    }
    return n;
}

// h of the small groups lives in the first P rows of the workspace's fp32 h: int16 h [P][F], then
// the sub-block factors [P][F/16] and sums [P][F/16] (2.5 P F bytes of the 4 P F available).
struct HLayout {
    int16_t *hq;
    float *hsc, *hsum;
};
HLayout h_layout(const Workspace &ws, int P, int F) {
    HLayout l;
    uint8_t *hb = reinterpret_cast<uint8_t *>(ws.h32);
    l.hq = reinterpret_cast<int16_t *>(hb);
    l.hsc = reinterpret_cast<float *>(hb + static_cast<size_t>(P) * F * 2);
    l.hsum = l.hsc + static_cast<size_t>(P) * (F / 16);
    return l;
}

}  // namespace

bool small_groups_supported(const DeviceWeights &w) {
    return w.fmt == 0 && w.D <= kMaxD && w.F <= kMaxF && w.D % 256 == 0 && w.F % 256 == 0;
}

int launch_prep_x(const Workspace &ws, const uint16_t *x, int T, int D, void *stream) {
    if (T <= 0) return 0;
    return launch_pdl(prep_x_kernel, dim3(T), dim3(256), 0, static_cast<cudaStream_t>(stream), x, T, D,
                      reinterpret_cast<uint4 *>(ws.xq), ws.x8, reinterpret_cast<float4 *>(ws.xsc));
}

int launch_small_up(const DeviceWeights &w, const Workspace &ws, int T, int k, void *stream) {
    static int seen[64];
    const int err = ensure_smem(reinterpret_cast<const void *>(small_up_kernel), kUpSmem, seen);
    if (err) return err;
    const HLayout l = h_layout(ws, T * k, w.F);
    UpParams p;
    p.w = w;
    p.list = ws.gemv_list;
    p.offsets = ws.offsets;
    p.perm = ws.perm;
    p.meta = ws.meta;
    p.grid = ws.grid;
    p.xq = reinterpret_cast<const uint4 *>(ws.xq);
    p.x8 = ws.x8;
    p.xsc = reinterpret_cast<const float4 *>(ws.xsc);
    p.hq = l.hq;
    p.hsc = l.hsc;
    p.hsum = l.hsum;
    p.k = k;
    p.status = ws.status;
    return launch_pdl(small_up_kernel, dim3(n_sms_sg()), dim3(kThreads), kUpSmem, static_cast<cudaStream_t>(stream), p);
}

int launch_small_down(const DeviceWeights &w, const Workspace &ws, int T, int k, void *stream) {
    static int seen[64];
    const int err = ensure_smem(reinterpret_cast<const void *>(small_down_kernel), kDnSmem, seen);
    if (err) return err;
    const HLayout l = h_layout(ws, T * k, w.F);
    DownParams p;
    p.w = w;
    p.small_pos = ws.small_pos;
    p.perm = ws.perm;
    p.topk_idx = ws.topk_idx;
    p.meta = ws.meta;
    p.hq = l.hq;
    p.hsc = l.hsc;
    p.hsum = l.hsum;
    p.y = ws.y;
    p.status = ws.status;
    return launch_pdl(small_down_kernel, dim3(n_sms_sg()), dim3(kThreads), kDnSmem, static_cast<cudaStream_t>(stream), p);
}

}  // namespace ds4moe
