// One-token step in a single cooperative kernel: routing, gate/up + SwiGLU, down and the
// gate-weighted combine into the residual.
//
// "DwarfStar" README, "运行大于 RAM 的模型": every new token is routed through the experts
// again, so each decode step streams the selected experts' packed rows once. At one token the
// step is a pure stream of bytes, so the kernel is built to keep HBM busy and to spend few
// instructions and little shared-memory bandwidth per streamed weight:
//   * one producer warp streams weight rows into a 4-stage shared-memory ring with 1-D TMA
//     bulk copies; it starts at once on the bf16 shared expert's rows (they need no routing),
//     so the ring fills while the first loads of x and the logits are still in flight
//     and interleaves them with the routed experts' rows, which wait for the top-k; each
//     warp reads its part of a stage into registers and frees the stage before the arithmetic;
//   * every CTA (one per SM) routes the token itself -- top-k of the router logits, ties to the
//     lower index -- so no launch or barrier separates routing from the experts;
//   * gate/up (phase 1): x is held in the table as int16 with a power-of-two scale per 1024-column
//     quarter (2^14 over the quarter's absolute maximum), as the pairs dp2a reads; lane l of every
//     compute warp owns row l & 15 of a unit's gate and up and a strided set of its 16-byte chunks,
//     so a unit ends with one shuffle and one store per lane (the finisher sums the warps).
//     An IQ2-style group of 8 weights is one 32-bit codebook word of nibbles
//     (m - 1, which is even; elements 0, 2, 4, 6 in the low nibbles, 1, 3, 5, 7 in the high ones)
//     and one 32-bit sign word of nibbles, 0x9 (keep) or 0x7 (negate): their XOR is, per nibble,
//     the signed weight plus 8 (m-1 ^ 9 = m + 8, m-1 ^ 7 = 8 - m, no carries). Two masks give
//     the even weights as bytes and 16 x the odd ones; dp2a multiplies them (unsigned) by the
//     int16 x pairs (signed) exactly, and 8 * sum(x) of the sub-block removes the offset. Each
//     lookup is one 4-byte word per lane, so a warp's lookup is one shared-memory wavefront.
//     Each 32-weight sub-block's integer sum is scaled once;
//   * a routed unit is 16 rows of one expert's gate and up, i.e. exactly one 16-column sub-block
//     of its down matrix, so the finisher quantises its 16 h values to int16 with a power-of-two
//     scale of their own, stored in the order q2k_idot reads them;
//   * down (phase 2): each thread keeps 32 columns of h (one expert) in registers for the whole
//     phase, its two sub-blocks brought to one power-of-two scale by an integer shift, in the order
//     that lets the Q2_K-style bit pairs be used with one mask per four codes and no table; a row's two
//     sub-blocks combine their scales and mins in integers, so only two conversions and the two
//     block factors remain in floating point; the bf16 shared expert runs in fp32 on fp32 h;
//   * the cross-warp sums of each unit go through shared memory to a finisher warp, double-
//     buffered and handed over with mbarriers, so compute warps never wait for one another; each
//     output row is summed in a fixed order and added to the residual once: deterministic.
// Every mbarrier wait is bounded (~2 s): a timeout sets DS4MOE_ETIMEOUT in the status word, and
// the warps keep their barrier hand-shakes (without computing) so that the CTA always finishes.
// The kernel is launched cooperatively, so all CTAs are resident together at the grid barrier.
#include <cuda_runtime.h>

#include <algorithm>
#include <cfloat>
#include <climits>

#include "step_common.cuh"

namespace ds4moe {
namespace {

constexpr int kCompute = 16;             // compute warps
constexpr int kProducer = kCompute;      // warp index of the weight streamer
constexpr int kFinisher = kCompute + 1;  // warp index of the unit finisher
constexpr int kThreads = (kCompute + 2) * 32;
constexpr int kStages = 4;
constexpr int kStageBytes = 38912;
constexpr int kRows1 = 16;   // gate/up rows per routed unit: one 16-column sub-block of down
constexpr int kRowsSh = 2;   // shared-expert gate/up rows per unit
constexpr int kRows2 = 4;    // output rows per down unit
static_assert(kRows1 == kIq2TileRows && kRows2 == kQ2kTileRows, "a unit is one weight tile per expert");
constexpr int kLead = 4;     // shared-expert units streamed before the first routed one
constexpr int kMaxD = 4096;
// Shared memory: [ring: kStages x kStageBytes][table: 256 slots of 256 bytes][barriers, scratch].
// Slot e holds codebook entry e in its first 128 bytes (one u32 replica per lane), and in its
// second 128 bytes: sign entry e (e < 128, one replica per lane); for 128 <= e < 192, x as int16
// dp2a pairs, 16 bytes per 8-column group, the 8 groups of 16-byte weight chunk q = e - 128 (two
// 32-column sub-blocks); for e >= 192, x in bf16 for the shared expert, 8-column group g in slot
// 192 + g / 8. A codebook byte offset is then lane * 4 | index << 8: one byte_perm builds it, and
// the table's base folds into the load.
constexpr int kTabOff = kStages * kStageBytes;
constexpr int kTabBytes = 256 * 256;
constexpr int kMiscOff = kTabOff + kTabBytes;
constexpr int kRedBuf = kCompute * 32;  // floats of one unit's partial sums (routed: one per lane and warp)
constexpr int kMaxSharedUnits = 16;     // shared-expert units of one CTA (their partial sums wait in smem)
// misc: mbarriers (14 slots), sidx[8], sgw[8], quarter scales of x[4], x8[128], red[2][kRedBuf],
// shared-unit partials [kMaxSharedUnits][kCompute][4], abort flag
constexpr int kSmemBytes = kMiscOff + 112 + 32 + 32 + 16 + 512 + 2 * kRedBuf * 4 + kMaxSharedUnits * kCompute * 16 + 64;
static_assert(kTabOff % 256 == 0, "table slots are 256-byte aligned");
static_assert(kMaxD / 8 <= 64 * 8, "x (int16 and bf16) fits the second halves of slots 128..255");

// Byte offsets in the table of 8-column group g of x: int16 dp2a pairs, and bf16.
__host__ __device__ constexpr int xq_offset(int g) { return (128 + (g >> 3)) * 256 + 128 + (g & 7) * 16; }
__host__ __device__ constexpr int xb_offset(int g) { return (192 + (g >> 3)) * 256 + 128 + (g & 7) * 16; }

// Named barriers (0 is __syncthreads). The per-unit hand-off between the compute warps and the
// finisher goes through mbarriers instead, so that no compute warp waits for another one.
constexpr int kBarAll = 1;      // compute warps + finisher
constexpr int kBarCompute = 2;  // compute warps
constexpr int kNAll = (kCompute + 1) * 32;
constexpr int kNCompute = kCompute * 32;

__device__ __forceinline__ uint64_t now_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

struct StepParams {
    DeviceWeights w;
    const uint16_t *x;     // bf16 [D]
    const float *logits;   // [E]
    int E;                 // experts the logits route over (a pooled handle: its store's)
    const int32_t *slot_of;  // null, or a pooled handle's expert -> slot map
    float *out;            // [D], += delta
    int k, mode;
    const uint8_t *grid;   // codebook magnitudes [256][8]
    int32_t *topk_idx;     // [k] (written by CTA 0)
    float *topk_w;         // [k]
    int16_t *hq;           // [k][F] the routed experts' h as int16, each 16-row sub-block in dp2a order
    int *hexp;             // [k][F/16] its power-of-two exponent: h = hq * 2^(hexp - 14)
    float *hsh;            // [F] shared expert's h (fp32)
    unsigned long long *bar;  // grid barrier: arrivals since the workspace was made
    unsigned int bar_extra;   // 0 (tests of the bounded wait: arrivals that never come)
    uint64_t *trace;       // null, or [gridDim][6] timestamps (ns)
    int *status;
};

__device__ __forceinline__ int count_of(int n) {
    const int b = static_cast<int>(blockIdx.x), g = static_cast<int>(gridDim.x);
    return n > b ? (n - 1 - b) / g + 1 : 0;
}

// A routed unit costs about kRoutedCost shared units of compute. The shared units are split into
// contiguous ranges in proportion to what each CTA's routed units (blockIdx.x + i * gridDim.x, so
// the first nr % G CTAs have one more) leave of an even share of the total; in closed form, so
// every thread computes its CTA's range [s0, s1) at once.
constexpr int kRoutedCost = 3;
// 32-bit arithmetic: the host admits a shape only if ns * G * (kRoutedCost * nr + ns) < 2^31.
__host__ __device__ inline unsigned shared_capacity_before(unsigned c, unsigned G, unsigned ns, unsigned nr) {
    const unsigned A = kRoutedCost * nr + ns, q = nr / G, rem = nr % G;
    return c * A - kRoutedCost * G * (c * q + (c < rem ? c : rem));
}
__host__ __device__ inline void shared_range(unsigned b, unsigned G, unsigned ns, unsigned nr, int *s0, int *s1) {
    const unsigned all = G * ns;  // shared_capacity_before(G)
    *s0 = all > 0 ? static_cast<int>(ns * shared_capacity_before(b, G, ns, nr) / all) : 0;
    *s1 = all > 0 ? static_cast<int>(ns * shared_capacity_before(b + 1, G, ns, nr) / all) : 0;
}

// Order of one CTA's gate/up units: kLead shared-expert units, then routed and shared
// alternately, then what remains. Routed units are blockIdx.x + i * gridDim.x; the CTA's shared
// units are the contiguous range s0 .. s0+ns-1 (shared_range).
struct Seq1 {
    int ts, tr, ns, nr, s0;
    __device__ bool next(bool &shared, int &unit) {
        if (ts < ns && (tr >= nr || ts < kLead + tr)) {
            shared = true;
            unit = s0 + ts++;
            return true;
        }
        if (tr < nr) {
            shared = false;
            unit = static_cast<int>(blockIdx.x) + tr++ * static_cast<int>(gridDim.x);
            return true;
        }
        return false;
    }
};

__device__ __forceinline__ Seq1 seq1_of(const StepParams &p) {
    Seq1 s;
    s.ts = s.tr = 0;
    const int nr = p.k * (p.w.F / kRows1);
    int s0 = 0, s1 = 0;
    shared_range(blockIdx.x, gridDim.x, p.w.has_shared ? p.w.F / kRowsSh : 0, nr, &s0, &s1);
    s.s0 = s0;
    s.ns = s1 - s0;
    s.nr = count_of(nr);
    return s;
}


// Sums four per-lane values over the warp; afterwards lane l holds the total of value (l >> 3) & 3.
__device__ __forceinline__ float reduce4(float v0, float v1, float v2, float v3, int lane) {
    const bool up16 = lane & 16, up8 = lane & 8;
    float a = up16 ? v2 : v0, b = up16 ? v3 : v1;
    const float sa = up16 ? v0 : v2, sb = up16 ? v1 : v3;
    a += __shfl_xor_sync(0xffffffffu, sa, 16);
    b += __shfl_xor_sync(0xffffffffu, sb, 16);
    float c = up8 ? b : a;
    const float sc = up8 ? a : b;
    c += __shfl_xor_sync(0xffffffffu, sc, 8);
    c += __shfl_xor_sync(0xffffffffu, c, 4);
    c += __shfl_xor_sync(0xffffffffu, c, 2);
    c += __shfl_xor_sync(0xffffffffu, c, 1);
    return c;
}

// Issues the bulk copies of one gate/up unit into a stage (one thread).
__device__ void issue1(const StepParams &p, const int *idx, bool shared, int unit, uint32_t dst, uint32_t bar) {
    const DeviceWeights &w = p.w;
    if (!shared) {
        const int per = w.F / kRows1;
        const int e = idx[unit / per];
        const int row0 = (unit % per) * kRows1;
        const uint32_t bytes = static_cast<uint32_t>(iq2_tile_bytes(w.nbD));  // gate and up rows, one tile
        mbar_expect_tx(bar, bytes);
        bulk_load(dst, w.iq2 + iq2_tile_offset(w, e, row0), bytes, bar);
    } else {
        const int row0 = unit * kRowsSh;
        const uint32_t b = static_cast<uint32_t>(kRowsSh * w.D * 2);
        mbar_expect_tx(bar, 2 * b);
        bulk_load(dst, w.sh_gate + static_cast<size_t>(row0) * w.D, b, bar);
        bulk_load(dst + b, w.sh_up + static_cast<size_t>(row0) * w.D, b, bar);
    }
}

// Issues the bulk copies of one down unit: kRows2 output rows of every routed expert and of
// the shared one.
__device__ void issue2(const StepParams &p, const int *idx, int unit, uint32_t dst, uint32_t bar) {
    const DeviceWeights &w = p.w;
    const int d0 = unit * kRows2;
    const uint32_t tb = static_cast<uint32_t>(q2k_tile_bytes(w.nbF));  // kRows2 rows of one expert
    const uint32_t shb = w.has_shared ? static_cast<uint32_t>(kRows2 * w.F * 2) : 0u;
    mbar_expect_tx(bar, p.k * tb + shb);
    for (int s = 0; s < p.k; s++) bulk_load(dst + s * tb, w.q2k + q2k_tile_offset(w, idx[s], d0), tb, bar);
    if (w.has_shared) bulk_load(dst + p.k * tb, w.sh_down + static_cast<size_t>(d0) * w.F, shb, bar);
}

// Top-k of the logits by one warp (ties to the lower index, NaN orders as -inf) and the gate
// weights of the selected experts (softmax over them, or normalised sigmoids).
template <int NJ>
__device__ void route_warp(const StepParams &p, int lane, int *sidx, float *sgw) {
    const int E = p.E;
    float key[NJ];
#pragma unroll
    for (int j = 0; j < NJ; j++) {
        const int e = lane + 32 * j;
        const float v = (e < E) ? __ldg(p.logits + e) : -INFINITY;
        key[j] = (v != v) ? -INFINITY : v;
    }
    uint32_t taken = 0;
    float my_v = -INFINITY;
    int my_i = 0;
    for (int r = 0; r < p.k; r++) {
        float bv = -INFINITY;
        int bi = INT_MAX;
#pragma unroll
        for (int j = 0; j < NJ; j++) {
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
    if (lane < p.k) num = gate_numerator(my_v, top, p.mode);
    const float den = warp_sum(num);
    if (lane < p.k) {
        sidx[lane] = p.slot_of ? p.slot_of[my_i] : my_i;  // a pooled handle's experts sit in slots
        sgw[lane] = num / den;
        if (blockIdx.x == 0) {
            p.topk_idx[lane] = my_i;
            p.topk_w[lane] = num / den;
        }
    }
}

// Order-preserving key of a logit: a larger float gives a larger unsigned key. NaN orders as
// -inf and -0 as +0 (they compare equal as floats, so the lower expert index wins the tie).
__device__ __forceinline__ uint32_t order_key(float v) {
    if (v != v) v = -INFINITY;
    if (v == 0.0f) v = 0.0f;
    const uint32_t u = __float_as_uint(v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Top-k of at most 256 logits by one warp, the same selection as route_warp: each lane sorts its
// eight (key, index) pairs once with a 19-comparator network (descending key, ascending index),
// then every round takes the largest head key over the warp with one reduction and, among the
// heads that hold it, the smallest expert index with a second; that lane drops its head.
__device__ void route_sorted8(const StepParams &p, int lane, int *sidx, float *sgw) {
    const int E = p.E;
    uint32_t key[8];
    int id[8];
#pragma unroll
    for (int j = 0; j < 8; j++) {
        const int e = lane + 32 * j;
        key[j] = e < E ? order_key(__ldg(p.logits + e)) : 0u;  // 0: no expert (below every logit)
        id[j] = e < E ? e : INT_MAX;
    }
    auto ce = [&](int a, int b) {  // position a takes the larger of (a, b)
        const bool sw = key[b] > key[a] || (key[b] == key[a] && id[b] < id[a]);
        const uint32_t ka = sw ? key[b] : key[a], kb = sw ? key[a] : key[b];
        const int ia = sw ? id[b] : id[a], ib = sw ? id[a] : id[b];
        key[a] = ka;
        key[b] = kb;
        id[a] = ia;
        id[b] = ib;
    };
    ce(0, 2); ce(1, 3); ce(4, 6); ce(5, 7);
    ce(0, 4); ce(1, 5); ce(2, 6); ce(3, 7);
    ce(0, 1); ce(2, 3); ce(4, 5); ce(6, 7);
    ce(2, 4); ce(3, 5);
    ce(1, 4); ce(3, 6);
    ce(1, 2); ce(3, 4); ce(5, 6);
    float my_v = -INFINITY;
    int my_i = 0;
    for (int r = 0; r < p.k; r++) {
        const uint32_t m = __reduce_max_sync(0xffffffffu, key[0]);
        const uint32_t win = __reduce_min_sync(0xffffffffu, key[0] == m ? static_cast<uint32_t>(id[0]) : 0xffffffffu);
        if (lane == r) {
            my_v = key_value(m);
            my_i = static_cast<int>(win);
        }
        if (key[0] == m && static_cast<uint32_t>(id[0]) == win) {
#pragma unroll
            for (int i = 0; i < 7; i++) {
                key[i] = key[i + 1];
                id[i] = id[i + 1];
            }
            key[7] = 0u;
            id[7] = INT_MAX;
        }
    }
    const float top = __shfl_sync(0xffffffffu, my_v, 0);
    float num = 0.0f;
    if (lane < p.k) num = gate_numerator(my_v, top, p.mode);
    const float den = warp_sum(num);
    if (lane < p.k) {
        sidx[lane] = p.slot_of ? p.slot_of[my_i] : my_i;  // a pooled handle's experts sit in slots
        sgw[lane] = num / den;
        if (blockIdx.x == 0) {
            p.topk_idx[lane] = my_i;
            p.topk_w[lane] = num / den;
        }
    }
}

// One IQ2-style 32-weight sub-block of a gate row and of an up row dotted with x: xb holds the
// sub-block's four 8-column groups as int16 pairs (x0,x2), (x4,x6), (x1,x3), (x5,x7), 16 bytes each,
// x8 = 8 * the sum of its 32 values; qg/qu = the rows' 4 codebook indices and sign/scale words;
// dg/du = the blocks' d times the x factor / 16; tab = the table, lane4 = 4 * lane.
__device__ __forceinline__ void iq2_sub2(uint2 qg, uint2 qu, float dg, float du, const uint8_t *xb, int x8,
                                         const uint8_t *tab, uint32_t lane4, float &pg, float &pu) {
    int ceg = -x8, cog = 0, ceu = -x8, cou = 0;  // even and odd elements; the offset of 8 removed up front
#pragma unroll
    for (int g = 0; g < 4; g++) {
        const uint32_t gvg = *reinterpret_cast<const uint32_t *>(tab + iq2_cb_off(qg.x, g, lane4));
        const uint32_t svg = *reinterpret_cast<const uint32_t *>(tab + iq2_sg_off(qg.y, g, lane4));
        const uint32_t gvu = *reinterpret_cast<const uint32_t *>(tab + iq2_cb_off(qu.x, g, lane4));
        const uint32_t svu = *reinterpret_cast<const uint32_t *>(tab + iq2_sg_off(qu.y, g, lane4));
        const uint32_t evg = (gvg ^ svg) & 0x0F0F0F0Fu, odg = (gvg ^ svg) & 0xF0F0F0F0u;
        const uint32_t evu = (gvu ^ svu) & 0x0F0F0F0Fu, odu = (gvu ^ svu) & 0xF0F0F0F0u;
        const uint4 xv = *reinterpret_cast<const uint4 *>(xb + 16 * g);
        ceg = dp2a_hi_su(xv.y, evg, dp2a_lo_su(xv.x, evg, ceg));
        cog = dp2a_hi_su(xv.w, odg, dp2a_lo_su(xv.z, odg, cog));
        ceu = dp2a_hi_su(xv.y, evu, dp2a_lo_su(xv.x, evu, ceu));
        cou = dp2a_hi_su(xv.w, odu, dp2a_lo_su(xv.z, odu, cou));
    }
    // the odd sums are multiples of 16: the shifts are exact; (s + 1) is each row's sub-block scale
    pg = fmaf(dg * small_int_to_float(static_cast<int>((qg.y >> 28) + 1u)), small_int_to_float(ceg + (cog >> 4)), pg);
    pu = fmaf(du * small_int_to_float(static_cast<int>((qu.y >> 28) + 1u)), small_int_to_float(ceu + (cou >> 4)), pu);
}

__device__ __forceinline__ float dot8_bf16(uint4 w, float4 xa, float4 xb, float acc) {
    acc = fmaf(bf16_lo(w.x), xa.x, acc);
    acc = fmaf(bf16_hi(w.x), xa.y, acc);
    acc = fmaf(bf16_lo(w.y), xa.z, acc);
    acc = fmaf(bf16_hi(w.y), xa.w, acc);
    acc = fmaf(bf16_lo(w.z), xb.x, acc);
    acc = fmaf(bf16_hi(w.z), xb.y, acc);
    acc = fmaf(bf16_lo(w.w), xb.z, acc);
    acc = fmaf(bf16_hi(w.w), xb.w, acc);
    return acc;
}

// Bounded grid barrier, one thread per CTA, on a 64-bit arrival counter that only grows: the
// CTAs of one call take tickets n*G .. n*G+G-1 and wait until the counter reaches (n+1)*G, so
// the counter never needs resetting. The add releases this CTA's writes (observed by this
// thread through the CTA barrier before it) at GPU scope; the polling load acquires the others'.
// extra: arrivals beyond the grid's to wait for (0; a test of the bounded wait sets more, which
// never come, so the wait runs out and reports ST_TIMEOUT).
__device__ bool grid_barrier(unsigned long long *count, int *status, unsigned int extra) {
    const unsigned long long G = gridDim.x;
    unsigned long long ticket;
    asm volatile("atom.add.release.gpu.global.u64 %0, [%1], 1;" : "=l"(ticket) : "l"(count) : "memory");
    const unsigned long long target = (ticket / G + 1ull) * G + extra;
    const long long t0 = clock64();
    while (true) {
        unsigned long long v;
        asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(count) : "memory");
        if (v >= target) return true;
        if (clock64() - t0 > kWaitCycles) {
            report(status, ST_TIMEOUT);
            return false;
        }
        __nanosleep(20);
    }
}

// NQ: 1024-column quarters of x (1, 2 or 4); each compute warp holds one of them in registers.
template <int NQ>
__global__ void __launch_bounds__(kThreads, 1) decode_step_kernel(StepParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // fixed offsets from the symbol, so that the table's base folds into its loads
    uint8_t *smem = smem_raw;
    uint8_t *ring = smem;                                                    // kStages x kStageBytes
    uint8_t *tab = smem + kTabOff;
    // mbarriers: full[S], empty[S], route, rfull[2], rempty[2]
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kMiscOff);
    int *sidx = reinterpret_cast<int *>(bars + 2 * kStages + 6);             // [8]
    float *sgw = reinterpret_cast<float *>(sidx + 8);                         // [8]
    float *xsc = sgw + 8;                                                     // [4] x factor of each quarter
    int *x8s = reinterpret_cast<int *>(xsc + 4);                              // [kMaxD / 32]
    float *red = reinterpret_cast<float *>(x8s + kMaxD / 32);                 // [2][kRedBuf]
    float *sacc = red + 2 * kRedBuf;                                          // [kMaxSharedUnits][kCompute][4]
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sacc + kMaxSharedUnits * kCompute * 4);
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + kStages);
    const uint32_t route_bar = smem_u32(bars + 2 * kStages);
    // rfull[b]: the 16 compute warps have written a unit's partial sums into red[b];
    // rempty[b]: the finisher has read them
    const uint32_t rfull = smem_u32(bars + 2 * kStages + 1), rempty = smem_u32(bars + 2 * kStages + 3);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const DeviceWeights &w = p.w;
    const int D = w.D, F = w.F, nbD = w.nbD, nbF = w.nbF;
    const int n2 = D / kRows2;
    uint64_t *tr = (p.trace && threadIdx.x == 0) ? p.trace + 6 * static_cast<size_t>(blockIdx.x) : nullptr;
    if (tr) tr[0] = now_ns();

    if (threadIdx.x == kProducer * 32) {
        for (int s = 0; s < kStages; s++) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, kCompute);
        }
        mbar_init(route_bar, 1);
        for (int b = 0; b < 2; b++) {
            mbar_init(rfull + 8 * b, kCompute);
            mbar_init(rempty + 8 * b, 1);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    // ---------------------------------------------------------------- producer
    if (warp == kProducer) {
        if (lane == 0) {
            int stage = 0, issued_parity[kStages];
            uint32_t phase = 0;
            for (int s = 0; s < kStages; s++) issued_parity[s] = -1;
            bool ok = true, routed = false;
            auto acquire = [&](bool needs_route) -> bool {
                if (needs_route && !routed) {
                    if (!mbar_wait(route_bar, 0u, abort_flag, p.status)) return false;
                    routed = true;
                }
                return mbar_wait(empty0 + 8 * stage, phase ^ 1u, abort_flag, p.status);
            };
            auto advance = [&]() {
                issued_parity[stage] = static_cast<int>(phase);
                if (++stage == kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            };
            Seq1 q = seq1_of(p);
            bool shared;
            int unit;
            while (ok && q.next(shared, unit)) {
                if (!acquire(!shared)) {
                    ok = false;
                    break;
                }
                issue1(p, sidx, shared, unit, smem_u32(ring + stage * kStageBytes), full0 + 8 * stage);
                advance();
            }
            for (int u = blockIdx.x; ok && u < n2; u += gridDim.x) {
                if (!acquire(true)) {
                    ok = false;
                    break;
                }
                issue2(p, sidx, u, smem_u32(ring + stage * kStageBytes), full0 + 8 * stage);
                advance();
            }
            if (!ok)
                for (int s = 0; s < kStages; s++)
                    if (issued_parity[s] >= 0) mbar_drain(full0 + 8 * s, static_cast<uint32_t>(issued_parity[s]));
        }
        return;  // the producer takes no part in the named barriers
    }

    const Seq1 seq0 = seq1_of(p);

    // ---------------------------------------------------------------- finisher
    if (warp == kFinisher) {
        // route first: the producer's routed units and the down phase wait for it
        if (p.E <= 256)
            route_sorted8(p, lane, sidx, sgw);
        else
            route_warp<32>(p, lane, sidx, sgw);
        __syncwarp();
        if (lane == 0) mbar_arrive(route_bar);
        int it = 0;
        Seq1 q = seq0;
        bool shared;
        int unit;
        while (q.next(shared, unit)) {
            if (shared) continue;  // the compute warps finish the shared units themselves
            const int buf = it & 1;
            const float *rb = red + buf * kRedBuf;
            wait_phase(rfull + 8 * buf, static_cast<uint32_t>(it >> 1) & 1u, abort_flag, p.status);
            {
                // lane r < 16: row r of the unit = column r of one down sub-block; the warps wrote
                // gate row r in lane r and up row r in lane 16 + r
                const int per = F / kRows1, slot = unit / per, row0 = (unit % per) * kRows1;
                float v = 0.0f;
#pragma unroll
                for (int ww = 0; ww < kCompute; ww++) v += rb[ww * 32 + lane];
                const float u = __shfl_down_sync(0xffffffffu, v, 16);
                const float hv = lane < kRows1 ? swiglu(v, u) : 0.0f;
                // int16 with the 16 values' power-of-two scale (2^14 over their absolute maximum)
                float m = fabsf(hv);
#pragma unroll
                for (int o = 8; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                int e = 0;
                frexpf(m, &e);
                e = m > 0.0f ? e : 0;
                if (lane < kRows1)
                    p.hq[static_cast<size_t>(slot) * F + row0 + q2k_h_pos(lane)] =
                        static_cast<int16_t>(__float2int_rn(hv * ldexpf(1.0f, 14 - e)));
                if (lane == 0) p.hexp[static_cast<size_t>(slot) * (F / 16) + row0 / 16] = e;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(rempty + 8 * buf);
            it++;
        }
        bar_sync(kBarAll, kNAll);  // this CTA's h is written
        for (int u = blockIdx.x; u < n2; u += gridDim.x, it++) {
            const int buf = it & 1;
            const float *rb = red + buf * kRedBuf;
            wait_phase(rfull + 8 * buf, static_cast<uint32_t>(it >> 1) & 1u, abort_flag, p.status);
            if (lane < kRows2) {
                float s = 0.0f;
#pragma unroll
                for (int ww = 0; ww < kCompute; ww++) s += rb[ww * 4 + lane];
                p.out[u * kRows2 + lane] += s;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(rempty + 8 * buf);
        }
        return;
    }

    // -------------------------------------------------------------------- compute warps: prologue
    const int tid = threadIdx.x;  // 0 .. kNCompute-1
    // all global loads of the prologue first, so that their latencies overlap
    const int qx = warp % NQ, rg = warp / NQ;
    const int c = qx * 32 + lane;  // this lane's 32-column sub-block of x
    const bool cval = c < D / 32;
    uint4 raw[4];  // this lane's 32 columns of x
#pragma unroll
    for (int j = 0; j < 4; j++)
        raw[j] = cval ? __ldg(reinterpret_cast<const uint4 *>(p.x) + 4 * c + j) : make_uint4(0, 0, 0, 0);
    const uint2 gown = __ldg(reinterpret_cast<const uint2 *>(p.grid) + warp + 16 * (lane & 15));  // for iq2_table_store
    const bool xfq = tid < D / 8;
    const uint4 xv = xfq ? __ldg(reinterpret_cast<const uint4 *>(p.x) + tid) : make_uint4(0, 0, 0, 0);
    // bf16 x for the shared expert: thread tid stores group tid (D <= 8 * kNCompute)
    if (xfq) *reinterpret_cast<uint4 *>(tab + xb_offset(tid)) = xv;
    // int16 x with the quarter's power-of-two scale, per group the pairs (x0,x2), (x4,x6), (x1,x3),
    // (x5,x7); x8 = 8 * their sum. The warps of the first row group store it for the routed units.
    uint32_t xr[16];
    float xinv;
    int x8 = 0;
    {
        float m = 0.0f;
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const uint32_t u4[4] = {raw[j].x, raw[j].y, raw[j].z, raw[j].w};
#pragma unroll
            for (int i = 0; i < 4; i++) m = fmaxf(m, fmaxf(fabsf(bf16_lo(u4[i])), fabsf(bf16_hi(u4[i]))));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        int e = 0;
        frexpf(m, &e);
        e = m > 0.0f ? e : 0;
        const float sc = ldexpf(1.0f, 14 - e);
        xinv = ldexpf(1.0f, e - 14) * 0.0625f;  // also carries the sub-block scale's 1/16
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const uint32_t u4[4] = {raw[j].x, raw[j].y, raw[j].z, raw[j].w};
            uint32_t q[8];
#pragma unroll
            for (int i = 0; i < 4; i++) {
                q[2 * i] = round_to_int_bits(bf16_lo(u4[i]) * sc);
                q[2 * i + 1] = round_to_int_bits(bf16_hi(u4[i]) * sc);
            }
#pragma unroll
            for (int i = 0; i < 8; i++) x8 += static_cast<int>(static_cast<int16_t>(q[i] & 0xffffu));
            xr[4 * j] = __byte_perm(q[0], q[2], 0x5410);
            xr[4 * j + 1] = __byte_perm(q[4], q[6], 0x5410);
            xr[4 * j + 2] = __byte_perm(q[1], q[3], 0x5410);
            xr[4 * j + 3] = __byte_perm(q[5], q[7], 0x5410);
        }
        x8 *= 8;
    }
    if (rg == 0 && cval) {  // lane: sub-block c = 4 groups of int16 x, their sum, the quarter's factor
#pragma unroll
        for (int j = 0; j < 4; j++)
            *reinterpret_cast<uint4 *>(tab + xq_offset(4 * c + j)) = make_uint4(xr[4 * j], xr[4 * j + 1], xr[4 * j + 2], xr[4 * j + 3]);
        x8s[c] = x8;
        if (lane == 0) xsc[qx] = xinv;
    }
    iq2_table_store(tab, gown, warp, lane);  // codebook and sign words, one replica per lane
    bar_sync(kBarCompute, kNCompute);
    if (tr) tr[1] = now_ns();

    // ring position rc: stage rc % kStages, parity (rc / kStages) & 1
    bool ok = true;
    auto wait_stage = [&](int rc) -> const uint8_t * {
        if (!ok || !wait_phase(full0 + 8 * (rc % kStages), static_cast<uint32_t>(rc / kStages) & 1u, abort_flag, p.status)) {
            ok = false;
            return nullptr;
        }
        return ring + (rc % kStages) * kStageBytes;
    };
    auto release_stage = [&](int rc) {
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * (rc % kStages));
    };

    // ---------------------------------------------------------------- phase 1: gate/up
    const uint32_t lane4 = static_cast<uint32_t>(lane) * 4u;
    const int swm = iq2_swz(w, 15);  // chunk permutation mask of the tiles' rows (iq2_swz)
    int rc = 0;  // ring position: units of both phases
    int hc = 0;  // hand-offs to the finisher: routed units, then down units
    {
        Seq1 q = seq0;
        bool shared;
        int unit;
        while (q.next(shared, unit)) {
            const int it = rc++;
            const uint8_t *st = wait_stage(it);
            if (shared) {
                // two bf16 rows of gate and up; thread tid takes columns 8*tid .. +7 (D <= 8 * kNCompute).
                // The stage is read into registers and released before the arithmetic.
                float g0 = 0.0f, u0 = 0.0f, g1 = 0.0f, u1 = 0.0f;
                if (st) {
                    const int nq = D / 8;
                    const bool qv = tid < nq;
                    const uint4 *sgw8 = reinterpret_cast<const uint4 *>(st);
                    const uint4 *suw8 = sgw8 + kRowsSh * nq;
                    uint4 wv[4];
                    if (qv) {
                        wv[0] = sgw8[tid];
                        wv[1] = sgw8[nq + tid];
                        wv[2] = suw8[tid];
                        wv[3] = suw8[nq + tid];
                    }
                    release_stage(it);
                    if (qv) {
                        const uint4 xw = *reinterpret_cast<const uint4 *>(tab + xb_offset(tid));
                        const float4 xa = make_float4(bf16_lo(xw.x), bf16_hi(xw.x), bf16_lo(xw.y), bf16_hi(xw.y));
                        const float4 xb = make_float4(bf16_lo(xw.z), bf16_hi(xw.z), bf16_lo(xw.w), bf16_hi(xw.w));
                        g0 = dot8_bf16(wv[0], xa, xb, g0);
                        g1 = dot8_bf16(wv[1], xa, xb, g1);
                        u0 = dot8_bf16(wv[2], xa, xb, u0);
                        u1 = dot8_bf16(wv[3], xa, xb, u1);
                    }
                }
                // no hand-off: the warp's sums wait in shared memory until the end of the phase
                const float v = reduce4(g0, u0, g1, u1, lane);
                if ((lane & 7) == 0) sacc[((q.ts - 1) * kCompute + warp) * 4 + (lane >> 3)] = v;
            } else {
                const int buf = hc & 1;
                float *rb = red + buf * kRedBuf;
                // lane l owns row l & 15 of the unit's gate and up and, of each row, the 16-byte chunks
                // q = 2 * warp + (l >> 4) + 32 i (two 32-weight sub-blocks each): it decodes whole
                // groups of its rows with x read from the table (half-warp broadcasts), so a unit
                // needs one shuffle and one store per lane instead of a reduction per row
                if (hc >= 2) wait_phase(rempty + 8 * buf, static_cast<uint32_t>((hc >> 1) - 1) & 1u, abort_flag, p.status);
                float pg = 0.0f, pu = 0.0f;
                if (st) {
                    const int r = lane & 15, rowb = nbD * 64, sw = r & swm;
                    const uint8_t *rgp = st + r * rowb, *rup = st + (kRows1 + r) * rowb;
                    const uint16_t *dgp = reinterpret_cast<const uint16_t *>(st + 2 * kRows1 * rowb) + r * nbD;
                    const uint16_t *dup = dgp + kRows1 * nbD;
#pragma unroll 1
                    for (int q = 2 * warp + (lane >> 4); q < 4 * nbD; q += 2 * kCompute) {
                        const uint4 qg4 = *reinterpret_cast<const uint4 *>(rgp + ((q ^ sw) << 4));
                        const uint4 qu4 = *reinterpret_cast<const uint4 *>(rup + ((q ^ sw) << 4));
                        const float xf = xsc[q >> 4];  // the quarter's x factor (1024 columns = 16 chunks)
                        const float dg = f16_to_f32(dgp[q >> 2]) * xf, du = f16_to_f32(dup[q >> 2]) * xf;
                        const uint8_t *xb = tab + xq_offset(8 * q);  // groups 8q .. 8q+7, 128 contiguous bytes
                        iq2_sub2(make_uint2(qg4.x, qg4.y), make_uint2(qu4.x, qu4.y), dg, du, xb, x8s[2 * q], tab,
                                 lane4, pg, pu);
                        iq2_sub2(make_uint2(qg4.z, qg4.w), make_uint2(qu4.z, qu4.w), dg, du, xb + 64, x8s[2 * q + 1],
                                 tab, lane4, pg, pu);
                    }
                    release_stage(it);
                }
                pg += __shfl_xor_sync(0xffffffffu, pg, 16);  // the row's two column halves
                pu += __shfl_xor_sync(0xffffffffu, pu, 16);
                rb[warp * 32 + lane] = (lane & 16) ? pu : pg;  // lanes 0-15 gate, 16-31 up
                __syncwarp();
                if (lane == 0) mbar_arrive(rfull + 8 * buf);
                hc++;
            }
        }
        // the CTA's shared-expert units: per row, the 16 warps' gate and up sums, then SwiGLU
        bar_sync(kBarCompute, kNCompute);
        const int nsu = q.ns;
        for (int i = tid; i < nsu * kRowsSh; i += kNCompute) {
            const int j = i / kRowsSh, r = i % kRowsSh;
            float g = 0.0f, u = 0.0f;
#pragma unroll
            for (int ww = 0; ww < kCompute; ww++) {
                g += sacc[(j * kCompute + ww) * 4 + 2 * r];
                u += sacc[(j * kCompute + ww) * 4 + 2 * r + 1];
            }
            p.hsh[(q.s0 + j) * kRowsSh + r] = swiglu(g, u);
        }
    }

    // ---------------------------------------------------------------- grid barrier: all h written
    bar_sync(kBarAll, kNAll);
    if (tr) tr[2] = now_ns();
    if (threadIdx.x == 0 && !grid_barrier(p.bar, p.status, p.bar_extra)) *abort_flag = 1;
    bar_sync(kBarCompute, kNCompute);
    if (tr) tr[3] = now_ns();

    // this thread's down columns: expert slot s2, columns 32*j2 .. +31 (two sub-blocks)
    const int s2 = tid >> 6, j2 = tid & 63;
    const bool sval = s2 < p.k;
    // the thread's 32 int16 h values (two sub-blocks, each with its own exponent) brought to one
    // power-of-two scale: the sub-block with the smaller exponent is shifted right (rounded) by
    // the difference; hp keeps q2k_idot's order, hs0/hs1 = the sub-blocks' integer sums
    uint32_t hp[16];
    int hs0 = 0, hs1 = 0;
    float gh = 0.0f;  // gate weight x the dequantisation factor
    float4 hs = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
    for (int i = 0; i < 16; i++) hp[i] = 0u;
    if (sval) {
        const uint4 *src = reinterpret_cast<const uint4 *>(p.hq + static_cast<size_t>(s2) * F + 32 * j2);
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const uint4 v = __ldcg(src + i);
            hp[4 * i] = v.x;
            hp[4 * i + 1] = v.y;
            hp[4 * i + 2] = v.z;
            hp[4 * i + 3] = v.w;
        }
        const int2 ex = __ldcg(reinterpret_cast<const int2 *>(p.hexp + static_cast<size_t>(s2) * (F / 16)) + j2);
        const int et = max(ex.x, ex.y);
#pragma unroll
        for (int sb = 0; sb < 2; sb++) {
            const int sh = min(et - (sb ? ex.y : ex.x), 16);
            int sum = 0;
#pragma unroll
            for (int i = 0; i < 8; i++) {
                int lo = static_cast<int>(static_cast<int16_t>(hp[8 * sb + i] & 0xffffu));
                int hi = static_cast<int>(hp[8 * sb + i]) >> 16;
                if (sh > 0) {
                    lo = (lo + (1 << (sh - 1))) >> sh;
                    hi = (hi + (1 << (sh - 1))) >> sh;
                }
                hp[8 * sb + i] = (static_cast<uint32_t>(lo) & 0xffffu) | (static_cast<uint32_t>(hi) << 16);
                sum += lo + hi;
            }
            if (sb) hs1 = sum; else hs0 = sum;
        }
        gh = sgw[s2] * ldexpf(1.0f, et - 14);
    }
    if (w.has_shared) hs = __ldcg(reinterpret_cast<const float4 *>(p.hsh) + tid);
    if (tr) tr[4] = now_ns();

    // ---------------------------------------------------------------- phase 2: down + combine
    // stage: per routed slot one down tile ([sq: kRows2 x nbF x 80][dd: kRows2 x nbF x 4]), then
    // the shared expert's kRows2 bf16 rows
    const int tb = kRows2 * nbF * 84;
    const int blk_off = s2 * tb + (j2 >> 3) * 80, dd_off = s2 * tb + kRows2 * nbF * 80 + (j2 >> 3) * 4;
    const int sh_off = p.k * tb + 8 * tid;
    for (int u = blockIdx.x; u < n2; u += gridDim.x) {
        const int r0 = rc++;   // ring position
        const int hcur = hc++;  // hand-off to the finisher
        const int buf = hcur & 1;
        float *rb = red + buf * kRedBuf;
        const uint8_t *st = wait_stage(r0);
        float acc[kRows2] = {0.0f, 0.0f, 0.0f, 0.0f};
        if (st) {
            uint2 qw[kRows2], bw[kRows2];
            uint32_t scw[kRows2], dd[kRows2];
#pragma unroll
            for (int r = 0; r < kRows2; r++) {
                if (sval) {
                    const uint8_t *blk = st + blk_off + r * nbF * 80;
                    qw[r] = *reinterpret_cast<const uint2 *>(blk + 16 + 8 * (j2 & 7));
                    scw[r] = *reinterpret_cast<const uint16_t *>(blk + 2 * (j2 & 7));
                    dd[r] = *reinterpret_cast<const uint32_t *>(st + dd_off + r * nbF * 4);
                }
                if (w.has_shared) bw[r] = *reinterpret_cast<const uint2 *>(st + sh_off + r * F * 2);
            }
            release_stage(r0);
#pragma unroll
            for (int r = 0; r < kRows2; r++) {
                if (sval) {
                    // sum_sb d sc_sb (q . h)_sb - dmin m_sb sum(h)_sb, in integers up to the two block factors;
                    // the two conversions go to the conversion unit, idle in this phase (rounded once)
                    const int a0 = q2k_idot(qw[r].x, hp), a1 = q2k_idot(qw[r].y, hp + 8);
                    const uint32_t sc = scw[r];
                    const int i1 = static_cast<int>(sc & 15u) * a0 + static_cast<int>((sc >> 8) & 15u) * a1;
                    const int i2 = static_cast<int>((sc >> 4) & 15u) * hs0 + static_cast<int>(sc >> 12) * hs1;
                    const float d = f16_to_f32(static_cast<uint16_t>(dd[r] & 0xffffu));
                    const float dmin = f16_to_f32(static_cast<uint16_t>(dd[r] >> 16));
                    acc[r] = gh * fmaf(d, __int2float_rn(i1), -dmin * __int2float_rn(i2));
                }
                if (w.has_shared) {
                    acc[r] = fmaf(bf16_lo(bw[r].x), hs.x, acc[r]);
                    acc[r] = fmaf(bf16_hi(bw[r].x), hs.y, acc[r]);
                    acc[r] = fmaf(bf16_lo(bw[r].y), hs.z, acc[r]);
                    acc[r] = fmaf(bf16_hi(bw[r].y), hs.w, acc[r]);
                }
            }
        }
        const float v = reduce4(acc[0], acc[1], acc[2], acc[3], lane);
        if (hcur >= 2) wait_phase(rempty + 8 * buf, static_cast<uint32_t>((hcur >> 1) - 1) & 1u, abort_flag, p.status);
        if ((lane & 7) == 0) rb[warp * 4 + (lane >> 3)] = v;
        __syncwarp();
        if (lane == 0) mbar_arrive(rfull + 8 * buf);
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

int decode_step_ctas() { return n_sms(); }

// Whether the fused single-token kernel covers this shape.
bool decode_step_supported(const DeviceWeights &w, int k) {
    if (w.fmt != 0) return false;  // the 2-bit formats only
    if (k < 1 || k > 8 || w.F != 2048 || w.D % 256 != 0 || w.D > kMaxD || w.E > 1024) return false;
    if (static_cast<size_t>(kRows1) * w.nbD * 132 > kStageBytes) return false;
    if (w.has_shared && static_cast<size_t>(kRowsSh) * 2 * w.D * 2 > kStageBytes) return false;
    const size_t down = static_cast<size_t>(k) * kRows2 * w.nbF * 84 + (w.has_shared ? kRows2 * w.F * 2 : 0);
    if (down > kStageBytes) return false;
    // every CTA's share of shared-expert units is non-negative and fits the partials area
    const unsigned G = n_sms();
    const unsigned ns = w.has_shared ? w.F / kRowsSh : 0, nr = k * (w.F / kRows1);
    if (static_cast<unsigned long long>(ns) * G * (kRoutedCost * nr + ns) >= (1ull << 31)) return false;
    if (ns > 0 && kRoutedCost * G * (nr / G + 1) > kRoutedCost * nr + ns) return false;  // every share >= 0
    for (unsigned c = 0; c < G; c++) {
        int s0 = 0, s1 = 0;
        shared_range(c, G, ns, nr, &s0, &s1);
        if (s1 - s0 > kMaxSharedUnits) return false;
    }
    return true;
}

int launch_decode_step(const DeviceWeights &w, const Workspace &ws, const uint16_t *x, const float *logits, int k,
                       int gate_mode, float *out, uint64_t *trace, int E_route, const int32_t *slot_of,
                       unsigned int bar_extra, void *stream) {
    static int seen[3][64];
    const int nq = w.D <= 1024 ? 1 : w.D <= 2048 ? 2 : 4;  // 1024-column quarters of x
    const void *kern = nq == 1   ? reinterpret_cast<const void *>(decode_step_kernel<1>)
                       : nq == 2 ? reinterpret_cast<const void *>(decode_step_kernel<2>)
                                 : reinterpret_cast<const void *>(decode_step_kernel<4>);
    int err = ensure_smem(kern, kSmemBytes, seen[nq == 1 ? 0 : nq == 2 ? 1 : 2]);
    if (err) return err;
    StepParams p;
    p.w = w;
    p.x = x;
    p.logits = logits;
    p.E = E_route;
    p.slot_of = slot_of;
    p.out = out;
    p.k = k;
    p.mode = gate_mode;
    p.grid = ws.grid;
    p.topk_idx = ws.topk_idx;
    p.topk_w = ws.topk_w;
    // h32 holds at least (k + 1) * F floats: int16 h and exponents of the routed experts, the shared h
    uint8_t *hb = reinterpret_cast<uint8_t *>(ws.h32);
    p.hq = reinterpret_cast<int16_t *>(hb);
    p.hexp = reinterpret_cast<int *>(hb + static_cast<size_t>(k) * w.F * 2);
    p.hsh = reinterpret_cast<float *>(p.hexp + static_cast<size_t>(k) * (w.F / 16));
    p.bar = reinterpret_cast<unsigned long long *>(ws.gbar);
    p.bar_extra = bar_extra;
    p.trace = trace;
    p.status = ws.status;
    void *args[] = {&p};
    return static_cast<int>(cudaLaunchCooperativeKernel(kern, dim3(n_sms()), dim3(kThreads), args, kSmemBytes,
                                                        static_cast<cudaStream_t>(stream)));
}

}  // namespace ds4moe
