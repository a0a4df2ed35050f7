// Fused dequant-GEMV path for decode-sized expert groups (and the shared expert at small T).
//
// Memory-bound: each routed expert's packed rows are streamed once per call with 128-bit
// coalesced loads, decoded in registers (the IQ2 grid lives in shared memory), and dotted
// with the group's tokens, staged in shared memory. Phase 1 computes
// h = silu(W_gate x) * (W_up x) for each row of F; phase 2 computes y = W_down h.
// Everything accumulates in fp32 on exact fp32 weight values.
//
// Source: "DwarfStar" README, "运行大于 RAM 的模型" -- every new token is routed through
// the experts again, so decode streams expert weights; "Part 5: 服务层" §6 -- the ready
// decode steps of several sessions run in one batched kernel, weights read once.
#include <cuda_runtime.h>

#include "common.cuh"
#include "step_common.cuh"

namespace ds4moe {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kUpRows = 16;        // routed rows (of F) per phase-1 item: 2 per warp
constexpr int kUpSharedRows = 8;   // shared-expert rows per phase-1 item: 1 per warp
constexpr int kDownRows = 32;      // routed rows (of D) per phase-2 item: 4 per warp
constexpr int kDownSharedRows = 8; // shared-expert rows per phase-2 item: 1 per warp

struct Items {
    int routed;       // routed items
    int total;        // routed + shared items
    int per_group;    // routed items per group
};

// Contiguous item range of this CTA, so consecutive items usually share a group and the
// staged tokens are reused. The routed items come first, then the shared expert's; the ranges
// split the bytes evenly (a routed item streams cr bytes, a shared one cs): item i starts at
// byte offset c_i, and CTA b takes the items with c_i in [B*b/G, B*(b+1)/G) of the total B.
__device__ __forceinline__ int item_at(long long c, int routed, long long cr, long long cs) {
    const long long cr_all = routed * cr;
    if (c <= cr_all) return static_cast<int>((c + cr - 1) / cr);
    return routed + static_cast<int>((c - cr_all + cs - 1) / cs);
}
__device__ __forceinline__ void cta_range(int routed, int shared, long long cr, long long cs, int &begin, int &end) {
    const long long B = routed * cr + shared * cs, G = gridDim.x;
    begin = item_at(B * blockIdx.x / G, routed, cr, cs);
    end = item_at(B * (blockIdx.x + 1) / G, routed, cr, cs);
}

// Swizzled index of 16-byte chunk c in a staged token row (bank-conflict-free for the
// lane-strided access patterns below).
__device__ __forceinline__ int swz8(int c) { return c ^ ((c >> 3) & 7); }
__device__ __forceinline__ int swz16(int c) { return c ^ ((c >> 4) & 7); }

__device__ __forceinline__ void dot8_bf16(const float w[8], uint4 xv, float &acc) {
    acc = fmaf(w[0], bf16_lo(xv.x), acc);
    acc = fmaf(w[1], bf16_hi(xv.x), acc);
    acc = fmaf(w[2], bf16_lo(xv.y), acc);
    acc = fmaf(w[3], bf16_hi(xv.y), acc);
    acc = fmaf(w[4], bf16_lo(xv.z), acc);
    acc = fmaf(w[5], bf16_hi(xv.z), acc);
    acc = fmaf(w[6], bf16_lo(xv.w), acc);
    acc = fmaf(w[7], bf16_hi(xv.w), acc);
}

__device__ __forceinline__ void bf16x8(uint4 v, float w[8]) {
    w[0] = bf16_lo(v.x); w[1] = bf16_hi(v.x); w[2] = bf16_lo(v.y); w[3] = bf16_hi(v.y);
    w[4] = bf16_lo(v.z); w[5] = bf16_hi(v.z); w[6] = bf16_lo(v.w); w[7] = bf16_hi(v.w);
}

__device__ __forceinline__ float dot4(float4 a, float4 b, float acc) {
    acc = fmaf(a.x, b.x, acc);
    acc = fmaf(a.y, b.y, acc);
    acc = fmaf(a.z, b.z, acc);
    return fmaf(a.w, b.w, acc);
}

// The 4-bit variant: sub-block j (32 weights) of a Q4_K-style block whose first 16 bytes are
// hdr: its scale d * sc_j and offset dmin * m_j, both exact in fp32.
__device__ __forceinline__ void q4_sub_scale(uint4 hdr, int j, float &ds, float &dm) {
    const float d = f16_to_f32(static_cast<uint16_t>(hdr.x & 0xffffu));
    const float dmin = f16_to_f32(static_cast<uint16_t>(hdr.x >> 16));
    const uint32_t low = ((j < 4 ? hdr.y : hdr.z) >> (8 * (j & 3))) & 0xffu;
    const uint32_t high = (hdr.w >> (8 * (j >> 1) + 4 * (j & 1))) & 15u;
    ds = __fmul_rn(d, static_cast<float>((low & 15u) | ((high & 3u) << 4)));
    dm = __fmul_rn(dmin, static_cast<float>((low >> 4) | ((high >> 2) << 4)));
}

// Eight 4-bit codes of one u32 (weight i in bits 4i..4i+3) as weights d sc q - dmin m, rounded once.
__device__ __forceinline__ void q4_group(uint32_t word, float ds, float dm, float w[8]) {
#pragma unroll
    for (int i = 0; i < 8; i++) w[i] = q2k_weight(ds, dm, (word >> (4 * i)) & 15u);
}

struct UpParams {
    DeviceWeights w;
    const uint16_t *x;  // bf16 [T][D]
    const int32_t *perm, *offsets, *gemv_list;
    const GroupMeta *meta;
    const uint8_t *grid;  // [256][8]
    float *h;             // [P+T][F]
    int T, k, P;
    int shared;           // shared expert on this path
    const int32_t *shared_flag;  // non-null: the shared expert only when *shared_flag (a repair)
    // the 4-bit variant: the tokens as int16 dp2a pairs (see prep_x_kernel), 8 x each 32-column
    // sub-block's sum of them, and each token's factor back to x
    const uint4 *xq;
    const int *x8;
    const float4 *xsc;
    int *status;  // the handle's status word (bounded waits of the streamed kernel)
};

// Phase 1: h[pos][r] = silu(gate_r . x) * (up_r . x) for the group's tokens.
template <int NT, bool Q4>
__global__ void __launch_bounds__(kThreads) gemv_up_kernel(UpParams p) {
    pdl_wait();
    extern __shared__ __align__(16) uint8_t smem[];
    uint2 *grid_s = reinterpret_cast<uint2 *>(smem);              // 256 x 8 B
    uint4 *xs = reinterpret_cast<uint4 *>(smem + 2048);           // [NT][D/8] swizzled
    const int D = p.w.D, F = p.w.F, nbD = p.w.nbD, D8 = D / 8;
    // the 4-bit variant also stages the int16 tokens: [NT][D/8] swizzled, then [NT][D/32], [NT]
    uint4 *xqs = xs + NT * D8;
    int *x8s = reinterpret_cast<int *>(xqs + (Q4 ? NT * D8 : 0));
    float *xfs = reinterpret_cast<float *>(x8s + (Q4 ? NT * (D / 32) : 0));
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < 256; i += kThreads) grid_s[i] = reinterpret_cast<const uint2 *>(p.grid)[i];

    const int n_gemv = p.meta->n_gemv;
    const int per_group = F / kUpRows;
    const int routed = n_gemv * per_group;
    const int n_shared = (p.shared && (!p.shared_flag || *p.shared_flag)) ? F / kUpSharedRows : 0;
    // bytes per item: 16 rows of gate and up in the routed format (per 256 columns), 8 bf16 rows
    const long long cr = 2LL * kUpRows * (Q4 ? 144 : 66), cs = 2LL * kUpSharedRows * 512;
    int begin, end;
    cta_range(routed, n_shared, cr, cs, begin, end);
    int staged_key = -1, staged_tok0 = -1;  // which tokens sit in xs
    __syncthreads();

    for (int item = begin; item < end; item++) {
        const bool is_routed = item < routed;
        int e = 0, off = 0, n = 0, r0 = 0, key = -2;
        if (is_routed) {
            const int gi = item / per_group;
            e = p.gemv_list[gi];
            off = p.offsets[e];
            n = p.offsets[e + 1] - off;
            r0 = (item % per_group) * kUpRows;
            key = e;
        } else {
            n = p.T;
            off = p.P;
            r0 = (item - routed) * kUpSharedRows;
        }
        for (int tok0 = 0; tok0 < n; tok0 += NT) {
            const int nt = min(NT, n - tok0);
            if (key != staged_key || tok0 != staged_tok0) {
                __syncthreads();
                for (int i = threadIdx.x; i < nt * D8; i += kThreads) {
                    const int j = i / D8, c = i - j * D8;
                    const int tok = is_routed ? p.perm[off + tok0 + j] / p.k : tok0 + j;
                    xs[j * D8 + swz8(c)] = reinterpret_cast<const uint4 *>(p.x + static_cast<size_t>(tok) * D)[c];
                    if (Q4) xqs[j * D8 + swz8(c)] = p.xq[static_cast<size_t>(tok) * D8 + c];
                }
                if (Q4) {
                    for (int i = threadIdx.x; i < nt * (D / 32); i += kThreads) {
                        const int j = i / (D / 32), c = i - j * (D / 32);
                        const int tok = is_routed ? p.perm[off + tok0 + j] / p.k : tok0 + j;
                        x8s[i] = p.x8[static_cast<size_t>(tok) * (D / 32) + c];
                    }
                    for (int j = threadIdx.x; j < nt; j += kThreads) {
                        const int tok = is_routed ? p.perm[off + tok0 + j] / p.k : tok0 + j;
                        xfs[j] = p.xsc[tok].x;
                    }
                }
                __syncthreads();
                staged_key = key;
                staged_tok0 = tok0;
            }
            if (is_routed && Q4) {
#pragma unroll 1
                for (int rr = 0; rr < kUpRows / kWarps; rr++) {
                    const int r = r0 + warp + rr * kWarps;
                    const uint8_t *rg = q4_row(p.w, 0, e, r), *ru = q4_row(p.w, 1, e, r);
                    float ag[NT], au[NT];
#pragma unroll
                    for (int j = 0; j < NT; j++) ag[j] = au[j] = 0.0f;
                    // 32-weight sub-blocks c of the row, U per lane at a time: all their loads in flight
                    // before any is used (a single token has little else to hide the latency with)
                    constexpr int U = NT == 1 ? 4 : 2;
                    const int nsub = nbD * 8;
                    for (int c0 = lane; c0 < nsub; c0 += 32 * U) {
                        uint4 hg[U], hu[U], vg[U], vu[U];
#pragma unroll
                        for (int t = 0; t < U; t++) {
                            const int c = min(c0 + 32 * t, nsub - 1), b = c >> 3, sub = c & 7;
                            hg[t] = __ldg(reinterpret_cast<const uint4 *>(rg + b * 144));
                            hu[t] = __ldg(reinterpret_cast<const uint4 *>(ru + b * 144));
                            vg[t] = __ldg(reinterpret_cast<const uint4 *>(rg + b * 144 + 16) + sub);
                            vu[t] = __ldg(reinterpret_cast<const uint4 *>(ru + b * 144 + 16) + sub);
                        }
#pragma unroll
                        for (int t = 0; t < U; t++) {
                            const int c = c0 + 32 * t, sub = c & 7;
                            if (c >= nsub) break;
                            float dsg, dmg, dsu, dmu;
                            q4_sub_scale(hg[t], sub, dsg, dmg);
                            q4_sub_scale(hu[t], sub, dsu, dmu);
                            // even codes of each group of 8 as bytes, odd codes as bytes: exact
                            // integer dot products with the int16 token pairs
                            uint32_t eg[4], og[4], eu[4], ou[4];
#pragma unroll
                            for (int g = 0; g < 4; g++) {
                                const uint32_t wgw = g == 0 ? vg[t].x : g == 1 ? vg[t].y : g == 2 ? vg[t].z : vg[t].w;
                                const uint32_t wuw = g == 0 ? vu[t].x : g == 1 ? vu[t].y : g == 2 ? vu[t].z : vu[t].w;
                                eg[g] = wgw & 0x0F0F0F0Fu;
                                og[g] = (wgw >> 4) & 0x0F0F0F0Fu;
                                eu[g] = wuw & 0x0F0F0F0Fu;
                                ou[g] = (wuw >> 4) & 0x0F0F0F0Fu;
                            }
#pragma unroll
                            for (int j = 0; j < NT; j++) {
                                if (j < nt) {
                                    int sg = 0, su = 0;
#pragma unroll
                                    for (int g = 0; g < 4; g++) {
                                        const uint4 xv = xqs[j * D8 + swz8(4 * c + g)];
                                        sg = dp2a_hi_su(xv.y, eg[g], dp2a_lo_su(xv.x, eg[g], sg));
                                        sg = dp2a_hi_su(xv.w, og[g], dp2a_lo_su(xv.z, og[g], sg));
                                        su = dp2a_hi_su(xv.y, eu[g], dp2a_lo_su(xv.x, eu[g], su));
                                        su = dp2a_hi_su(xv.w, ou[g], dp2a_lo_su(xv.z, ou[g], su));
                                    }
                                    const float sx = static_cast<float>(x8s[j * (D / 32) + c] >> 3);  // sum of the 32 int16 x
                                    ag[j] = fmaf(dsg, static_cast<float>(sg), fmaf(-dmg, sx, ag[j]));
                                    au[j] = fmaf(dsu, static_cast<float>(su), fmaf(-dmu, sx, au[j]));
                                }
                            }
                        }
                    }
#pragma unroll
                    for (int j = 0; j < NT; j++) {
                        if (j < nt) {
                            // the int16 tokens carry the factor xf back to x
                            const float g = warp_sum(ag[j]) * xfs[j], u = warp_sum(au[j]) * xfs[j];
                            if (lane == 0) p.h[static_cast<size_t>(off + tok0 + j) * F + r] = swiglu(g, u);
                        }
                    }
                }
            } else if (is_routed) {
#pragma unroll 1
                for (int rr = 0; rr < kUpRows / kWarps; rr++) {
                    const int r = r0 + warp + rr * kWarps;
                    const uint4 *qg = reinterpret_cast<const uint4 *>(iq2_qs_row(p.w, 0, e, r));
                    const uint4 *qu = reinterpret_cast<const uint4 *>(iq2_qs_row(p.w, 1, e, r));
                    const uint16_t *dg = iq2_d_row(p.w, 0, e, r);
                    const uint16_t *du = iq2_d_row(p.w, 1, e, r);
                    float ag[NT], au[NT];
#pragma unroll
                    for (int j = 0; j < NT; j++) ag[j] = au[j] = 0.0f;
                    for (int c = lane; c < nbD * 4; c += 32) {
                        const int cs = c ^ iq2_swz(p.w, r);
                        const uint4 vg = __ldg(qg + cs), vu = __ldg(qu + cs);
                        const float sdg = f16_to_f32(__ldg(dg + (c >> 2)));
                        const float sdu = f16_to_f32(__ldg(du + (c >> 2)));
#pragma unroll
                        for (int sb = 0; sb < 2; sb++) {
                            const uint32_t ig = sb ? vg.z : vg.x, wgd = sb ? vg.w : vg.y;
                            const uint32_t iu = sb ? vu.z : vu.x, wud = sb ? vu.w : vu.y;
                            const float scg = iq2_scale(sdg, wgd), scu = iq2_scale(sdu, wud);
#pragma unroll
                            for (int g = 0; g < 4; g++) {
                                float wg[8], wu[8];
                                iq2_group(grid_s[(ig >> (8 * g)) & 255u], (wgd >> (7 * g)) & 127u, scg, wg);
                                iq2_group(grid_s[(iu >> (8 * g)) & 255u], (wud >> (7 * g)) & 127u, scu, wu);
                                const int xc = swz8(8 * c + 4 * sb + g);
#pragma unroll
                                for (int j = 0; j < NT; j++) {
                                    if (j < nt) {
                                        const uint4 xv = xs[j * D8 + xc];
                                        dot8_bf16(wg, xv, ag[j]);
                                        dot8_bf16(wu, xv, au[j]);
                                    }
                                }
                            }
                        }
                    }
#pragma unroll
                    for (int j = 0; j < NT; j++) {
                        if (j < nt) {
                            const float g = warp_sum(ag[j]), u = warp_sum(au[j]);
                            if (lane == 0) p.h[static_cast<size_t>(off + tok0 + j) * F + r] = swiglu(g, u);
                        }
                    }
                }
            } else {
                const int r = r0 + warp;
                const uint4 *sg = reinterpret_cast<const uint4 *>(p.w.sh_gate + static_cast<size_t>(r) * D);
                const uint4 *su = reinterpret_cast<const uint4 *>(p.w.sh_up + static_cast<size_t>(r) * D);
                float ag[NT], au[NT];
#pragma unroll
                for (int j = 0; j < NT; j++) ag[j] = au[j] = 0.0f;
                constexpr int US = NT == 1 ? 8 : 1;  // 16-byte chunks per lane in flight
                for (int c0 = lane; c0 < D8; c0 += 32 * US) {
                    uint4 vg[US], vu[US];
#pragma unroll
                    for (int t = 0; t < US; t++) {
                        const int c = min(c0 + 32 * t, D8 - 1);
                        vg[t] = __ldg(sg + c);
                        vu[t] = __ldg(su + c);
                    }
#pragma unroll
                    for (int t = 0; t < US; t++) {
                        const int c = c0 + 32 * t;
                        if (c >= D8) break;
                        float wg[8], wu[8];
                        bf16x8(vg[t], wg);
                        bf16x8(vu[t], wu);
                        const int xc = swz8(c);
#pragma unroll
                        for (int j = 0; j < NT; j++) {
                            if (j < nt) {
                                const uint4 xv = xs[j * D8 + xc];
                                dot8_bf16(wg, xv, ag[j]);
                                dot8_bf16(wu, xv, au[j]);
                            }
                        }
                    }
                }
#pragma unroll
                for (int j = 0; j < NT; j++) {
                    if (j < nt) {
                        const float g = warp_sum(ag[j]), u = warp_sum(au[j]);
                        if (lane == 0) p.h[static_cast<size_t>(off + tok0 + j) * F + r] = swiglu(g, u);
                    }
                }
            }
        }
    }
}

struct DownParams {
    DeviceWeights w;
    const int32_t *offsets, *gemv_list;
    const GroupMeta *meta;
    const float *h;  // [P+T][F]
    float *y;        // [P+T][D]
    int T, P;
    int shared;
    const int32_t *shared_flag;  // non-null: the shared expert only when *shared_flag (a repair)
    // the 4-bit variant, when given: each pair's h as int16 dp2a pairs (prep_h_kernel), the sum
    // of each 32-column sub-block of them, and the factor back to h
    const uint4 *hq;
    const int *hsum;
    const float *hsc;
    int *status;  // the handle's status word (bounded waits of the streamed kernel)
};

// The 4-bit variant's down rows: each pair's fp32 h row as int16 pairs (h0,h2), (h4,h6), (h1,h3),
// (h5,h7) per 8-column group with a power-of-two scale of its own, 2^(14-e) for the exponent e of
// the row's largest |h|; the sum of each 32-column sub-block of them; the factor 2^(e-14) back.
// One CTA per row (256 threads, one 8-column group per thread and pass).
__global__ void __launch_bounds__(256) prep_h_kernel(const float *__restrict__ h, int rows, int F,
                                                     uint4 *__restrict__ hq, int *__restrict__ hsum,
                                                     float *__restrict__ hsc) {
    pdl_wait();
    __shared__ float wmax[8];
    const int row = blockIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (row >= rows) return;
    const float4 *hr = reinterpret_cast<const float4 *>(h + static_cast<size_t>(row) * F);
    float m = 0.0f;
    for (int i = threadIdx.x; i < F / 4; i += 256) {
        const float4 v = hr[i];
        m = fmaxf(m, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
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
    for (int gi = threadIdx.x; gi < F / 8; gi += 256) {  // F / 8 is a multiple of 32: whole warps
        const float4 a = hr[2 * gi], b = hr[2 * gi + 1];
        const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        uint32_t q[8];
        int sum = 0;
#pragma unroll
        for (int i = 0; i < 8; i++) {
            q[i] = round_to_int_bits(v[i] * sc);
            sum += static_cast<int>(static_cast<int16_t>(q[i] & 0xffffu));
        }
        hq[static_cast<size_t>(row) * (F / 8) + gi] =
            make_uint4(__byte_perm(q[0], q[2], 0x5410), __byte_perm(q[4], q[6], 0x5410),
                       __byte_perm(q[1], q[3], 0x5410), __byte_perm(q[5], q[7], 0x5410));
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        if ((gi & 3) == 0) hsum[static_cast<size_t>(row) * (F / 32) + (gi >> 2)] = sum;
    }
    if (threadIdx.x == 0) hsc[row] = ldexpf(1.0f, e - 14);
}

// Phase 2: y[pos][r] = down_r . h[pos] for the group's tokens.
template <int NT, bool Q4>
__global__ void __launch_bounds__(kThreads) gemv_down_kernel(DownParams p) {
    pdl_wait();
    extern __shared__ __align__(16) uint8_t smem[];
    float4 *hs = reinterpret_cast<float4 *>(smem);  // [NT][F/4] swizzled
    const int D = p.w.D, F = p.w.F, nbF = p.w.nbF, F4 = F / 4, F8 = F / 8;
    // the 4-bit variant with int16 h: [NT][F/8] swizzled, then [NT][F/32] sums, [NT] factors
    const bool ih = Q4 && p.hq != nullptr;
    uint4 *hqs = reinterpret_cast<uint4 *>(hs + NT * F4);
    int *hsums = reinterpret_cast<int *>(hqs + (Q4 ? NT * F8 : 0));
    float *hfs = reinterpret_cast<float *>(hsums + (Q4 ? NT * (F / 32) : 0));
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int n_gemv = p.meta->n_gemv;
    const int per_group = D / kDownRows;
    const int routed = n_gemv * per_group;
    const int n_shared = (p.shared && (!p.shared_flag || *p.shared_flag)) ? D / kDownSharedRows : 0;
    // bytes per item: 32 rows in the routed format (per 256 columns), 8 bf16 rows
    const long long cr = static_cast<long long>(kDownRows) * (Q4 ? 144 : 84), cs = kDownSharedRows * 512LL;
    int begin, end;
    cta_range(routed, n_shared, cr, cs, begin, end);
    int staged_key = -1, staged_tok0 = -1;

    for (int item = begin; item < end; item++) {
        const bool is_routed = item < routed;
        int e = 0, off = 0, n = 0, r0 = 0, key = -2;
        if (is_routed) {
            const int gi = item / per_group;
            e = p.gemv_list[gi];
            off = p.offsets[e];
            n = p.offsets[e + 1] - off;
            r0 = (item % per_group) * kDownRows;
            key = e;
        } else {
            n = p.T;
            off = p.P;
            r0 = (item - routed) * kDownSharedRows;
        }
        for (int tok0 = 0; tok0 < n; tok0 += NT) {
            const int nt = min(NT, n - tok0);
            if (key != staged_key || tok0 != staged_tok0) {
                __syncthreads();
                for (int i = threadIdx.x; i < nt * F4; i += kThreads) {
                    const int j = i / F4, c = i - j * F4;
                    hs[j * F4 + swz16(c)] = reinterpret_cast<const float4 *>(p.h + static_cast<size_t>(off + tok0 + j) * F)[c];
                }
                if (ih && is_routed) {
                    for (int i = threadIdx.x; i < nt * F8; i += kThreads) {
                        const int j = i / F8, c = i - j * F8;
                        hqs[j * F8 + swz8(c)] = p.hq[static_cast<size_t>(off + tok0 + j) * F8 + c];
                    }
                    for (int i = threadIdx.x; i < nt * (F / 32); i += kThreads) {
                        const int j = i / (F / 32), c = i - j * (F / 32);
                        hsums[i] = p.hsum[static_cast<size_t>(off + tok0 + j) * (F / 32) + c];
                    }
                    for (int j = threadIdx.x; j < nt; j += kThreads) hfs[j] = p.hsc[off + tok0 + j];
                }
                __syncthreads();
                staged_key = key;
                staged_tok0 = tok0;
            }
            if (is_routed && Q4 && NT == 1) {
                constexpr int RP = 2;  // rows per pass: their loads in flight together
#pragma unroll 1
                for (int rr = 0; rr < kDownRows / kWarps; rr += RP) {
                    const uint8_t *rdq[RP];
                    float acc[RP][NT];
#pragma unroll
                    for (int q = 0; q < RP; q++) {
                        rdq[q] = q4_row(p.w, 2, e, r0 + warp + (rr + q) * kWarps);
#pragma unroll
                        for (int j = 0; j < NT; j++) acc[q][j] = 0.0f;
                    }
                    const int nsub = nbF * 8;
                    for (int c0 = lane; c0 < nsub; c0 += 64) {  // two 32-weight sub-blocks per lane and row at a time
                        uint4 hd2[RP][2], vd2[RP][2];
#pragma unroll
                        for (int q = 0; q < RP; q++)
#pragma unroll
                            for (int t = 0; t < 2; t++) {
                                const int c = min(c0 + 32 * t, nsub - 1), b = c >> 3, sub = c & 7;
                                hd2[q][t] = __ldg(reinterpret_cast<const uint4 *>(rdq[q] + b * 144));
                                vd2[q][t] = __ldg(reinterpret_cast<const uint4 *>(rdq[q] + b * 144 + 16) + sub);
                            }
#pragma unroll
                        for (int q = 0; q < RP; q++)
#pragma unroll
                        for (int t = 0; t < 2; t++) {
                        const int c = c0 + 32 * t, sub = c & 7;
                        if (c >= nsub) break;
                        const uint4 hd = hd2[q][t], vd = vd2[q][t];
                        float ds, dm;
                        q4_sub_scale(hd, sub, ds, dm);
                        if (ih) {  // exact integer dot products of the codes with the int16 h
                            uint32_t ev[4], ov[4];
#pragma unroll
                            for (int g = 0; g < 4; g++) {
                                const uint32_t wd = g == 0 ? vd.x : g == 1 ? vd.y : g == 2 ? vd.z : vd.w;
                                ev[g] = wd & 0x0F0F0F0Fu;
                                ov[g] = (wd >> 4) & 0x0F0F0F0Fu;
                            }
#pragma unroll
                            for (int j = 0; j < NT; j++) {
                                if (j < nt) {
                                    int sd = 0;
#pragma unroll
                                    for (int g = 0; g < 4; g++) {
                                        const uint4 hv = hqs[j * F8 + swz8(4 * c + g)];
                                        sd = dp2a_hi_su(hv.y, ev[g], dp2a_lo_su(hv.x, ev[g], sd));
                                        sd = dp2a_hi_su(hv.w, ov[g], dp2a_lo_su(hv.z, ov[g], sd));
                                    }
                                    acc[q][j] = fmaf(ds, static_cast<float>(sd),
                                                     fmaf(-dm, static_cast<float>(hsums[j * (F / 32) + c]), acc[q][j]));
                                }
                            }
                            continue;
                        }
#pragma unroll
                        for (int g = 0; g < 4; g++) {
                            float wv[8];
                            q4_group(g == 0 ? vd.x : g == 1 ? vd.y : g == 2 ? vd.z : vd.w, ds, dm, wv);
#pragma unroll
                            for (int j = 0; j < NT; j++) {
                                if (j < nt) {
                                    const float4 h0 = hs[j * F4 + swz16(8 * c + 2 * g)], h1 = hs[j * F4 + swz16(8 * c + 2 * g + 1)];
                                    acc[q][j] = dot4(make_float4(wv[0], wv[1], wv[2], wv[3]), h0, acc[q][j]);
                                    acc[q][j] = dot4(make_float4(wv[4], wv[5], wv[6], wv[7]), h1, acc[q][j]);
                                }
                            }
                        }
                        }
                    }
#pragma unroll
                    for (int q = 0; q < RP; q++)
#pragma unroll
                        for (int j = 0; j < NT; j++) {
                            if (j < nt) {
                                const float v = warp_sum(acc[q][j]) * (ih ? hfs[j] : 1.0f);
                                if (lane == 0) p.y[static_cast<size_t>(off + tok0 + j) * D + r0 + warp + (rr + q) * kWarps] = v;
                            }
                        }
                }
            } else if (is_routed && Q4) {  // several tokens: one row at a time
#pragma unroll 1
                for (int rr = 0; rr < kDownRows / kWarps; rr++) {
                    const int r = r0 + warp + rr * kWarps;
                    const uint8_t *rd = q4_row(p.w, 2, e, r);
                    float acc[NT];
#pragma unroll
                    for (int j = 0; j < NT; j++) acc[j] = 0.0f;
                    const int nsub = nbF * 8;
                    for (int c0 = lane; c0 < nsub; c0 += 64) {  // two 32-weight sub-blocks per lane at a time
                        uint4 hd2[2], vd2[2];
#pragma unroll
                        for (int t = 0; t < 2; t++) {
                            const int c = min(c0 + 32 * t, nsub - 1), b = c >> 3, sub = c & 7;
                            hd2[t] = __ldg(reinterpret_cast<const uint4 *>(rd + b * 144));
                            vd2[t] = __ldg(reinterpret_cast<const uint4 *>(rd + b * 144 + 16) + sub);
                        }
#pragma unroll
                        for (int t = 0; t < 2; t++) {
                        const int c = c0 + 32 * t, sub = c & 7;
                        if (c >= nsub) break;
                        const uint4 hd = hd2[t], vd = vd2[t];
                        float ds, dm;
                        q4_sub_scale(hd, sub, ds, dm);
                        if (ih) {  // exact integer dot products of the codes with the int16 h
                            uint32_t ev[4], ov[4];
#pragma unroll
                            for (int g = 0; g < 4; g++) {
                                const uint32_t wd = g == 0 ? vd.x : g == 1 ? vd.y : g == 2 ? vd.z : vd.w;
                                ev[g] = wd & 0x0F0F0F0Fu;
                                ov[g] = (wd >> 4) & 0x0F0F0F0Fu;
                            }
#pragma unroll
                            for (int j = 0; j < NT; j++) {
                                if (j < nt) {
                                    int sd = 0;
#pragma unroll
                                    for (int g = 0; g < 4; g++) {
                                        const uint4 hv = hqs[j * F8 + swz8(4 * c + g)];
                                        sd = dp2a_hi_su(hv.y, ev[g], dp2a_lo_su(hv.x, ev[g], sd));
                                        sd = dp2a_hi_su(hv.w, ov[g], dp2a_lo_su(hv.z, ov[g], sd));
                                    }
                                    acc[j] = fmaf(ds, static_cast<float>(sd),
                                                  fmaf(-dm, static_cast<float>(hsums[j * (F / 32) + c]), acc[j]));
                                }
                            }
                            continue;
                        }
#pragma unroll
                        for (int g = 0; g < 4; g++) {
                            float wv[8];
                            q4_group(g == 0 ? vd.x : g == 1 ? vd.y : g == 2 ? vd.z : vd.w, ds, dm, wv);
#pragma unroll
                            for (int j = 0; j < NT; j++) {
                                if (j < nt) {
                                    const float4 h0 = hs[j * F4 + swz16(8 * c + 2 * g)], h1 = hs[j * F4 + swz16(8 * c + 2 * g + 1)];
                                    acc[j] = dot4(make_float4(wv[0], wv[1], wv[2], wv[3]), h0, acc[j]);
                                    acc[j] = dot4(make_float4(wv[4], wv[5], wv[6], wv[7]), h1, acc[j]);
                                }
                            }
                        }
                        }
                    }
#pragma unroll
                    for (int j = 0; j < NT; j++) {
                        if (j < nt) {
                            const float v = warp_sum(acc[j]) * (ih ? hfs[j] : 1.0f);
                            if (lane == 0) p.y[static_cast<size_t>(off + tok0 + j) * D + r] = v;
                        }
                    }
                }
            } else if (is_routed) {
#pragma unroll 1
                for (int rr = 0; rr < kDownRows / kWarps; rr++) {
                    const int r = r0 + warp + rr * kWarps;
                    const uint8_t *sq = q2k_sq_row(p.w, e, r);
                    const uint32_t *dd = q2k_dd_row(p.w, e, r);
                    float acc[NT];
#pragma unroll
                    for (int j = 0; j < NT; j++) acc[j] = 0.0f;
                    for (int c = lane; c < nbF * 4; c += 32) {
                        const int b = c >> 2, part = c & 3;
                        const uint4 qv = __ldg(reinterpret_cast<const uint4 *>(sq + b * 80 + 16) + part);
                        const uint32_t scw = __ldg(reinterpret_cast<const uint32_t *>(sq + b * 80) + part);
                        const uint32_t ddw = __ldg(dd + b);
                        const float d = f16_to_f32(static_cast<uint16_t>(ddw & 0xffffu));
                        const float dmin = f16_to_f32(static_cast<uint16_t>(ddw >> 16));
#pragma unroll
                        for (int sub = 0; sub < 4; sub++) {
                            const uint32_t sc = (scw >> (8 * sub)) & 15u, mn = (scw >> (8 * sub + 4)) & 15u;
                            const float ds = __fmul_rn(d, static_cast<float>(sc));
                            const float dm = __fmul_rn(dmin, static_cast<float>(mn));
                            const uint32_t qw = sub == 0 ? qv.x : sub == 1 ? qv.y : sub == 2 ? qv.z : qv.w;
                            float wv[16];
#pragma unroll
                            for (int i = 0; i < 16; i++) wv[i] = q2k_weight(ds, dm, (qw >> (2 * i)) & 3u);
#pragma unroll
                            for (int j = 0; j < NT; j++) {
                                if (j < nt) {
#pragma unroll
                                    for (int q4 = 0; q4 < 4; q4++) {
                                        const float4 hv = hs[j * F4 + swz16(16 * c + 4 * sub + q4)];
                                        acc[j] = dot4(make_float4(wv[4 * q4], wv[4 * q4 + 1], wv[4 * q4 + 2], wv[4 * q4 + 3]), hv, acc[j]);
                                    }
                                }
                            }
                        }
                    }
#pragma unroll
                    for (int j = 0; j < NT; j++) {
                        if (j < nt) {
                            const float v = warp_sum(acc[j]);
                            if (lane == 0) p.y[static_cast<size_t>(off + tok0 + j) * D + r] = v;
                        }
                    }
                }
            } else {
                const int r = r0 + warp;
                const uint4 *sd = reinterpret_cast<const uint4 *>(p.w.sh_down + static_cast<size_t>(r) * F);
                float acc[NT];
#pragma unroll
                for (int j = 0; j < NT; j++) acc[j] = 0.0f;
                constexpr int US = NT == 1 ? 8 : 1;  // 16-byte chunks per lane in flight
                for (int c0 = lane; c0 < F8; c0 += 32 * US) {
                    uint4 vd[US];
#pragma unroll
                    for (int t = 0; t < US; t++) vd[t] = __ldg(sd + min(c0 + 32 * t, F8 - 1));
#pragma unroll
                    for (int t = 0; t < US; t++) {
                        const int c = c0 + 32 * t;
                        if (c >= F8) break;
                        float wv[8];
                        bf16x8(vd[t], wv);
#pragma unroll
                        for (int j = 0; j < NT; j++) {
                            if (j < nt) {
                                const float4 h0 = hs[j * F4 + swz16(2 * c)], h1 = hs[j * F4 + swz16(2 * c + 1)];
                                acc[j] = dot4(make_float4(wv[0], wv[1], wv[2], wv[3]), h0, acc[j]);
                                acc[j] = dot4(make_float4(wv[4], wv[5], wv[6], wv[7]), h1, acc[j]);
                            }
                        }
                    }
                }
#pragma unroll
                for (int j = 0; j < NT; j++) {
                    if (j < nt) {
                        const float v = warp_sum(acc[j]);
                        if (lane == 0) p.y[static_cast<size_t>(off + tok0 + j) * D + r] = v;
                    }
                }
            }
        }
    }
}

// Device dequantisation of one resident matrix (tests): the same decode as the kernels.
__global__ void dequant_kernel(DeviceWeights w, int expert, int matrix, const uint8_t *grid, float *dst32,
                               uint16_t *dst16) {
    const int D = w.D, F = w.F;
    const int rows = matrix == DS4MOE_DOWN ? D : F, cols = matrix == DS4MOE_DOWN ? F : D;
    const size_t nchunks = static_cast<size_t>(rows) * cols / 64;  // 64 weights per chunk
    for (size_t ci = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; ci < nchunks;
         ci += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const size_t r = ci / (cols / 64);
        const int c = static_cast<int>(ci - r * (cols / 64));
        float v[64];
        if (w.fmt == 1) {  // the 4-bit variant: chunk c = sub-blocks 2c, 2c+1
            const int m = matrix == DS4MOE_DOWN ? 2 : matrix == DS4MOE_GATE ? 0 : 1;
            const uint8_t *row = q4_row(w, m, expert, static_cast<int>(r));
            const int b = c >> 2;
            const uint4 hdr = *reinterpret_cast<const uint4 *>(row + b * 144);
            for (int half = 0; half < 2; half++) {
                const int sub = 2 * (c & 3) + half;
                float ds, dm;
                q4_sub_scale(hdr, sub, ds, dm);
                const uint4 q = *(reinterpret_cast<const uint4 *>(row + b * 144 + 16) + sub);
                q4_group(q.x, ds, dm, v + 32 * half);
                q4_group(q.y, ds, dm, v + 32 * half + 8);
                q4_group(q.z, ds, dm, v + 32 * half + 16);
                q4_group(q.w, ds, dm, v + 32 * half + 24);
            }
        } else if (matrix == DS4MOE_DOWN) {
            const uint8_t *sq = q2k_sq_row(w, expert, static_cast<int>(r));
            const int b = c >> 2, part = c & 3;
            const uint4 qv = *(reinterpret_cast<const uint4 *>(sq + b * 80 + 16) + part);
            const uint32_t scw = *(reinterpret_cast<const uint32_t *>(sq + b * 80) + part);
            const uint32_t ddw = q2k_dd_row(w, expert, static_cast<int>(r))[b];
            const float d = f16_to_f32(static_cast<uint16_t>(ddw & 0xffffu));
            const float dmin = f16_to_f32(static_cast<uint16_t>(ddw >> 16));
            for (int sub = 0; sub < 4; sub++) {
                const uint32_t sc = (scw >> (8 * sub)) & 15u, mn = (scw >> (8 * sub + 4)) & 15u;
                const float ds = __fmul_rn(d, static_cast<float>(sc));
                const float dm = __fmul_rn(dmin, static_cast<float>(mn));
                const uint32_t qw = sub == 0 ? qv.x : sub == 1 ? qv.y : sub == 2 ? qv.z : qv.w;
                for (int i = 0; i < 16; i++) v[16 * sub + i] = q2k_weight(ds, dm, (qw >> (2 * i)) & 3u);
            }
        } else {
            const int m = matrix == DS4MOE_GATE ? 0 : 1;
            const uint8_t *qs = iq2_qs_row(w, m, expert, static_cast<int>(r));
            const uint16_t *dp = iq2_d_row(w, m, expert, static_cast<int>(r));
            const uint4 q = *(reinterpret_cast<const uint4 *>(qs) + (c ^ iq2_swz(w, static_cast<int>(r))));
            const float d = f16_to_f32(dp[c >> 2]);
            for (int sb = 0; sb < 2; sb++) {
                const uint32_t iw = sb ? q.z : q.x, sw = sb ? q.w : q.y;
                const float sc = iq2_scale(d, sw);
                for (int g = 0; g < 4; g++) {
                    const uint2 ge = reinterpret_cast<const uint2 *>(grid)[(iw >> (8 * g)) & 255u];
                    iq2_group(ge, (sw >> (7 * g)) & 127u, sc, v + 32 * sb + 8 * g);
                }
            }
        }
        const size_t o = r * cols + static_cast<size_t>(c) * 64;
        for (int i = 0; i < 64; i++) {
            if (dst32) dst32[o + i] = v[i];
            if (dst16) dst16[o + i] = __half_as_ushort(__float2half_rn(v[i]));
        }
    }
}

// ------------------------------------------------------------------ one token, 4-bit: streamed
//
// A single token reads every byte once and does little arithmetic per byte, so the kernels
// above leave their warps waiting on loads. These two keep the loads off the compute warps: one
// producer warp bulk-copies each item's packed rows (and, for down, the item's h) into a ring
// of shared-memory stages, and two groups of eight compute warps decode and dot from shared
// memory, the groups taking the items in turn. Each group has stages of its own (stage
// g + G*i, i < S/G, for group g of G) and is their only consumer, so it never waits for a phase
// more than one ahead of the last it consumed (a parity wait cannot tell those apart). One CTA
// per SM; items are split over the CTAs by bytes as above. Every wait is bounded; a warp that
// gives up keeps its barrier arrivals without computing, so the CTA always finishes, and the
// producer lets all its copies land before it exits.

constexpr int kSWarps = 8;                               // compute warps per group
constexpr int kSGroups = 2;                              // groups, taking items in turn
constexpr int kSThreads = 32 * (kSGroups * kSWarps + 1);  // and one producer warp
constexpr int kSStageMax = 65536;              // bytes of one ring stage at most
constexpr int kSMaxStages = 6;
constexpr int kSDownRows = 32;                 // routed down rows per item (four per warp)
constexpr int kSDownSharedRows = 8;            // shared down rows per item (one per warp)

struct StreamCfg {
    int stage_bytes;  // one ring stage (multiple of 128)
    int stages;       // ring depth
    int sh_rows;      // shared gate/up rows per item (a power of two dividing kSWarps)
    int ring_off;     // the x / table region follows the ring at this offset
};

// Phase 1 for one token: item = 8 rows of gate and of up of one routed expert (one row per
// warp), or sh_rows bf16 rows of the shared gate and up (8 / sh_rows warps per row, each a
// column range; the row's first warp adds the partial sums).
__global__ void __launch_bounds__(kSThreads, 1) gemv_up_stream_kernel(UpParams p, StreamCfg cfg) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int D = p.w.D, F = p.w.F, nbD = p.w.nbD, D8 = D / 8;
    const int row_bytes = nbD * 144;
    uint8_t *ring = smem;
    uint4 *xs = reinterpret_cast<uint4 *>(smem + cfg.ring_off);  // bf16 x [D]
    uint4 *xq_raw = xs + D8;                                     // int16 pairs as prepared [D/8]
    uint4 *xqs = xq_raw + D8;                                    // the same, swizzled
    int *x8s = reinterpret_cast<int *>(xqs + D8);                // [D/32]
    uint64_t *bars = reinterpret_cast<uint64_t *>(x8s + D / 32);  // full[S], empty[S], xbar
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 2 * cfg.stages + 1);
    float *part = reinterpret_cast<float *>(bars + 2 * cfg.stages + 2);  // [kSGroups][2][kSWarps][2]
    // per stage: the h row of the item's pair, written by the producer before it arms the stage
    int *info = reinterpret_cast<int *>(part + kSGroups * 2 * kSWarps * 2);
    const int S = cfg.stages, SB = cfg.stage_bytes;
    auto full = [&](int s) { return smem_u32(bars + s); };
    auto empty = [&](int s) { return smem_u32(bars + S + s); };
    const uint32_t xbar = smem_u32(bars + 2 * S);
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int cg = wid / kSWarps, warp = wid - cg * kSWarps;  // compute group, warp within it

    const int n_gemv = p.meta->n_gemv;
    const int per_group = F / kSWarps;
    const int routed = n_gemv * per_group;
    const int n_shared = p.shared ? F / cfg.sh_rows : 0;
    const long long cr = 2LL * kSWarps * 144, cs = 2LL * cfg.sh_rows * 512;  // bytes per 256 columns
    int begin, end;
    cta_range(routed, n_shared, cr, cs, begin, end);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; s++) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), kSWarps);
        }
        mbar_init(xbar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (cg == kSGroups) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            const uint32_t xbytes = static_cast<uint32_t>(D * 2 + D * 2 + D / 32 * 4);
            mbar_expect_tx(xbar, xbytes);
            bulk_load(smem_u32(xs), p.x, D * 2, xbar);
            bulk_load(smem_u32(xq_raw), p.xq, D * 2, xbar);
            bulk_load(smem_u32(x8s), p.x8, D / 32 * 4, xbar);
            const int SG = S / kSGroups;  // stages per group
            int issued[kSMaxStages];
            for (int s = 0; s < kSMaxStages; s++) issued[s] = -1;
            for (int item = begin; item < end; item++) {
                const int j = item - begin, q = j / kSGroups;
                const int stage = j - q * kSGroups + kSGroups * (q % SG);  // group j % G, its q-th item
                const uint32_t phase = static_cast<uint32_t>(q / SG) & 1u;  // the stage's fill parity
                if (!wait_phase(empty(stage), phase ^ 1u, abort_flag, p.status) || *abort_flag) break;
                const uint32_t dst = smem_u32(ring + stage * SB);
                if (item < routed) {
                    const int e = p.gemv_list[item / per_group], r0 = (item % per_group) * kSWarps;
                    const uint32_t nb = static_cast<uint32_t>(kSWarps * row_bytes);
                    info[4 * stage] = p.offsets[e];  // visible to the group through the stage's barrier
                    mbar_expect_tx(full(stage), 2 * nb);
                    bulk_load(dst, q4_row(p.w, 0, e, r0), nb, full(stage));
                    bulk_load(dst + nb, q4_row(p.w, 1, e, r0), nb, full(stage));
                } else {
                    const int r0 = (item - routed) * cfg.sh_rows;
                    const uint32_t nb = static_cast<uint32_t>(cfg.sh_rows * D * 2);
                    mbar_expect_tx(full(stage), 2 * nb);
                    bulk_load(dst, p.w.sh_gate + static_cast<size_t>(r0) * D, nb, full(stage));
                    bulk_load(dst + nb, p.w.sh_up + static_cast<size_t>(r0) * D, nb, full(stage));
                }
                issued[stage] = static_cast<int>(phase);
            }
            // every copy lands before the CTA can exit, whatever the compute warps did
            mbar_drain(xbar, 0);
            for (int s = 0; s < S; s++)
                if (issued[s] >= 0) mbar_drain(full(s), static_cast<uint32_t>(issued[s]));
        }
        return;
    }

    // -------------------------------------------------------------- compute warps
    bool ok = wait_phase(xbar, 0, abort_flag, p.status);
    if (ok)
        for (int i = threadIdx.x; i < D8; i += kSGroups * kSWarps * 32) xqs[swz8(i)] = xq_raw[i];
    bar_sync(kSGroups + 1, kSGroups * kSWarps * 32);
    const float xf = p.xsc[0].x;  // the int16 token's factor back to x
    const int nsub = nbD * 8;
    const int wpr = kSWarps / cfg.sh_rows, cols8 = D8 / wpr;  // shared items: warps per row, chunks per warp
    for (int item = begin + cg; item < end; item += kSGroups) {
        const int q = (item - begin) / kSGroups;  // this group's q-th item
        const int stage = cg + kSGroups * (q % (S / kSGroups));
        const uint32_t phase = static_cast<uint32_t>(q / (S / kSGroups)) & 1u;
        ok = ok && wait_phase(full(stage), phase, abort_flag, p.status);
        const uint8_t *st = ring + stage * SB;
        if (item < routed) {
            if (ok) {
                const int off = info[4 * stage];  // the pair's h row (set by the producer)
                const int r = (item % per_group) * kSWarps + warp;
                const uint8_t *rg = st + warp * row_bytes, *ru = st + (kSWarps + warp) * row_bytes;
                float ag[2] = {0.0f, 0.0f}, au[2] = {0.0f, 0.0f};
                // two sub-blocks per lane at a time and one dp2a chain per 8-weight group (the
                // integer sums are exact in any order): independent work for the scheduler
                for (int c0 = lane; c0 < nsub; c0 += 64) {
#pragma unroll
                    for (int t = 0; t < 2; t++) {
                        const int c = c0 + 32 * t;
                        if (c >= nsub) break;
                        const int b = c >> 3, sub = c & 7;
                        const uint4 hg = *reinterpret_cast<const uint4 *>(rg + b * 144);
                        const uint4 hu = *reinterpret_cast<const uint4 *>(ru + b * 144);
                        const uint4 vg = *(reinterpret_cast<const uint4 *>(rg + b * 144 + 16) + sub);
                        const uint4 vu = *(reinterpret_cast<const uint4 *>(ru + b * 144 + 16) + sub);
                        float dsg, dmg, dsu, dmu;
                        q4_sub_scale(hg, sub, dsg, dmg);
                        q4_sub_scale(hu, sub, dsu, dmu);
                        int sgp[4], sup[4];
#pragma unroll
                        for (int g = 0; g < 4; g++) {
                            const uint32_t wgw = g == 0 ? vg.x : g == 1 ? vg.y : g == 2 ? vg.z : vg.w;
                            const uint32_t wuw = g == 0 ? vu.x : g == 1 ? vu.y : g == 2 ? vu.z : vu.w;
                            const uint4 xv = xqs[swz8(4 * c + g)];
                            const uint32_t eg = wgw & 0x0F0F0F0Fu, og = (wgw >> 4) & 0x0F0F0F0Fu;
                            const uint32_t eu = wuw & 0x0F0F0F0Fu, ou = (wuw >> 4) & 0x0F0F0F0Fu;
                            sgp[g] = dp2a_hi_su(xv.w, og, dp2a_lo_su(xv.z, og, dp2a_hi_su(xv.y, eg, dp2a_lo_su(xv.x, eg, 0))));
                            sup[g] = dp2a_hi_su(xv.w, ou, dp2a_lo_su(xv.z, ou, dp2a_hi_su(xv.y, eu, dp2a_lo_su(xv.x, eu, 0))));
                        }
                        const int sg = (sgp[0] + sgp[1]) + (sgp[2] + sgp[3]);
                        const int su = (sup[0] + sup[1]) + (sup[2] + sup[3]);
                        const float sx = static_cast<float>(x8s[c] >> 3);  // sum of the sub-block's 32 int16 x
                        ag[t] = fmaf(dsg, static_cast<float>(sg), fmaf(-dmg, sx, ag[t]));
                        au[t] = fmaf(dsu, static_cast<float>(su), fmaf(-dmu, sx, au[t]));
                    }
                }
                const float g = warp_sum(ag[0] + ag[1]) * xf, u = warp_sum(au[0] + au[1]) * xf;
                if (lane == 0) p.h[static_cast<size_t>(off) * F + r] = swiglu(g, u);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty(stage));
        } else {
            const int row = warp / wpr, q = warp - row * wpr;
            float g = 0.0f, u = 0.0f;
            if (ok) {
                const uint4 *sg = reinterpret_cast<const uint4 *>(st + static_cast<size_t>(row) * D * 2) + q * cols8;
                const uint4 *su = reinterpret_cast<const uint4 *>(st + static_cast<size_t>(cfg.sh_rows + row) * D * 2) + q * cols8;
                const uint4 *xr = xs + q * cols8;
                for (int c = lane; c < cols8; c += 32) {
                    float wg[8], wu[8];
                    bf16x8(sg[c], wg);
                    bf16x8(su[c], wu);
                    const uint4 xv = xr[c];
                    dot8_bf16(wg, xv, g);
                    dot8_bf16(wu, xv, u);
                }
                g = warp_sum(g);
                u = warp_sum(u);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty(stage));
            // two buffers per group: one barrier per item suffices
            float *pp = part + (cg * 2 + (((item - begin) / kSGroups) & 1)) * 2 * kSWarps;
            if (lane == 0) {
                pp[2 * warp] = g;
                pp[2 * warp + 1] = u;
            }
            bar_sync(1 + cg, kSWarps * 32);
            if (q == 0 && lane == 0 && ok) {
                float G = 0.0f, U = 0.0f;
                for (int i = 0; i < wpr; i++) {
                    G += pp[2 * (warp + i)];
                    U += pp[2 * (warp + i) + 1];
                }
                p.h[static_cast<size_t>(p.P) * F + (item - routed) * cfg.sh_rows + row] = swiglu(G, U);
            }
        }
    }
}

// Phase 2 for one token: item = 32 rows of one routed expert's down (four per warp) with the
// pair's int16 h, or 8 bf16 rows of the shared down (one per warp) with the fp32 shared h.
__global__ void __launch_bounds__(kSThreads, 1) gemv_down_stream_kernel(DownParams p, StreamCfg cfg) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int D = p.w.D, F = p.w.F, nbF = p.w.nbF, F8 = F / 8;
    const int row_bytes = nbF * 144;
    const uint32_t wbytes = static_cast<uint32_t>(kSDownRows * row_bytes);  // a routed item's rows
    const uint32_t sbytes = static_cast<uint32_t>(kSDownSharedRows * F * 2);  // a shared item's rows
    uint8_t *ring = smem;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + cfg.ring_off);  // full[S], empty[S]
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 2 * cfg.stages);
    // per stage: the pair's y row and h factor, written by the producer before it arms the stage
    int *info = reinterpret_cast<int *>(bars + 2 * cfg.stages + 1);
    const int S = cfg.stages, SB = cfg.stage_bytes;
    auto full = [&](int s) { return smem_u32(bars + s); };
    auto empty = [&](int s) { return smem_u32(bars + S + s); };
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int cg = wid / kSWarps, warp = wid - cg * kSWarps;  // compute group, warp within it

    const int n_gemv = p.meta->n_gemv;
    const int per_group = D / kSDownRows;
    const int routed = n_gemv * per_group;
    const int n_shared = p.shared ? D / kSDownSharedRows : 0;
    const long long cr = static_cast<long long>(kSDownRows) * 144, cs = kSDownSharedRows * 512LL;
    int begin, end;
    cta_range(routed, n_shared, cr, cs, begin, end);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; s++) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), kSWarps);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (cg == kSGroups) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            const int SG = S / kSGroups;  // stages per group
            int issued[kSMaxStages];
            for (int s = 0; s < kSMaxStages; s++) issued[s] = -1;
            for (int item = begin; item < end; item++) {
                const int j = item - begin, q = j / kSGroups;
                const int stage = j - q * kSGroups + kSGroups * (q % SG);  // group j % G, its q-th item
                const uint32_t phase = static_cast<uint32_t>(q / SG) & 1u;  // the stage's fill parity
                if (!wait_phase(empty(stage), phase ^ 1u, abort_flag, p.status) || *abort_flag) break;
                const uint32_t dst = smem_u32(ring + stage * SB);
                if (item < routed) {  // rows, then the pair's int16 h and its sub-block sums
                    const int e = p.gemv_list[item / per_group], r0 = (item % per_group) * kSDownRows;
                    const int off = p.offsets[e];
                    info[4 * stage] = off;  // visible to the group through the stage's barrier
                    info[4 * stage + 1] = __float_as_int(p.hsc[off]);
                    mbar_expect_tx(full(stage), wbytes + F * 2 + F / 32 * 4);
                    bulk_load(dst, q4_row(p.w, 2, e, r0), wbytes, full(stage));
                    bulk_load(dst + wbytes, p.hq + static_cast<size_t>(off) * F8, F * 2, full(stage));
                    bulk_load(dst + wbytes + F * 2, p.hsum + static_cast<size_t>(off) * (F / 32), F / 32 * 4, full(stage));
                } else {  // rows, then the shared h (fp32)
                    const int r0 = (item - routed) * kSDownSharedRows;
                    mbar_expect_tx(full(stage), sbytes + F * 4);
                    bulk_load(dst, p.w.sh_down + static_cast<size_t>(r0) * F, sbytes, full(stage));
                    bulk_load(dst + sbytes, p.h + static_cast<size_t>(p.P) * F, F * 4, full(stage));
                }
                issued[stage] = static_cast<int>(phase);
            }
            // every copy lands before the CTA can exit, whatever the compute warps did
            for (int s = 0; s < S; s++)
                if (issued[s] >= 0) mbar_drain(full(s), static_cast<uint32_t>(issued[s]));
        }
        return;
    }

    // -------------------------------------------------------------- compute warps
    bool ok = true;
    const int nsub = nbF * 8;
    for (int item = begin + cg; item < end; item += kSGroups) {
        const int q = (item - begin) / kSGroups;  // this group's q-th item
        const int stage = cg + kSGroups * (q % (S / kSGroups));
        const uint32_t phase = static_cast<uint32_t>(q / (S / kSGroups)) & 1u;
        ok = ok && wait_phase(full(stage), phase, abort_flag, p.status);
        const uint8_t *st = ring + stage * SB;
        if (ok && item < routed) {
            const int r0 = (item % per_group) * kSDownRows;
            const int off = info[4 * stage];  // the pair's y row and h factor (set by the producer)
            const float hf = __int_as_float(info[4 * stage + 1]);
            const uint4 *hq = reinterpret_cast<const uint4 *>(st + wbytes);
            const int *hsum = reinterpret_cast<const int *>(st + wbytes + F * 2);
#pragma unroll 1
            for (int rr = 0; rr < kSDownRows / kSWarps; rr++) {
                const int rl = warp + rr * kSWarps;  // row within the item
                const uint8_t *rd = st + rl * row_bytes;
                float accs[2] = {0.0f, 0.0f};
                for (int c0 = lane; c0 < nsub; c0 += 64) {  // two sub-blocks per lane at a time
#pragma unroll
                    for (int t = 0; t < 2; t++) {
                    const int c = c0 + 32 * t;
                    if (c >= nsub) break;
                    const int b = c >> 3, sub = c & 7;
                    const uint4 hd = *reinterpret_cast<const uint4 *>(rd + b * 144);
                    const uint4 vd = *(reinterpret_cast<const uint4 *>(rd + b * 144 + 16) + sub);
                    float ds, dm;
                    q4_sub_scale(hd, sub, ds, dm);
                    // the four 8-weight groups in an order rotated by (c >> 1) & 3, so the lanes of a
                    // quarter warp read eight different bank groups of h (the integer sum is exact)
                    const int rot = (c >> 1) & 3;
                    uint4 w4 = vd;
                    if (rot & 1) w4 = make_uint4(w4.y, w4.z, w4.w, w4.x);
                    if (rot & 2) w4 = make_uint4(w4.z, w4.w, w4.x, w4.y);
                    int sdp[4];  // one dp2a chain per 8-weight group (exact integer sums)
#pragma unroll
                    for (int g = 0; g < 4; g++) {
                        const uint32_t wd = g == 0 ? w4.x : g == 1 ? w4.y : g == 2 ? w4.z : w4.w;
                        const uint32_t ev = wd & 0x0F0F0F0Fu, ov = (wd >> 4) & 0x0F0F0F0Fu;
                        const uint4 hv = hq[4 * c + ((g + rot) & 3)];
                        sdp[g] = dp2a_hi_su(hv.w, ov, dp2a_lo_su(hv.z, ov, dp2a_hi_su(hv.y, ev, dp2a_lo_su(hv.x, ev, 0))));
                    }
                    const int sd = (sdp[0] + sdp[1]) + (sdp[2] + sdp[3]);
                    accs[t] = fmaf(ds, static_cast<float>(sd), fmaf(-dm, static_cast<float>(hsum[c]), accs[t]));
                    }
                }
                const float v = warp_sum(accs[0] + accs[1]) * hf;
                if (lane == 0) p.y[static_cast<size_t>(off) * D + r0 + rl] = v;
            }
        } else if (ok) {
            const int r = (item - routed) * kSDownSharedRows + warp;
            const uint4 *sd = reinterpret_cast<const uint4 *>(st + static_cast<size_t>(warp) * F * 2);
            const float4 *hs = reinterpret_cast<const float4 *>(st + sbytes);
            float acc = 0.0f;
            for (int c = lane; c < F8; c += 32) {
                float wv[8];
                bf16x8(sd[c], wv);
                acc = dot4(make_float4(wv[0], wv[1], wv[2], wv[3]), hs[2 * c], acc);
                acc = dot4(make_float4(wv[4], wv[5], wv[6], wv[7]), hs[2 * c + 1], acc);
            }
            const float v = warp_sum(acc);
            if (lane == 0) p.y[static_cast<size_t>(p.P) * D + r] = v;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty(stage));
    }
}

int sm_count() {
    static int n = 0;
    if (!n) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 148;
    }
    return n;
}

// CTAs of a kernel resident on one SM at once (registers, shared memory, threads), so the
// grid is one wave. Cached for the last shared-memory size asked.
template <class Kernel>
int resident_ctas(Kernel kernel, size_t smem, int &cached_smem, int &cached_n) {
    if (cached_smem != static_cast<int>(smem)) {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kThreads, smem) != cudaSuccess || n < 1) n = 1;
        cached_n = n;
        cached_smem = static_cast<int>(smem);
    }
    return cached_n;
}

template <int NT, bool Q4>
int launch_up_nt(const UpParams &p, cudaStream_t s) {
    static int seen[64];
    const size_t smem = 2048 + static_cast<size_t>(NT) * p.w.D * 2 +
                        (Q4 ? static_cast<size_t>(NT) * (p.w.D * 2 + p.w.D / 32 * 4 + 4) : 0);
    static int cached_smem = -1, cached_n = 0;
    const int err = ensure_smem(reinterpret_cast<const void *>(gemv_up_kernel<NT, Q4>), static_cast<int>(smem), seen);
    if (err) return err;
    const int per_sm = resident_ctas(gemv_up_kernel<NT, Q4>, smem, cached_smem, cached_n);
    return launch_pdl(gemv_up_kernel<NT, Q4>, dim3(sm_count() * per_sm), dim3(kThreads), smem, s, p);
}

template <int NT, bool Q4>
int launch_down_nt(const DownParams &p, cudaStream_t s) {
    static int seen[64];
    const size_t smem = static_cast<size_t>(NT) * p.w.F * 4 +
                        (Q4 ? static_cast<size_t>(NT) * (p.w.F * 2 + p.w.F / 32 * 4 + 4) : 0);
    static int cached_smem = -1, cached_n = 0;
    const int err = ensure_smem(reinterpret_cast<const void *>(gemv_down_kernel<NT, Q4>), static_cast<int>(smem), seen);
    if (err) return err;
    const int per_sm = resident_ctas(gemv_down_kernel<NT, Q4>, smem, cached_smem, cached_n);
    return launch_pdl(gemv_down_kernel<NT, Q4>, dim3(sm_count() * per_sm), dim3(kThreads), smem, s, p);
}

// Ring plans of the streamed kernels; stages == 0 when they do not fit one CTA's shared memory.
constexpr size_t kSmemLimit = 227 * 1024;

StreamCfg plan_up_stream(const DeviceWeights &w, size_t &smem) {
    StreamCfg c{0, 0, 0, 0};
    const size_t D = static_cast<size_t>(w.D);
    // stages as small as a routed item, so that more of them are in flight: shared items of as
    // many rows as fit one (at least one)
    const size_t routed = 2ull * kSWarps * w.nbD * 144;
    int sh = kSWarps;
    while (sh > 1 && 2 * sh * D * 2 > routed) sh >>= 1;
    const size_t shared = 2ull * sh * D * 2;
    const size_t stage = ((routed > shared ? routed : shared) + 127) / 128 * 128;
    if (stage > static_cast<size_t>(kSStageMax) || 2 * sh * D * 2 > static_cast<size_t>(kSStageMax)) return c;
    // x as bf16, as int16 pairs twice (as prepared, swizzled), the sub-block sums, barriers, partial sums
    const size_t fixed = 6 * D + D / 8 + (2 * kSMaxStages + 2) * 8 + kSGroups * 2 * kSWarps * 2 * 4 + kSMaxStages * 16;
    int S = kSMaxStages / kSGroups * kSGroups;  // a multiple of the groups: each has S / G stages
    while (S >= kSGroups && S * stage + fixed > kSmemLimit) S -= kSGroups;
    if (S < kSGroups) return c;
    c.stage_bytes = static_cast<int>(stage);
    c.stages = S;
    c.sh_rows = sh;
    c.ring_off = static_cast<int>(S * stage);
    smem = S * stage + fixed;
    return c;
}

StreamCfg plan_down_stream(const DeviceWeights &w, size_t &smem) {
    StreamCfg c{0, 0, 0, 0};
    const size_t F = static_cast<size_t>(w.F);
    const size_t routed = static_cast<size_t>(kSDownRows) * w.nbF * 144 + F * 2 + F / 32 * 4;
    const size_t shared = static_cast<size_t>(kSDownSharedRows) * F * 2 + F * 4;
    const size_t stage = ((routed > shared ? routed : shared) + 127) / 128 * 128;
    if (stage > static_cast<size_t>(kSStageMax) || F % 128 != 0) return c;
    const size_t fixed = (2 * kSMaxStages + 1) * 8 + 8 + kSMaxStages * 16;
    int S = kSMaxStages / kSGroups * kSGroups;  // a multiple of the groups: each has S / G stages
    while (S >= kSGroups && S * stage + fixed > kSmemLimit) S -= kSGroups;
    if (S < kSGroups) return c;
    c.stage_bytes = static_cast<int>(stage);
    c.stages = S;
    c.sh_rows = kSDownSharedRows;
    c.ring_off = static_cast<int>(S * stage);
    smem = S * stage + fixed;
    return c;
}

int launch_up_stream(const UpParams &p, const StreamCfg &c, size_t smem, cudaStream_t s) {
    static int seen[64];
    const int err = ensure_smem(reinterpret_cast<const void *>(gemv_up_stream_kernel), static_cast<int>(smem), seen);
    if (err) return err;
    gemv_up_stream_kernel<<<sm_count(), kSThreads, smem, s>>>(p, c);
    return static_cast<int>(cudaGetLastError());
}

int launch_down_stream(const DownParams &p, const StreamCfg &c, size_t smem, cudaStream_t s) {
    static int seen[64];
    const int err = ensure_smem(reinterpret_cast<const void *>(gemv_down_stream_kernel), static_cast<int>(smem), seen);
    if (err) return err;
    gemv_down_stream_kernel<<<sm_count(), kSThreads, smem, s>>>(p, c);
    return static_cast<int>(cudaGetLastError());
}

}  // namespace

int launch_gemv_up(const DeviceWeights &w, const Workspace &ws, const uint16_t *x, int T, int k, bool shared_on_gemv,
                   void *stream, const int32_t *shared_flag) {
    UpParams p;
    p.w = w;
    p.x = x;
    p.perm = ws.perm;
    p.offsets = ws.offsets;
    p.gemv_list = ws.gemv_list;
    p.meta = ws.meta;
    p.grid = ws.grid;
    p.h = ws.h32;
    p.T = T;
    p.k = k;
    p.P = T * k;
    p.shared = shared_on_gemv && w.has_shared;
    p.shared_flag = shared_flag;
    p.xq = reinterpret_cast<const uint4 *>(ws.xq);
    p.x8 = ws.x8;
    p.xsc = reinterpret_cast<const float4 *>(ws.xsc);
    p.status = ws.status;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (w.fmt == 1 && T == 1 && !shared_flag) {  // streamed when its ring fits and every copy source is 16-byte aligned
        size_t smem = 0;
        const StreamCfg c = plan_up_stream(w, smem);
        const bool aligned = ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(ws.xq) |
                               reinterpret_cast<uintptr_t>(ws.x8)) & 15u) == 0;
        if (c.stages > 0 && aligned) return launch_up_stream(p, c, smem, s);
    }
    if (w.fmt == 1) return T == 1 ? launch_up_nt<1, true>(p, s) : launch_up_nt<8, true>(p, s);
    return T == 1 ? launch_up_nt<1, false>(p, s) : launch_up_nt<8, false>(p, s);
}

int launch_prep_h(const Workspace &ws, int rows, int F, void *stream) {
    if (rows <= 0) return 0;
    return launch_pdl(prep_h_kernel, dim3(rows), dim3(256), 0, static_cast<cudaStream_t>(stream),
                      static_cast<const float *>(ws.h32), rows, F, reinterpret_cast<uint4 *>(ws.hq4), ws.hsum4, ws.hsc4);
}

int launch_gemv_down(const DeviceWeights &w, const Workspace &ws, int T, int k, bool shared_on_gemv, void *stream,
                     bool int16_h, const int32_t *shared_flag) {
    DownParams p;
    p.w = w;
    p.offsets = ws.offsets;
    p.gemv_list = ws.gemv_list;
    p.meta = ws.meta;
    p.h = ws.h32;
    p.y = ws.y;
    p.T = T;
    p.P = T * k;
    p.shared = shared_on_gemv && w.has_shared;
    p.shared_flag = shared_flag;
    p.hq = int16_h ? reinterpret_cast<const uint4 *>(ws.hq4) : nullptr;
    p.hsum = ws.hsum4;
    p.hsc = ws.hsc4;
    p.status = ws.status;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (w.fmt == 1 && T == 1 && int16_h) {  // streamed when its ring fits and every copy source is 16-byte aligned
        size_t smem = 0;
        const StreamCfg c = plan_down_stream(w, smem);
        const bool aligned = ((reinterpret_cast<uintptr_t>(ws.hq4) | reinterpret_cast<uintptr_t>(ws.hsum4) |
                               reinterpret_cast<uintptr_t>(ws.h32)) & 15u) == 0;
        if (c.stages > 0 && aligned) return launch_down_stream(p, c, smem, s);
    }
    if (w.fmt == 1) return T == 1 ? launch_down_nt<1, true>(p, s) : launch_down_nt<8, true>(p, s);
    return T == 1 ? launch_down_nt<1, false>(p, s) : launch_down_nt<8, false>(p, s);
}

int launch_dequant(const DeviceWeights &w, const uint8_t *grid, int expert, int matrix, float *dst32,
                   uint16_t *dst16, void *stream) {
    dequant_kernel<<<sm_count() * 4, 128, 0, static_cast<cudaStream_t>(stream)>>>(w, expert, matrix, grid, dst32,
                                                                                 dst16);
    return static_cast<int>(cudaGetLastError());
}

}  // namespace ds4moe
