// Single-token expert groups (every group at T = 1): fused dequant-GEMV kernels tuned for the instruction
// budget of streaming 2-bit rows at HBM speed.
//
// "DwarfStar" README, "运行大于 RAM 的模型": every new token is routed through the experts
// again, so each decode step streams the selected experts' packed rows once. At one token
// the rows are read once and used once, so the kernels are bound by HBM bandwidth and by
// the instructions spent decoding each weight. Design points:
//   * each warp owns a few weight rows; lane l covers 64 consecutive columns of every
//     2048-column phase, so its slice of x sits in registers for all rows of the item;
//   * IQ2-style rows: x is held as fp16x2, scaled per phase by a power of two so that every
//     partial sum stays far inside fp16 range; the grid entry is fetched as the fp16 high
//     bytes of its magnitudes (1, 3, 5, 7 have zero low bytes), the 8 signs are spread into
//     the fp16 sign bits with two multiplies, and 4 HFMA2 accumulate a group; G*x is exact
//     in fp16 (3 + 8 significant bits), the sub-block sum is folded into fp32 with its scale;
//   * Q2_K-style rows: sum q*h - dm*sum h per 16-weight sub-block; each code byte is mapped
//     by a shared-memory table to its four fp16 codes, 2 HFMA2 per byte;
//   * the bf16 shared expert: fp32 FFMA on exact bf16 -> fp32 weights;
//   * lookup tables are replicated per half-warp lane so random indices never collide on
//     a shared-memory bank.
#include <cuda_runtime.h>

#include "common.cuh"

namespace ds4moe {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRW = 4;    // routed rows per warp item
constexpr int kSRW = 1;   // shared-expert rows per warp item
constexpr int kSPhase = 1024; // columns per register phase of bf16 rows (32 per lane)

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }
__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }

// Power-of-two scale s with max|v| * s in [0.5, 1) (1 for an all-zero slice); returns 1/s too.
__device__ __forceinline__ void pow2_scale(float amax, float &s, float &inv) {
    int e = 0;
    frexpf(amax, &e);  // amax = m * 2^e, m in [0.5, 1)
    e = amax > 0.0f ? e : 0;
    s = ldexpf(1.0f, -e);
    inv = ldexpf(1.0f, e);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// One group of 8 IQ2-style weights dotted with 8 fp16 x values (4 half2), accumulated.
// ent: fp16 high bytes of the grid magnitudes; s7: the 7 stored sign bits.
__device__ __forceinline__ __half2 iq2_group_dot(uint2 ent, uint32_t s7, const uint32_t *xv, __half2 acc) {
    const uint32_t m_lo = s7 * 0x10204080u;                        // bits 0..3 -> 7, 15, 23, 31
    const uint32_t m_hi = s7 * 0x01020408u + (__popc(s7) << 31);   // bits 4..6 -> 7, 15, 23; parity -> 31
    const uint32_t lo = ent.x ^ (m_lo & 0x80808080u);
    const uint32_t hi = ent.y ^ (m_hi & 0x80808080u);
    acc = __hfma2(u2h(__byte_perm(lo, 0u, 0x1404)), u2h(xv[0]), acc);
    acc = __hfma2(u2h(__byte_perm(lo, 0u, 0x3424)), u2h(xv[1]), acc);
    acc = __hfma2(u2h(__byte_perm(hi, 0u, 0x1404)), u2h(xv[2]), acc);
    acc = __hfma2(u2h(__byte_perm(hi, 0u, 0x3424)), u2h(xv[3]), acc);
    return acc;
}

__device__ __forceinline__ float hsum(__half2 a) {
    const float2 f = __half22float2(a);
    return f.x + f.y;
}

// fp16 high byte of magnitude m in {1, 3, 5, 7}
__device__ __forceinline__ uint32_t mag_hibyte(uint32_t m) {
    return m == 1u ? 0x3Cu : m == 3u ? 0x42u : m == 5u ? 0x45u : 0x47u;
}

struct DecParams {
    DeviceWeights w;
    const uint16_t *x;  // bf16 [T][D]
    const int32_t *offsets, *single_list, *perm;
    const GroupMeta *meta;
    const uint8_t *grid;
    float *h;  // [P+T][F]
    float *y;  // [P+T][D]
    int P, k;
    int shared;  // the shared expert of the single token (T = 1)
};

// ------------------------------------------------------------------ phase 1: gate/up + SwiGLU

__global__ void __launch_bounds__(kThreads) decode_up_kernel(DecParams p) {
    pdl_wait();
    __shared__ uint2 gtab[256 * 16];  // [entry][copy]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < 256 * 16; i += kThreads) {
        const int e = i >> 4;
        const uint8_t *g = p.grid + 8 * e;
        uint2 v;
        v.x = mag_hibyte(g[0]) | (mag_hibyte(g[1]) << 8) | (mag_hibyte(g[2]) << 16) | (mag_hibyte(g[3]) << 24);
        v.y = mag_hibyte(g[4]) | (mag_hibyte(g[5]) << 8) | (mag_hibyte(g[6]) << 16) | (mag_hibyte(g[7]) << 24);
        gtab[i] = v;
    }
    __syncthreads();
    const uint2 *gt = gtab + (lane & 15);
    const int D = p.w.D, F = p.w.F, nbD = p.w.nbD;
    const int nchunk = nbD * 4;  // 64-column chunks per row
    const int per_group = F / kRW;
    const int routed = p.meta->n_single * per_group;
    const int total = routed + (p.shared ? F / kSRW : 0);
    const int gw = blockIdx.x * kWarps + warp, W = gridDim.x * kWarps;

    for (int item = gw; item < total; item += W) {
        if (item < routed) {
            const int e = p.single_list[item / per_group];
            const int r0 = (item % per_group) * kRW;
            const int pos = p.offsets[e];
            const uint4 *xg = reinterpret_cast<const uint4 *>(p.x + static_cast<size_t>(p.perm[pos] / p.k) * D);
            float ag[kRW], au[kRW];
#pragma unroll
            for (int r = 0; r < kRW; r++) ag[r] = au[r] = 0.0f;
            for (int ph = 0; ph * 32 < nchunk; ph++) {
                const int c = ph * 32 + lane;
                const bool live = c < nchunk;
                // x slice: 64 bf16 -> scaled fp16x2
                uint32_t xh[32];
                float amax = 0.0f;
                uint4 xr[8];
#pragma unroll
                for (int j = 0; j < 8; j++) {
                    xr[j] = live ? __ldg(xg + 8 * c + j) : make_uint4(0, 0, 0, 0);
                    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(bf16_lo(xr[j].x)), fabsf(bf16_hi(xr[j].x))),
                                             fmaxf(fabsf(bf16_lo(xr[j].y)), fabsf(bf16_hi(xr[j].y)))));
                    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(bf16_lo(xr[j].z)), fabsf(bf16_hi(xr[j].z))),
                                             fmaxf(fabsf(bf16_lo(xr[j].w)), fabsf(bf16_hi(xr[j].w)))));
                }
                float xs, xinv;
                pow2_scale(warp_max(amax), xs, xinv);
#pragma unroll
                for (int j = 0; j < 8; j++) {
                    xh[4 * j + 0] = h2u(__floats2half2_rn(bf16_lo(xr[j].x) * xs, bf16_hi(xr[j].x) * xs));
                    xh[4 * j + 1] = h2u(__floats2half2_rn(bf16_lo(xr[j].y) * xs, bf16_hi(xr[j].y) * xs));
                    xh[4 * j + 2] = h2u(__floats2half2_rn(bf16_lo(xr[j].z) * xs, bf16_hi(xr[j].z) * xs));
                    xh[4 * j + 3] = h2u(__floats2half2_rn(bf16_lo(xr[j].w) * xs, bf16_hi(xr[j].w) * xs));
                }
                if (live) {
                    const int b = c >> 2;
                    uint4 qg[kRW], qu[kRW];
                    float dg[kRW], du[kRW];
#pragma unroll
                    for (int r = 0; r < kRW; r++) {
                        const int cs = c ^ iq2_swz(p.w, r0 + r);  // chunk c = 4 * b + part
                        qg[r] = __ldg(reinterpret_cast<const uint4 *>(iq2_qs_row(p.w, 0, e, r0 + r)) + cs);
                        qu[r] = __ldg(reinterpret_cast<const uint4 *>(iq2_qs_row(p.w, 1, e, r0 + r)) + cs);
                        dg[r] = f16_to_f32(__ldg(iq2_d_row(p.w, 0, e, r0 + r) + b)) * xinv;
                        du[r] = f16_to_f32(__ldg(iq2_d_row(p.w, 1, e, r0 + r) + b)) * xinv;
                    }
#pragma unroll
                    for (int r = 0; r < kRW; r++) {
#pragma unroll
                        for (int sb = 0; sb < 2; sb++) {
                            const uint32_t igw = sb ? qg[r].z : qg[r].x, sgw = sb ? qg[r].w : qg[r].y;
                            const uint32_t iuw = sb ? qu[r].z : qu[r].x, suw = sb ? qu[r].w : qu[r].y;
                            __half2 hg = __float2half2_rn(0.0f), hu = __float2half2_rn(0.0f);
#pragma unroll
                            for (int g = 0; g < 4; g++) {
                                const uint32_t *xv = xh + 16 * sb + 4 * g;
                                hg = iq2_group_dot(gt[((igw >> (8 * g)) & 255u) << 4], (sgw >> (7 * g)) & 127u, xv, hg);
                                hu = iq2_group_dot(gt[((iuw >> (8 * g)) & 255u) << 4], (suw >> (7 * g)) & 127u, xv, hu);
                            }
                            ag[r] = fmaf(iq2_scale(dg[r], sgw), hsum(hg), ag[r]);
                            au[r] = fmaf(iq2_scale(du[r], suw), hsum(hu), au[r]);
                        }
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < kRW; r++) {
                const float g = warp_sum(ag[r]), u = warp_sum(au[r]);
                if (lane == r) p.h[static_cast<size_t>(pos) * F + r0 + r] = swiglu(g, u);
            }
        } else {
            // shared expert of the single token, bf16 rows, fp32
            const uint4 *xg = reinterpret_cast<const uint4 *>(p.x);
            const int r0 = (item - routed) * kSRW;
            float ag[kSRW], au[kSRW];
#pragma unroll
            for (int r = 0; r < kSRW; r++) ag[r] = au[r] = 0.0f;
            for (int ph = 0; ph * kSPhase < D; ph++) {
                const int c0 = ph * kSPhase + 32 * lane;  // 32 columns of this lane
                if (c0 >= D) continue;
                float xf[32];
#pragma unroll
                for (int j = 0; j < 4; j++) {
                    const uint4 v = __ldg(xg + c0 / 8 + j);
                    xf[8 * j + 0] = bf16_lo(v.x); xf[8 * j + 1] = bf16_hi(v.x);
                    xf[8 * j + 2] = bf16_lo(v.y); xf[8 * j + 3] = bf16_hi(v.y);
                    xf[8 * j + 4] = bf16_lo(v.z); xf[8 * j + 5] = bf16_hi(v.z);
                    xf[8 * j + 6] = bf16_lo(v.w); xf[8 * j + 7] = bf16_hi(v.w);
                }
                uint4 wg[kSRW][4], wu[kSRW][4];
#pragma unroll
                for (int r = 0; r < kSRW; r++) {
                    const uint4 *sg = reinterpret_cast<const uint4 *>(p.w.sh_gate + static_cast<size_t>(r0 + r) * D + c0);
                    const uint4 *su = reinterpret_cast<const uint4 *>(p.w.sh_up + static_cast<size_t>(r0 + r) * D + c0);
#pragma unroll
                    for (int j = 0; j < 4; j++) {
                        wg[r][j] = __ldg(sg + j);
                        wu[r][j] = __ldg(su + j);
                    }
                }
#pragma unroll
                for (int r = 0; r < kSRW; r++) {
#pragma unroll
                    for (int j = 0; j < 4; j++) {
                        const uint32_t g4[4] = {wg[r][j].x, wg[r][j].y, wg[r][j].z, wg[r][j].w};
                        const uint32_t u4[4] = {wu[r][j].x, wu[r][j].y, wu[r][j].z, wu[r][j].w};
#pragma unroll
                        for (int i = 0; i < 4; i++) {
                            ag[r] = fmaf(bf16_lo(g4[i]), xf[8 * j + 2 * i], ag[r]);
                            ag[r] = fmaf(bf16_hi(g4[i]), xf[8 * j + 2 * i + 1], ag[r]);
                            au[r] = fmaf(bf16_lo(u4[i]), xf[8 * j + 2 * i], au[r]);
                            au[r] = fmaf(bf16_hi(u4[i]), xf[8 * j + 2 * i + 1], au[r]);
                        }
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < kSRW; r++) {
                const float g = warp_sum(ag[r]), u = warp_sum(au[r]);
                if (lane == r) p.h[static_cast<size_t>(p.P) * F + r0 + r] = swiglu(g, u);
            }
        }
    }
}

// ------------------------------------------------------------------ phase 2: down

__global__ void __launch_bounds__(kThreads) decode_down_kernel(DecParams p) {
    pdl_wait();
    __shared__ uint2 qtab[256 * 16];  // [code byte][copy]: four fp16 codes
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < 256 * 16; i += kThreads) {
        const uint32_t b = static_cast<uint32_t>(i >> 4);
        const uint32_t hq[4] = {0x0000u, 0x3C00u, 0x4000u, 0x4200u};  // fp16 of 0, 1, 2, 3
        qtab[i] = make_uint2(hq[b & 3] | (hq[(b >> 2) & 3] << 16), hq[(b >> 4) & 3] | (hq[(b >> 6) & 3] << 16));
    }
    __syncthreads();
    const uint2 *qt = qtab + (lane & 15);
    const int D = p.w.D, F = p.w.F, nbF = p.w.nbF;
    const int nchunk = nbF * 4;
    const int per_group = D / kRW;
    const int routed = p.meta->n_single * per_group;
    const int total = routed + (p.shared ? D / kSRW : 0);
    const int gw = blockIdx.x * kWarps + warp, W = gridDim.x * kWarps;

    for (int item = gw; item < total; item += W) {
        if (item < routed) {
            const int e = p.single_list[item / per_group];
            const int r0 = (item % per_group) * kRW;
            const int pos = p.offsets[e];
            const float4 *hg = reinterpret_cast<const float4 *>(p.h + static_cast<size_t>(pos) * F);
            float acc[kRW];
#pragma unroll
            for (int r = 0; r < kRW; r++) acc[r] = 0.0f;
            for (int ph = 0; ph * 32 < nchunk; ph++) {
                const int c = ph * 32 + lane;
                const bool live = c < nchunk;
                float hf[64];
                float amax = 0.0f;
#pragma unroll
                for (int j = 0; j < 16; j++) {
                    const float4 v = live ? __ldg(hg + 16 * c + j) : make_float4(0.f, 0.f, 0.f, 0.f);
                    hf[4 * j] = v.x; hf[4 * j + 1] = v.y; hf[4 * j + 2] = v.z; hf[4 * j + 3] = v.w;
                    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
                }
                float hs, hinv;
                pow2_scale(warp_max(amax), hs, hinv);
                uint32_t hh[32];
                float sh[4];
#pragma unroll
                for (int s = 0; s < 4; s++) {
                    float t = 0.0f;
#pragma unroll
                    for (int i = 0; i < 16; i++) t += hf[16 * s + i];
                    sh[s] = t;
                }
#pragma unroll
                for (int j = 0; j < 32; j++) hh[j] = h2u(__floats2half2_rn(hf[2 * j] * hs, hf[2 * j + 1] * hs));
                if (live) {
                    const int b = c >> 2, part = c & 3;
                    uint4 qv[kRW];
                    uint32_t scw[kRW], ddw[kRW];
#pragma unroll
                    for (int r = 0; r < kRW; r++) {
                        const uint8_t *sq = q2k_sq_row(p.w, e, r0 + r) + b * 80;
                        qv[r] = __ldg(reinterpret_cast<const uint4 *>(sq + 16) + part);
                        scw[r] = __ldg(reinterpret_cast<const uint32_t *>(sq) + part);
                        ddw[r] = __ldg(q2k_dd_row(p.w, e, r0 + r) + b);
                    }
#pragma unroll
                    for (int r = 0; r < kRW; r++) {
                        const float d = f16_to_f32(static_cast<uint16_t>(ddw[r] & 0xffffu));
                        const float dmin = f16_to_f32(static_cast<uint16_t>(ddw[r] >> 16));
#pragma unroll
                        for (int sub = 0; sub < 4; sub++) {
                            const uint32_t qw = sub == 0 ? qv[r].x : sub == 1 ? qv[r].y : sub == 2 ? qv[r].z : qv[r].w;
                            __half2 a = __float2half2_rn(0.0f);
#pragma unroll
                            for (int bb = 0; bb < 4; bb++) {
                                const uint2 q4 = qt[((qw >> (8 * bb)) & 255u) << 4];
                                a = __hfma2(u2h(q4.x), u2h(hh[8 * sub + 2 * bb]), a);
                                a = __hfma2(u2h(q4.y), u2h(hh[8 * sub + 2 * bb + 1]), a);
                            }
                            const uint32_t sc = (scw[r] >> (8 * sub)) & 15u, mn = (scw[r] >> (8 * sub + 4)) & 15u;
                            const float ds = d * static_cast<float>(sc) * hinv;
                            const float dm = dmin * static_cast<float>(mn);
                            acc[r] = fmaf(ds, hsum(a), acc[r]);
                            acc[r] = fmaf(-dm, sh[sub], acc[r]);
                        }
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < kRW; r++) {
                const float v = warp_sum(acc[r]);
                if (lane == r) p.y[static_cast<size_t>(pos) * D + r0 + r] = v;
            }
        } else {
            const int r0 = (item - routed) * kSRW;
            const float4 *hg = reinterpret_cast<const float4 *>(p.h + static_cast<size_t>(p.P) * F);
            float acc[kSRW];
#pragma unroll
            for (int r = 0; r < kSRW; r++) acc[r] = 0.0f;
            for (int ph = 0; ph * kSPhase < F; ph++) {
                const int c0 = ph * kSPhase + 32 * lane;
                if (c0 >= F) continue;
                float hf[32];
#pragma unroll
                for (int j = 0; j < 8; j++) {
                    const float4 v = __ldg(hg + c0 / 4 + j);
                    hf[4 * j] = v.x; hf[4 * j + 1] = v.y; hf[4 * j + 2] = v.z; hf[4 * j + 3] = v.w;
                }
                uint4 wv[kSRW][4];
#pragma unroll
                for (int r = 0; r < kSRW; r++) {
                    const uint4 *sd = reinterpret_cast<const uint4 *>(p.w.sh_down + static_cast<size_t>(r0 + r) * F + c0);
#pragma unroll
                    for (int j = 0; j < 4; j++) wv[r][j] = __ldg(sd + j);
                }
#pragma unroll
                for (int r = 0; r < kSRW; r++) {
#pragma unroll
                    for (int j = 0; j < 4; j++) {
                        const uint32_t w4[4] = {wv[r][j].x, wv[r][j].y, wv[r][j].z, wv[r][j].w};
#pragma unroll
                        for (int i = 0; i < 4; i++) {
                            acc[r] = fmaf(bf16_lo(w4[i]), hf[8 * j + 2 * i], acc[r]);
                            acc[r] = fmaf(bf16_hi(w4[i]), hf[8 * j + 2 * i + 1], acc[r]);
                        }
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < kSRW; r++) {
                const float v = warp_sum(acc[r]);
                if (lane == r) p.y[static_cast<size_t>(p.P) * D + r0 + r] = v;
            }
        }
    }
}

int sm_count_dec() {
    static int n = 0;
    if (!n) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 148;
    }
    return n;
}

DecParams make(const DeviceWeights &w, const Workspace &ws, const uint16_t *x, int T, int k, bool shared) {
    DecParams p;
    p.w = w;
    p.x = x;
    p.offsets = ws.offsets;
    p.single_list = ws.single_list;
    p.perm = ws.perm;
    p.meta = ws.meta;
    p.grid = ws.grid;
    p.h = ws.h32;
    p.y = ws.y;
    p.P = T * k;
    p.k = k;
    p.shared = shared && w.has_shared && T == 1;
    return p;
}

}  // namespace

int launch_decode_up(const DeviceWeights &w, const Workspace &ws, const uint16_t *x, int T, int k, bool shared,
                     void *stream) {
    return launch_pdl(decode_up_kernel, dim3(sm_count_dec() * 4), dim3(kThreads), 0, static_cast<cudaStream_t>(stream),
                      make(w, ws, x, T, k, shared));
}

int launch_decode_down(const DeviceWeights &w, const Workspace &ws, int T, int k, bool shared, void *stream) {
    return launch_pdl(decode_down_kernel, dim3(sm_count_dec() * 4), dim3(kThreads), 0, static_cast<cudaStream_t>(stream),
                      make(w, ws, nullptr, T, k, shared));
}

}  // namespace ds4moe
