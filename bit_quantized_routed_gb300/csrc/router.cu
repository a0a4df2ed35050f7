// Router logits in front of routing: logits[t][e] = sum_d x[t][d] * W[e][d] + bias[e], bf16 x and
// router weights, fp32 bias and sums.
//
// "DwarfStar 深度解析" §3.4.3 and the "DwarfStar" README, "模型权重": the router stays
// unquantised. The top-k that follows selects experts by comparing these fp32 values, so the
// summation order is fixed (and documented in the header): the columns are cut into 1024-column
// segments; in a segment, lane l of a warp adds, in increasing d, the products of the columns d with
// (d / 8) % 32 == l (one fp32 FMA chain; a bf16 x bf16 product is exact in fp32), and the 32 partial
// sums are combined by xor-shuffles 16, 8, 4, 2, 1; the segment sums are added in increasing order,
// then the bias. A CTA computes TT tokens x 4 experts with one warp per segment, so even one token
// spreads the router's bytes over E / 4 x (D / 1024) warps, each with all its loads in flight at once.
// Calls of 64 tokens or more (E a multiple of 128) run on the tensor cores instead (router_tc.cu).
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace ds4moe {
namespace {

constexpr int kEE = 4;       // experts per CTA
constexpr int kMaxSeg = 8;   // d_model <= 8192

__device__ __forceinline__ void fma8(float &acc, const uint4 xv, const uint4 wv) {
    const uint32_t xs[4] = {xv.x, xv.y, xv.z, xv.w}, ws[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
    for (int q = 0; q < 4; q++) {  // columns in increasing order
        acc = __fmaf_rn(bf16_lo(xs[q]), bf16_lo(ws[q]), acc);
        acc = __fmaf_rn(bf16_hi(xs[q]), bf16_hi(ws[q]), acc);
    }
}

template <int TT>
__global__ void __launch_bounds__(kMaxSeg * 32) router_kernel(const uint16_t *__restrict__ x,
                                                              const uint16_t *__restrict__ w,
                                                              const float *__restrict__ bias, int T, int D, int E,
                                                              float *__restrict__ logits) {
    __shared__ float part[kMaxSeg][TT][kEE];
    const int lane = threadIdx.x & 31, seg = threadIdx.x >> 5, nseg = blockDim.x >> 5;
    const int egroups = E / kEE;
    const int t0 = (blockIdx.x / egroups) * TT, e0 = (blockIdx.x % egroups) * kEE;
    const int nb = D / 256, b0 = seg * 4, b1 = min(b0 + 4, nb);  // this segment's 256-column blocks
    const uint4 *xr[TT];
#pragma unroll
    for (int i = 0; i < TT; i++)
        xr[i] = reinterpret_cast<const uint4 *>(x + static_cast<size_t>(min(t0 + i, T - 1)) * D) + lane;
    const uint4 *wr = reinterpret_cast<const uint4 *>(w + static_cast<size_t>(e0) * D) + lane;
    float acc[TT][kEE];
#pragma unroll
    for (int i = 0; i < TT; i++)
#pragma unroll
        for (int e = 0; e < kEE; e++) acc[i][e] = 0.0f;
    if constexpr (TT == 1) {  // the whole segment's loads in flight at once
        uint4 xv[4], wv[4][kEE];
#pragma unroll
        for (int s = 0; s < 4; s++)
            if (b0 + s < b1) {
                xv[s] = __ldg(xr[0] + 32 * (b0 + s));
#pragma unroll
                for (int e = 0; e < kEE; e++) wv[s][e] = __ldg(wr + static_cast<size_t>(e) * (D / 8) + 32 * (b0 + s));
            }
#pragma unroll
        for (int s = 0; s < 4; s++)
            if (b0 + s < b1)
#pragma unroll
                for (int e = 0; e < kEE; e++) fma8(acc[0][e], xv[s], wv[s][e]);
    } else {
        for (int b = b0; b < b1; b++) {
            uint4 xv[TT], wv[kEE];
#pragma unroll
            for (int i = 0; i < TT; i++) xv[i] = __ldg(xr[i] + 32 * b);
#pragma unroll
            for (int e = 0; e < kEE; e++) wv[e] = __ldg(wr + static_cast<size_t>(e) * (D / 8) + 32 * b);
#pragma unroll
            for (int i = 0; i < TT; i++)
#pragma unroll
                for (int e = 0; e < kEE; e++) fma8(acc[i][e], xv[i], wv[e]);
        }
    }
#pragma unroll
    for (int i = 0; i < TT; i++)
#pragma unroll
        for (int e = 0; e < kEE; e++) {
            float v = acc[i][e];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
            if (lane == 0) part[seg][i][e] = v;
        }
    __syncthreads();
    if (threadIdx.x < TT * kEE) {
        const int i = threadIdx.x / kEE, e = threadIdx.x % kEE;
        if (t0 + i < T) {
            float v = part[0][i][e];
            for (int g = 1; g < nseg; g++) v = __fadd_rn(v, part[g][i][e]);
            if (bias) v = __fadd_rn(v, bias[e0 + e]);
            logits[static_cast<size_t>(t0 + i) * E + e0 + e] = v;
        }
    }
}

template <int TT>
int launch_tt(const uint16_t *x, const uint16_t *w, const float *bias, int T, int D, int E, float *logits,
              cudaStream_t s) {
    const int blocks = ((T + TT - 1) / TT) * (E / kEE);
    const int nseg = (D / 256 + 3) / 4;
    router_kernel<TT><<<blocks, nseg * 32, 0, s>>>(x, w, bias, T, D, E, logits);
    return static_cast<int>(cudaGetLastError());
}

}  // namespace

int launch_router(const uint16_t *x, const uint16_t *w, const float *bias, int T, int D, int E, float *logits,
                  void *stream) {
    if (T == 0) return 0;
    if (router_tc_supported(T, D, E)) return launch_router_tc(x, w, bias, T, D, E, logits, stream);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return T < 4 ? launch_tt<1>(x, w, bias, T, D, E, logits, s) : launch_tt<4>(x, w, bias, T, D, E, logits, s);
}

}  // namespace ds4moe
