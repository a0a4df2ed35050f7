// Device helpers shared by the kernels: block decoding, warp reductions, status reporting.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "internal.h"

namespace ds4moe {

constexpr int kWarp = 32;

// Raises a kernel's dynamic shared-memory limit to at least `bytes` on the current device,
// once per (kernel, device): the launch path then makes no attribute call per launch.
// seen: per-kernel array of 64 device slots holding the largest size set so far.
inline int ensure_smem(const void *kernel, int bytes, int *seen) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (dev >= 0 && dev < 64 && seen[dev] >= bytes) return 0;
    const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return static_cast<int>(e);
    if (dev >= 0 && dev < 64) seen[dev] = bytes;
    return 0;
}

__device__ __forceinline__ void report(int *status, int bits) {
    if (status) atomicOr(status, bits);
}

// Programmatic dependent launch: the kernels of a call are launched with launch_pdl, so each may
// be scheduled while the kernel before it in the stream drains; the first thing each of them does
// is wait here until that kernel has completed and its writes are visible (a no-op when launched
// without the attribute), so nothing is read or written before its inputs are final.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Launch with the programmatic-stream-serialisation attribute (see pdl_wait).
template <typename... KArgs, typename... Args>
inline int launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return static_cast<int>(cudaLaunchKernelEx(&cfg, kernel, args...));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Gate numerator of a selected logit v against the first (largest) selected logit top, both
// with NaN already taken as -inf ("DwarfStar 深度解析" §2.1 routes each token by its logits; the
// weights below are this library's reading): softmax mode exp(v - top), counted as exp(0) = 1
// where v equals top, also when both are infinite (the limit of equal logits: an all -inf
// selection gets 1/k each, a +inf logit takes the weight from every finite one); sigmoid mode
// the same over log sigmoid(v) = min(v, 0) - log1p(exp(-|v|)), since sigmoid(v) / sum of
// sigmoids is the softmax of the log-sigmoids, which never underflows to 0 / 0.
__device__ __forceinline__ float gate_numerator(float v, float top, int mode) {
    if (mode != DS4MOE_GATE_SOFTMAX) {
        v = fminf(v, 0.0f) - log1pf(expf(-fabsf(v)));
        top = fminf(top, 0.0f) - log1pf(expf(-fabsf(top)));
    }
    return v == top ? 1.0f : expf(v - top);
}

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

__device__ __forceinline__ float f16_to_f32(uint16_t h) { return __half2float(__ushort_as_half(h)); }

// silu(v) * u with the fast exponential; |error| ~ 1e-7 relative.
__device__ __forceinline__ float swiglu(float v, float u) { return v / (1.0f + __expf(-v)) * u; }
// The same with the quotient from the fast-division intrinsic (within 2 ulp; for v below about
// -87 the denominator exceeds 2^126 and the quotient is 0, the limit of silu there): for the
// tensor-core epilogue, where the division is a visible share of the time.
__device__ __forceinline__ float swiglu_fast(float v, float u) { return __fdividef(v, 1.0f + __expf(-v)) * u; }

// ---------------------------------------------------------------- IQ2-style decode
// One group of 8 weights: w_i = scale * G[idx][i] * sign_i, exact in fp32.
// grid_entry: the 8 magnitude bytes of G[idx] (lo word = elements 0..3);
// s7: the 7 stored sign bits; element 7's sign is their parity.
__device__ __forceinline__ void iq2_group(uint2 grid_entry, uint32_t s7, float scale, float w[8]) {
    const uint32_t signs = s7 | ((__popc(s7) & 1u) << 7);
#pragma unroll
    for (int i = 0; i < 8; i++) {
        const uint32_t m = ((i < 4 ? grid_entry.x : grid_entry.y) >> (8 * (i & 3))) & 0xffu;
        const float v = __fmul_rn(scale, static_cast<float>(m));
        w[i] = __uint_as_float(__float_as_uint(v) ^ (((signs >> i) & 1u) << 31));
    }
}

// Scale of one 32-weight sub-block: d * (s+1) / 16, exact in fp32.
__device__ __forceinline__ float iq2_scale(float d, uint32_t word) {
    return __fmul_rn(__fmul_rn(d, static_cast<float>((word >> 28) + 1u)), 0.0625f);
}

// ---------------------------------------------------------------- Q2_K-style decode
// Weight with code q in a sub-block with ds = d*sc and dm = dmin*m (both exact):
// one rounding of the exact ds*q - dm.
__device__ __forceinline__ float q2k_weight(float ds, float dm, uint32_t q) {
    return __fmaf_rn(ds, static_cast<float>(q), -dm);
}

}  // namespace ds4moe
