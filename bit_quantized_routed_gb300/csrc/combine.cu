// Gate-weighted combine into the residual:
//   out[t] += y_shared[t] + sum over slots s (in slot order) of g[t,s] * y[pos(t,s)].
// A gather per token (no atomics), so the result is bit-reproducible run to run.
#include <cuda_runtime.h>

#include <algorithm>

#include "common.cuh"

namespace ds4moe {
namespace {

__global__ void __launch_bounds__(256) combine_kernel(const float *__restrict__ y, const int32_t *__restrict__ inv,
                                                      const float *__restrict__ g, int T, int k, int D, int P,
                                                      int shared, float *__restrict__ out) {
    const int D4 = D / 4;
    const size_t n = static_cast<size_t>(T) * D4;
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const int t = static_cast<int>(i / D4);
        const int c = static_cast<int>(i - static_cast<size_t>(t) * D4);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (shared) acc = reinterpret_cast<const float4 *>(y + static_cast<size_t>(P + t) * D)[c];
        for (int s = 0; s < k; s++) {
            const int pos = inv[t * k + s];
            const float gw = g[t * k + s];
            const float4 v = reinterpret_cast<const float4 *>(y + static_cast<size_t>(pos) * D)[c];
            acc.x = fmaf(gw, v.x, acc.x);
            acc.y = fmaf(gw, v.y, acc.y);
            acc.z = fmaf(gw, v.z, acc.z);
            acc.w = fmaf(gw, v.w, acc.w);
        }
        float4 *o = reinterpret_cast<float4 *>(out + static_cast<size_t>(t) * D) + c;
        float4 r = *o;
        r.x += acc.x;
        r.y += acc.y;
        r.z += acc.z;
        r.w += acc.w;
        *o = r;
    }
}

}  // namespace

int launch_combine(const DeviceWeights &w, const Workspace &ws, int T, int k, float *out, void *stream) {
    const size_t n = static_cast<size_t>(T) * (w.D / 4);
    const int blocks = static_cast<int>(std::min<size_t>((n + 255) / 256, 152 * 16));
    combine_kernel<<<blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(ws.y, ws.inv, ws.topk_w, T, k, w.D, T * k,
                                                                          w.has_shared ? 1 : 0, out);
    return static_cast<int>(cudaGetLastError());
}

}  // namespace ds4moe
