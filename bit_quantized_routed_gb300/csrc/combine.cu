// Gate-weighted combine into the residual:
//   out[t] += y_shared[t] + sum over slots s (in slot order) of g[t,s] * y[pos(t,s)].
// A gather per token (no atomics), so the result is bit-reproducible run to run. The rows the
// tensor-core down GEMM produced hold fp16 values in the first half of their fp32 slot; the
// kernel tells them apart by the same test the grouping used to send a group there.
#include <cuda_runtime.h>

#include <algorithm>

#include "common.cuh"

namespace ds4moe {
namespace {

struct CombineParams {
    const float *y;          // [P+T] rows of D fp32 (or D fp16 in the slot's first half)
    const int32_t *inv;      // [T*k] row of each (token, slot)
    const float *g;          // [T*k] gate weights
    const int32_t *idx;      // [T*k] expert (slot) of each (token, slot)
    const int32_t *counts;   // [E] tokens per expert
    const uint8_t *tc_ok;    // [E] the expert may run on the tensor cores
    int T, k, D, P, E;
    int gemm_min;            // > 0: groups of at least this many tokens ran on the tensor cores
    int shared;              // rows P.. hold the shared expert's output
    int shared_f16;          // ... in fp16
    const int32_t *ovf;      // [E+1] or null: the expert's tensor-core rows were recomputed in fp32
    float *out;
};

__device__ __forceinline__ void load8(const float *row, int c, bool f16, float v[8]) {
    if (f16) {
        const uint4 u = reinterpret_cast<const uint4 *>(row)[c];  // 8 fp16 values, columns 8c .. 8c+7
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w[i]));
            v[2 * i] = f.x;
            v[2 * i + 1] = f.y;
        }
    } else {
        const float4 a = reinterpret_cast<const float4 *>(row)[2 * c];
        const float4 b = reinterpret_cast<const float4 *>(row)[2 * c + 1];
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
}

// One CTA per token (grid-stride over tokens); each thread 8 columns at a time.
__global__ void __launch_bounds__(256) combine_kernel(CombineParams p) {
    pdl_wait();
    __shared__ int s_pos[32];
    __shared__ float s_g[32];
    __shared__ int s_f16[32];
    const int D8 = p.D / 8;
    // the shared expert's rows: fp16 unless its tensor-core result was recomputed in fp32
    const bool sh16 = p.shared_f16 != 0 && !(p.ovf && p.ovf[p.E]);
    for (int t = blockIdx.x; t < p.T; t += gridDim.x) {
        if (threadIdx.x < p.k) {
            const int s = threadIdx.x;
            const int e = p.idx[t * p.k + s];
            s_pos[s] = p.inv[t * p.k + s];
            s_g[s] = p.g[t * p.k + s];
            // (an index outside [0, E) has been reported by the grouping kernel, which grouped it as expert 0)
            const int ec = (e >= 0 && e < p.E) ? e : 0;
            s_f16[s] = p.gemm_min > 0 && p.counts[ec] >= p.gemm_min && p.tc_ok[ec] && !(p.ovf && p.ovf[ec]);
        }
        __syncthreads();
        for (int c = threadIdx.x; c < D8; c += blockDim.x) {
            // the residual's load is issued first and the slots' loads four at a time, so that
            // several rows are in flight per thread
            float4 *o = reinterpret_cast<float4 *>(p.out + static_cast<size_t>(t) * p.D) + 2 * c;
            float4 a = o[0], b = o[1];
            float acc[8];
            if (p.shared) {
                load8(p.y + static_cast<size_t>(p.P + t) * p.D, c, sh16, acc);
            } else {
#pragma unroll
                for (int i = 0; i < 8; i++) acc[i] = 0.0f;
            }
#pragma unroll 4
            for (int s = 0; s < p.k; s++) {
                float v[8];
                load8(p.y + static_cast<size_t>(s_pos[s]) * p.D, c, s_f16[s] != 0, v);
                const float gw = s_g[s];
#pragma unroll
                for (int i = 0; i < 8; i++) acc[i] = fmaf(gw, v[i], acc[i]);
            }
            a.x += acc[0]; a.y += acc[1]; a.z += acc[2]; a.w += acc[3];
            b.x += acc[4]; b.y += acc[5]; b.z += acc[6]; b.w += acc[7];
            o[0] = a;
            o[1] = b;
        }
        __syncthreads();
    }
}

// One CTA of 1024 threads (E <= 1024): the experts whose tensor-core results overflowed fp16, in
// expert order, as the GEMV kernels' work list (meta->n_gemv of them); the shared expert's flag
// stays in ovf[E].
__global__ void __launch_bounds__(1024) repair_list_kernel(const int32_t *__restrict__ ovf, int E,
                                                           int32_t *__restrict__ list, GroupMeta *meta) {
    pdl_wait();
    __shared__ int wcount[32];
    const int e = threadIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const bool f = e < E && ovf[e] != 0;
    const unsigned m = __ballot_sync(0xffffffffu, f);
    if (lane == 0) wcount[warp] = __popc(m);
    __syncthreads();
    if (warp == 0) {  // exclusive prefix of the warps' counts
        const int c = wcount[lane];
        int x = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        wcount[lane] = x - c;
        if (lane == 31) {
            meta->n_gemv = x;
            meta->n_gemm = meta->n_single = meta->n_small_pairs = meta->n_tiles = meta->n_full = 0;
        }
    }
    __syncthreads();
    if (f) list[wcount[warp] + __popc(m & ((1u << lane) - 1u))] = e;
}

}  // namespace

int launch_repair_list(const DeviceWeights &w, const Workspace &ws, int, void *stream) {
    return launch_pdl(repair_list_kernel, dim3(1), dim3(1024), 0, static_cast<cudaStream_t>(stream),
                      static_cast<const int32_t *>(ws.ovf), w.E, ws.repair_list, ws.meta2);
}

int launch_combine(const DeviceWeights &w, const Workspace &ws, int T, int k, int gemm_min, bool shared_f16,
                   float *out, void *stream) {
    CombineParams p;
    p.y = ws.y;
    p.inv = ws.inv;
    p.g = ws.topk_w;
    p.idx = ws.topk_idx;
    p.counts = ws.counts;
    p.tc_ok = w.tc_ok;
    p.T = T;
    p.k = k;
    p.D = w.D;
    p.P = T * k;
    p.E = w.E;
    p.gemm_min = gemm_min;
    p.shared = w.has_shared ? 1 : 0;
    p.shared_f16 = (w.has_shared && shared_f16) ? 1 : 0;
    p.ovf = ws.ovf;
    p.out = out;
    const int blocks = std::min(T, 152 * 8);
    return launch_pdl(combine_kernel, dim3(blocks), dim3(256), 0, static_cast<cudaStream_t>(stream), p);
}

}  // namespace ds4moe
