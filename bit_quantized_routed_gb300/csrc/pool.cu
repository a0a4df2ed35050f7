// Streamed experts: a pool of expert slots in device memory in front of a host-resident store.
//
// "DwarfStar" README, "运行大于 RAM 的模型": a model larger than memory keeps its routed
// experts outside it and loads the ones each token routes to. Here the store is pinned,
// device-mapped host memory (on a Grace system the GPU reads it over NVLink-C2C) holding every
// expert in the device layout, and the pool is a fixed number of slots in HBM. Per call, after
// routing and in stream order:
//   * pool_assign_kernel (one CTA) gives every touched expert a slot -- a resident expert keeps
//     its slot; each missing expert, in increasing expert order, takes the free slot (not used
//     by this call) with the oldest last use, empty slots first, ties to the lower slot -- and
//     rewrites the call's top-k indices to slot indices, so the grouping and expert kernels run
//     unchanged over the slots;
//   * pool_fill_kernel copies the missing experts' packed rows from the store into their slots
//     with 16-byte loads spread over the whole GPU.
#include <cuda_runtime.h>

#include "common.cuh"

namespace ds4moe {
namespace {

constexpr int kAssignThreads = 1024;  // one thread per expert (E <= 1024) and per slot

// Exclusive prefix sum of v over the CTA's 1024 threads; *total = the sum. tmp: 32 ints.
__device__ int scan1024(int v, int *tmp, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) tmp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = tmp[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        tmp[lane] = w;
    }
    __syncthreads();
    const int base = warp ? tmp[warp - 1] : 0;
    *total = tmp[31];
    __syncthreads();
    return base + x - v;
}

__global__ void __launch_bounds__(kAssignThreads) pool_assign_kernel(SlotPool sp, int32_t *__restrict__ idx, int P,
                                                                     int *status) {
    __shared__ uint8_t touched[1024];
    __shared__ int slot_by_rank[1024];
    __shared__ unsigned long long key[1024];
    __shared__ int tmp[32];
    const int t = threadIdx.x, E = sp.E, S = sp.S;
    touched[t] = 0;
    __syncthreads();
    for (int p = t; p < P; p += kAssignThreads) {
        const int e = idx[p];
        if (e >= 0 && e < E)
            touched[e] = 1;
        else
            report(status, ST_BADIDX);
    }
    __syncthreads();
    const unsigned long long call = sp.ctr[0] + 1;
    const bool mine = t < E && touched[t];
    const int cur = t < E ? sp.slot_of[t] : -1;
    const bool hit = mine && cur >= 0, miss = mine && cur < 0;
    int n_miss = 0, n_hit = 0;
    const int miss_rank = scan1024(miss ? 1 : 0, tmp, &n_miss);
    scan1024(hit ? 1 : 0, tmp, &n_hit);
    if (n_miss + n_hit > S) {  // more experts than slots: change nothing, keep the indices in range
        for (int p = t; p < P; p += kAssignThreads) idx[p] = 0;
        if (t == 0) {
            sp.ctr[3] = 0;
            report(status, ST_CAPACITY);
        }
        return;
    }
    // free slots (not used by this call) ranked by (last use, slot): key = last use << 32 | slot,
    // the largest key for a slot in use
    if (t < S) {
        const int ex = sp.expert_of[t];
        const bool free_slot = !(ex >= 0 && touched[ex]);
        key[t] = free_slot ? (static_cast<unsigned long long>(sp.stamp[t]) << 32) | static_cast<unsigned>(t) : ~0ull;
    }
    __syncthreads();  // every slot's state read before any is changed
    if (t < S && key[t] != ~0ull) {
        const unsigned long long mine_key = key[t];
        int rank = 0;
        for (int s = 0; s < S; s++) rank += key[s] < mine_key ? 1 : 0;
        slot_by_rank[rank] = t;
    }
    __syncthreads();
    if (miss) {
        const int s = slot_by_rank[miss_rank];
        const int old = sp.expert_of[s];
        if (old >= 0) sp.slot_of[old] = -1;  // an untouched expert: no other thread reads it
        sp.slot_of[t] = s;
        sp.expert_of[s] = t;
        sp.stamp[s] = static_cast<uint32_t>(call);
        sp.miss[2 * miss_rank] = t;
        sp.miss[2 * miss_rank + 1] = s;
    }
    if (hit) sp.stamp[cur] = static_cast<uint32_t>(call);
    __syncthreads();
    for (int p = t; p < P; p += kAssignThreads) {
        const int e = idx[p];
        idx[p] = (e >= 0 && e < E) ? sp.slot_of[e] : 0;
    }
    if (t == 0) {
        sp.ctr[0] = call;
        sp.ctr[1] += static_cast<unsigned long long>(n_hit);
        sp.ctr[2] += static_cast<unsigned long long>(n_miss);
        sp.ctr[3] = static_cast<unsigned long long>(n_miss);
    }
}

constexpr int kFillThreads = 512;
constexpr size_t kFillChunk = 64 * 1024;  // bytes per work item

// Work item i: miss i / per, chunk i % per of that expert's gate/up range followed by its down
// range (per = chunks of both). Both ranges are whole multiples of 16 bytes.
__global__ void __launch_bounds__(kFillThreads) pool_fill_kernel(SlotPool sp, uint8_t *__restrict__ iq2,
                                                                 uint8_t *__restrict__ q2k, uint8_t *__restrict__ tc_ok) {
    const int n_miss = static_cast<int>(sp.ctr[3]);
    const size_t cu = (sp.up_bytes + kFillChunk - 1) / kFillChunk, cd = (sp.down_bytes + kFillChunk - 1) / kFillChunk;
    const size_t per = cu + cd, items = static_cast<size_t>(n_miss) * per;
    for (size_t i = blockIdx.x; i < items; i += gridDim.x) {
        const int m = static_cast<int>(i / per);
        const size_t c = i % per;
        const int e = sp.miss[2 * m], s = sp.miss[2 * m + 1];
        const uint8_t *src;
        uint8_t *dst;
        size_t n;
        if (c < cu) {
            const size_t off = c * kFillChunk;
            src = sp.host_iq2 + static_cast<size_t>(e) * sp.up_bytes + off;
            dst = iq2 + static_cast<size_t>(s) * sp.up_bytes + off;
            n = min(kFillChunk, sp.up_bytes - off);
        } else {
            const size_t off = (c - cu) * kFillChunk;
            src = sp.host_q2k + static_cast<size_t>(e) * sp.down_bytes + off;
            dst = q2k + static_cast<size_t>(s) * sp.down_bytes + off;
            n = min(kFillChunk, sp.down_bytes - off);
        }
        const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
        uint4 *d4 = reinterpret_cast<uint4 *>(dst);
        const int n4 = static_cast<int>(n / 16);
        // four loads in flight per thread before the stores
        for (int j = threadIdx.x; j < n4; j += 4 * kFillThreads) {
            uint4 v[4];
#pragma unroll
            for (int u = 0; u < 4; u++) {
                const int q = j + u * kFillThreads;
                if (q < n4) v[u] = __ldcs(s4 + q);
            }
#pragma unroll
            for (int u = 0; u < 4; u++) {
                const int q = j + u * kFillThreads;
                if (q < n4) d4[q] = v[u];
            }
        }
        if (c == 0 && threadIdx.x == 0) tc_ok[s] = sp.host_tc_ok[e];
    }
}

}  // namespace

int launch_pool_assign(const SlotPool &sp, int32_t *idx, int P, int *status, void *stream) {
    pool_assign_kernel<<<1, kAssignThreads, 0, static_cast<cudaStream_t>(stream)>>>(sp, idx, P, status);
    return static_cast<int>(cudaGetLastError());
}

int launch_pool_fill(const SlotPool &sp, const DeviceWeights &w, int n_sms, void *stream) {
    pool_fill_kernel<<<2 * n_sms, kFillThreads, 0, static_cast<cudaStream_t>(stream)>>>(sp, w.iq2, w.q2k, w.tc_ok);
    return static_cast<int>(cudaGetLastError());
}

}  // namespace ds4moe
