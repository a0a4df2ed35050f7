// Top-k routing and grouping of (token, slot) pairs by expert.
//
// Routing: "DwarfStar 深度解析" §2.1 -- each token picks its experts dynamically -- and
// §3.4.3 -- the router stays at full precision, so selection compares the fp32 logits
// exactly. Ties go to the lower expert index (this library's reading). Grouping: the
// stable counting sort that lets each expert's weights be streamed once per call for all
// of its tokens ("Part 5: 服务层" §6: read-only weight work done once for the whole batch).
#include <cuda_runtime.h>

#include <cfloat>
#include <climits>

#include "common.cuh"

namespace ds4moe {
namespace {

// One warp per token; lane L holds experts L, L+32, ... (PER of them).
template <int PER>
__global__ void __launch_bounds__(256) route_kernel(const float *__restrict__ logits, int T, int E, int k,
                                                    int mode, int32_t *__restrict__ idx,
                                                    float *__restrict__ wout) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    const float *l = logits + static_cast<size_t>(t) * E;
    float key[PER];
#pragma unroll
    for (int j = 0; j < PER; j++) {
        const int e = lane + 32 * j;
        const float v = e < E ? l[e] : -INFINITY;
        key[j] = (v != v) ? -INFINITY : v;  // NaN orders as -inf
    }
    uint32_t taken = 0;
    float my_v = -INFINITY;
    int my_i = 0;
    for (int r = 0; r < k; r++) {
        float bv = -INFINITY;
        int bi = INT_MAX;
#pragma unroll
        for (int j = 0; j < PER; j++) {
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
    if (lane < k) num = gate_numerator(my_v, top, mode);
    const float den = warp_sum(num);
    if (lane < k) {
        idx[static_cast<size_t>(t) * k + lane] = my_i;
        wout[static_cast<size_t>(t) * k + lane] = num / den;
    }
}

constexpr int kGroupThreads = 1024;
constexpr int kGroupWarps = kGroupThreads / 32;

// Exclusive scan over the block (1024 threads). tmp: 32 ints of shared memory.
__device__ int block_exclusive_scan(int v, int *tmp, int *total) {
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
        int s = tmp[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        tmp[lane] = s;
    }
    __syncthreads();
    const int base = warp ? tmp[warp - 1] : 0;
    if (total) *total = tmp[kGroupWarps - 1];
    __syncthreads();
    return base + x - v;
}

// Single-CTA stable counting sort. Warp w owns the contiguous pair range
// [w*chunk, (w+1)*chunk); per-warp histograms give every warp its base position per expert,
// then each warp walks its range in order, ranking equal experts inside each batch of 32
// with __match_any_sync, so positions follow (token, slot) order exactly.
__global__ void __launch_bounds__(kGroupThreads, 1)
    group_kernel(const int32_t *__restrict__ idx, int P, int E, int gemm_min, const uint8_t *__restrict__ tc_ok,
                 int32_t *__restrict__ counts, int32_t *__restrict__ offsets, int32_t *__restrict__ perm,
                 int32_t *__restrict__ inv, int32_t *__restrict__ gemv_list, int32_t *__restrict__ gemm_list,
                 int32_t *__restrict__ single_list, int32_t *__restrict__ tile_prefix, int32_t *__restrict__ tile_desc,
                 int32_t *__restrict__ small_pos, GroupMeta *meta, int *status, int32_t *__restrict__ ovf) {
    pdl_wait();
    if (ovf) {  // the call's overflow flags start clear (E + 1 of them)
        for (int i = threadIdx.x; i <= E; i += kGroupThreads) ovf[i] = 0;
    }
    extern __shared__ int sm[];
    int *hist = sm;                      // [kGroupWarps][E]: counts, then base positions
    int *tmp = sm + kGroupWarps * E;     // [32]
    int *part = tmp + 32;                // [E] tokens of each tensor-core expert's ragged last tile (0: none)
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < kGroupWarps * E; i += kGroupThreads) hist[i] = 0;
    __syncthreads();
    const int chunk = (P + kGroupWarps - 1) / kGroupWarps;
    const int p0 = warp * chunk, p1 = min(P, p0 + chunk);
    int *my = hist + warp * E;
    for (int p = p0 + lane; p < p1; p += 32) {
        int e = idx[p];
        if (e < 0 || e >= E) {
            report(status, ST_BADIDX);
            e = 0;
        }
        atomicAdd(&my[e], 1);
    }
    __syncthreads();
    // per expert: total and exclusive prefix over warps; then scan over experts
    const int e = threadIdx.x;
    int tot = 0;
    if (e < E) {
        for (int w = 0; w < kGroupWarps; w++) {
            const int c = hist[w * E + e];
            hist[w * E + e] = tot;
            tot += c;
        }
    }
    int all = 0;
    const int off = block_exclusive_scan(e < E ? tot : 0, tmp, &all);
    if (e < E) {
        counts[e] = tot;
        offsets[e] = off;
        for (int w = 0; w < kGroupWarps; w++) hist[w * E + e] += off;
    }
    if (e == 0) offsets[E] = all;
    // GEMV / tensor-core work lists, each in expert order; experts whose weights do not fit
    // fp16 stay on the GEMV path
    const bool big = e < E && tot > 0 && gemm_min > 0 && tot >= gemm_min && (!tc_ok || tc_ok[e]);
    const bool single = single_list && e < E && tot == 1 && !big;  // one-token groups, own list
    const bool small = e < E && tot > 0 && !big && !single;
    int n_small = 0, n_big = 0, n_tiles = 0, n_single = 0;
    const int psg = block_exclusive_scan(single ? 1 : 0, tmp, &n_single);
    if (single) single_list[psg] = e;
    const int ps = block_exclusive_scan(small ? 1 : 0, tmp, &n_small);
    const int pb = block_exclusive_scan(big ? 1 : 0, tmp, &n_big);
    const int pt = block_exclusive_scan(big ? (tot + kGemmBN - 1) / kGemmBN : 0, tmp, &n_tiles);
    // tensor-core token tiles, longest first: the full tiles in expert order, then each expert's
    // ragged last tile by decreasing size (ties to the lower expert), so that the GEMMs' CTAs,
    // which take tiles in a fixed stride, take tiles of similar cost side by side
    const int nfull = big ? tot / kGemmBN : 0;
    const int rag = big ? tot % kGemmBN : 0;
    int n_full = 0;
    const int pf = block_exclusive_scan(nfull, tmp, &n_full);
    if (e < E) part[e] = rag;
    __syncthreads();
    int rank = 0;
    if (rag > 0)
        for (int o = 0; o < E; o++) rank += (part[o] > rag || (part[o] == rag && o < e)) ? 1 : 0;
    if (small && gemv_list) gemv_list[ps] = e;
    // positions of the small groups' pairs, in expert order (the small-group down kernel's slots)
    int n_small_pairs = 0;
    const int pp = block_exclusive_scan(small ? tot : 0, tmp, &n_small_pairs);
    if (small && small_pos)
        for (int r = 0; r < tot; r++) small_pos[pp + r] = off + r;
    if (big && gemm_list) gemm_list[pb] = e;
    if (big && tile_prefix) tile_prefix[pb] = pt;
    if (threadIdx.x == 0 && tile_prefix) tile_prefix[n_big] = n_tiles;
    // one descriptor per tensor-core token tile (expert, first row, tokens), in tile order
    if (big && tile_desc) {
        for (int lt = 0; lt < nfull; lt++)
            reinterpret_cast<int4 *>(tile_desc)[pf + lt] = make_int4(e, off + lt * kGemmBN, kGemmBN, 0);
        if (rag > 0)
            reinterpret_cast<int4 *>(tile_desc)[n_full + rank] = make_int4(e, off + nfull * kGemmBN, rag, 0);
    }
    if (threadIdx.x == 0 && meta) {
        meta->n_gemv = n_small;
        meta->n_gemm = n_big;
        meta->n_single = n_single;
        meta->n_small_pairs = n_small_pairs;
        meta->n_tiles = n_tiles;
        meta->n_full = n_full;
    }
    __syncthreads();
    // stable positions
    for (int base = p0; base < p1; base += 32) {
        const int p = base + lane;
        const bool live = p < p1;
        int ex = live ? idx[p] : -1;
        if (live && (ex < 0 || ex >= E)) ex = 0;
        const unsigned peers = __match_any_sync(0xffffffffu, ex);
        const int rank = __popc(peers & ((1u << lane) - 1u));
        const int leader = __ffs(peers) - 1;
        int pos = 0;
        if (live) pos = my[ex] + rank;
        __syncwarp();
        if (live && lane == leader) my[ex] += __popc(peers);
        __syncwarp();
        if (live) {
            perm[pos] = p;
            inv[p] = pos;
        }
    }
}

}  // namespace

int launch_route(const float *logits, int T, int E, int k, int gate_mode, int32_t *idx, float *w,
                 void *stream) {
    if (T == 0) return 0;
    const int per = (E + 31) / 32;
    const int warps = 8;
    dim3 grid((T + warps - 1) / warps), block(32 * warps);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int rc;
    if (per <= 1)
        rc = launch_pdl(route_kernel<1>, grid, block, 0, s, logits, T, E, k, gate_mode, idx, w);
    else if (per <= 2)
        rc = launch_pdl(route_kernel<2>, grid, block, 0, s, logits, T, E, k, gate_mode, idx, w);
    else if (per <= 4)
        rc = launch_pdl(route_kernel<4>, grid, block, 0, s, logits, T, E, k, gate_mode, idx, w);
    else if (per <= 8)
        rc = launch_pdl(route_kernel<8>, grid, block, 0, s, logits, T, E, k, gate_mode, idx, w);
    else if (per <= 16)
        rc = launch_pdl(route_kernel<16>, grid, block, 0, s, logits, T, E, k, gate_mode, idx, w);
    else
        rc = launch_pdl(route_kernel<32>, grid, block, 0, s, logits, T, E, k, gate_mode, idx, w);
    return rc;
}

int launch_group(const int32_t *idx, int T, int k, int E, int gemm_min, const uint8_t *tc_ok, int32_t *counts,
                 int32_t *offsets, int32_t *perm, int32_t *inv, int32_t *gemv_list, int32_t *gemm_list,
                 int32_t *single_list, int32_t *tile_prefix, int32_t *tile_desc, int32_t *small_pos, GroupMeta *meta, int *status,
                 void *stream, int32_t *ovf) {
    const int P = T * k;
    const size_t smem = (static_cast<size_t>(kGroupWarps) * E + 32 + E) * sizeof(int);
    static int seen[64];
    const int err = ensure_smem(reinterpret_cast<const void *>(group_kernel), static_cast<int>(smem), seen);
    if (err) return err;
    return launch_pdl(group_kernel, dim3(1), dim3(kGroupThreads), smem, static_cast<cudaStream_t>(stream), idx, P, E,
                      gemm_min, tc_ok, counts, offsets, perm, inv, gemv_list, gemm_list, single_list, tile_prefix,
                      tile_desc, small_pos, meta, status, ovf);
}

}  // namespace ds4moe
