// Router logits on the tensor cores, for calls of many tokens: logits[t][e] = sum_d x[t][d] * W[e][d]
// + bias[e] as a bf16 x bf16 -> fp32 GEMM (tcgen05, accumulators in tensor memory).
//
// "DwarfStar" README, "模型权重", and "DwarfStar 深度解析" §3.4.3: the router stays unquantised (bf16
// weights and an fp32 bias are this library's reading). The contraction is dense, D columns per
// logit, so from 64 tokens on it runs here instead of on the CUDA cores (router.cu): a CTA computes
// 128 experts x 128 tokens, the router rows as the MMA's M side and the tokens as its N side, both
// copied by TMA (128-byte swizzled K-major tiles of 64 columns, six stages); one thread issues
// tcgen05.mma (kind::f16 with bf16 operands, K = 16 per instruction) into 128 fp32 accumulator
// columns; four warps read them back, add the bias and store fp32 logits (a warp writes 32
// consecutive experts of one token). Each 16-column step adds its 16 exact products to the fp32
// accumulator: the order is the hardware's within a step and fixed across steps, so a call's
// logits are the same on every run.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace ds4moe {
namespace {

constexpr int kRtM = 128;                                  // experts per CTA (MMA M, TMEM lanes)
constexpr int kRtN = 128;                                  // tokens per CTA (MMA N, TMEM columns)
constexpr int kRtK = 64;                                   // columns per stage: one 128-byte swizzle row
constexpr int kRtStages = 6;
constexpr int kRtTileBytes = kRtM * kRtK * 2;              // 16 KB (the router tile; the token tile is the same)
constexpr int kRtStageBytes = 2 * kRtTileBytes;            // 32 KB
constexpr int kRtThreads = 192;                            // copies, MMA, four read-back warps
constexpr int kRtSmem = kRtStages * kRtStageBytes + 1024 + 256;

// Timeouts of the tensor-core router's bounded waits (ST_TIMEOUT), read and cleared by
// ds4moe_router_last_status().
__device__ int g_router_status;

struct RouterMaps {
    CUtensorMap x;  // [T][D] bf16, 64 x 128 boxes
    CUtensorMap w;  // [E][D] bf16, 64 x 128 boxes
};

// Instruction descriptor of kind::f16 with bf16 A and B (K-major), fp32 accumulate, M x N.
__device__ __forceinline__ uint32_t idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ uint32_t desc_lo(uint32_t saddr) { return ((saddr >> 4) & 0x3FFFu) | (1u << 16); }
constexpr uint32_t kDescHi = (1024u >> 4) | (1u << (46 - 32)) | (2u << (61 - 32));

__global__ void __launch_bounds__(kRtThreads, 1) router_tc_kernel(const __grid_constant__ RouterMaps maps,
                                                                  const float *__restrict__ bias, int T, int D, int E,
                                                                  float *__restrict__ logits) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kRtStages * kRtStageBytes);
    // bars: full[S], empty[S], acc_full, spare
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + 2 * kRtStages + 2);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
    int *status = &g_router_status;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e_tiles = E / kRtM;
    const int e0 = (static_cast<int>(blockIdx.x) % e_tiles) * kRtM;
    const int t0 = (static_cast<int>(blockIdx.x) / e_tiles) * kRtN;
    const int num_kb = D / kRtK;
    auto full = [&](int s) { return smem_u32(bars + s); };
    auto empty = [&](int s) { return smem_u32(bars + kRtStages + s); };
    const uint32_t acc_full = smem_u32(bars + 2 * kRtStages), spare = smem_u32(bars + 2 * kRtStages + 1);
    auto w_tile = [&](int s) { return smem_u32(smem + s * kRtStageBytes); };
    auto x_tile = [&](int s) { return smem_u32(smem + s * kRtStageBytes + kRtTileBytes); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < kRtStages; s++) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(spare, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_holder)),
                     "r"(kRtN)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        // ---------------------------------------------------------- TMA: router rows and token rows
        if (lane == 0) {
            int issued_parity[kRtStages];
#pragma unroll
            for (int s = 0; s < kRtStages; s++) issued_parity[s] = -1;
            bool ok = true;
            for (int kb = 0; kb < num_kb; kb++) {
                const int s = kb % kRtStages;
                const uint32_t ph = static_cast<uint32_t>(kb / kRtStages) & 1u;
                if (!mbar_wait(empty(s), ph ^ 1u, abort_flag, status)) {
                    ok = false;
                    break;
                }
                mbar_expect_tx(full(s), kRtStageBytes);
                tma_load_2d(w_tile(s), &maps.w, kb * kRtK, e0, full(s));
                tma_load_2d(x_tile(s), &maps.x, kb * kRtK, t0, full(s));  // rows past T read as zeros
                issued_parity[s] = static_cast<int>(ph);
            }
            if (!ok)  // let copies still in flight land before the CTA exits
                for (int s = 0; s < kRtStages; s++)
                    if (issued_parity[s] >= 0) mbar_drain(full(s), static_cast<uint32_t>(issued_parity[s]));
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issue (one thread)
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(kRtM, kRtN);
            bool ok = true, issued = false;
            for (int kb = 0; kb < num_kb; kb++) {
                const int s = kb % kRtStages;
                const uint32_t ph = static_cast<uint32_t>(kb / kRtStages) & 1u;
                if (!mbar_wait(full(s), ph, abort_flag, status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a_lo = desc_lo(w_tile(s)), b_lo = desc_lo(x_tile(s));
#pragma unroll
                for (int k = 0; k < kRtK / 16; k++)  // 32 bytes of each row per K step
                    tc_mma(tmem, a_lo + 2u * k, b_lo + 2u * k, kDescHi, idesc, (kb | k) != 0);
                issued = true;
                tc_commit(empty(s));
            }
            if (ok) {
                tc_commit(acc_full);
            } else if (issued) {  // wait for the MMAs in flight before the memory goes away
                tc_commit(spare);
                mbar_drain(spare, 0);
            }
        }
    } else {
        // ---------------------------------------------------------- read-back: warp w, TMEM lanes 32 (w % 4) ..
        const int q = warp & 3;
        const int e = e0 + q * 32 + lane;
        if (mbar_wait(acc_full, 0, abort_flag, status)) {
            tc_fence_after();
            const float b = bias ? bias[e] : 0.0f;
            for (int c0 = 0; c0 < kRtN && t0 + c0 < T; c0 += 16) {  // uniform over the warp
                uint32_t v[16];
                tmem_ld16_start(tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(c0), v);
                tmem_wait_ld(v);
#pragma unroll
                for (int j = 0; j < 16; j++) {
                    const int t = t0 + c0 + j;
                    if (t < T) {
                        const float l = __uint_as_float(v[j]);
                        logits[static_cast<size_t>(t) * E + e] = bias ? __fadd_rn(l, b) : l;
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kRtN) : "memory");
    }
}

// One 2-D bf16 tensor map: [rows][cols] row-major, 64 x 128 boxes, 128-byte swizzle.
int encode_bf16_map(CUtensorMap *map, const void *base, int rows, int cols) {
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    if (!encode) {
        cudaDriverEntryPointQueryResult q;
        void *fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn) {
            cudaGetLastError();
            return 1;
        }
        encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
    const cuuint32_t box[2] = {kRtK, 128};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? 0 : 1;
}

}  // namespace

bool router_tc_supported(int T, int D, int E) { return T >= 64 && E % kRtM == 0 && D % kRtK == 0; }

int launch_router_tc(const uint16_t *x, const uint16_t *w, const float *bias, int T, int D, int E, float *logits,
                     void *stream) {
    static int seen[64];  // per device: the kernel's shared-memory attribute is set
    const int err = ensure_smem(reinterpret_cast<const void *>(router_tc_kernel), kRtSmem, seen);
    if (err) return err;
    RouterMaps maps;
    if (encode_bf16_map(&maps.x, x, T, D) || encode_bf16_map(&maps.w, w, E, D)) return static_cast<int>(cudaErrorInvalidValue);
    const int blocks = (E / kRtM) * ((T + kRtN - 1) / kRtN);
    router_tc_kernel<<<blocks, kRtThreads, kRtSmem, static_cast<cudaStream_t>(stream)>>>(maps, bias, T, D, E, logits);
    return static_cast<int>(cudaGetLastError());
}

int router_read_status(int *st) {
    if (cudaMemcpyFromSymbol(st, g_router_status, sizeof(int)) != cudaSuccess) return 1;
    const int zero = 0;
    return cudaMemcpyToSymbol(g_router_status, &zero, sizeof(int)) != cudaSuccess ? 1 : 0;
}

}  // namespace ds4moe
