// The bf16 shared expert's gate/up + SwiGLU for a few tokens (T <= 48), on warp-level bf16 MMAs.
//
// "DwarfStar 深度解析" §3.4.3: the shared expert is always on and kept in bf16, so at decode
// batch sizes its 2 x d_ff x d_model weights are one more pure stream of bytes (half of them at one
// token). The tcgen05 kernel tiles it 128 weight rows per CTA, which leaves most SMs idle when the
// token count is small; here a CTA takes 16 rows (F/16 CTAs), its 16 warps split d_model, and each
// warp streams its slice of the rows straight from HBM into mma.sync.m16n8k16 operands:
//   * bf16 x bf16 products are exact and accumulate in fp32, as on every other path;
//   * the K order inside each 32-column step is permuted the same way for weights and tokens, so
//     every thread reads 16 contiguous bytes of a row (all sectors used) and of a token;
//   * the 16 warps' partial tiles are summed in shared memory in a fixed order (deterministic),
//     and h = silu(gate) * up is written as fp16 into the rows the tensor-core down GEMM reads.
#include <cuda_runtime.h>

#include "common.cuh"

namespace ds4moe {
namespace {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kRows = 16;       // weight rows per CTA (the MMA's M)
constexpr int kMaxTiles = 6;    // 8-token tiles: T <= 48 (more would spill registers)

// D = A * B + D for one m16n8k16 tile, bf16 operands, fp32 accumulators.
__device__ __forceinline__ void mma_bf16(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

struct SharedParams {
    const uint16_t *x;   // bf16 [T][D]
    const uint16_t *wg;  // bf16 [F][D]
    const uint16_t *wu;
    uint16_t *h16;       // fp16 [T][F]: the shared expert's rows of the tensor-core path's h
    int T, D, F;
    int32_t *ovf_shared;  // set when an h value exceeds fp16: the shared expert is recomputed in fp32
};

// Fragment mapping of one 32-column step s (columns 32s .. 32s+31): thread (g = lane >> 2,
// c = lane & 3) reads columns 32s + 8c .. +7 of weight rows g and g + 8 and of token g of each
// 8-token tile. Of those 8 columns, 0-1 and 2-3 are the MMA k pairs (2c, 2c+1) and (2c+8, 2c+9) of
// the step's first k16 MMA, 4-5 and 6-7 those of its second; weights and tokens use the same map.
template <int NT>
__global__ void __launch_bounds__(kThreads, 1) shared_up_kernel(SharedParams p) {
    pdl_wait();
    extern __shared__ float red[];  // [kWarps][2][kRows][NT * 8]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
    const int D = p.D, F = p.F, T = p.T, row0 = blockIdx.x * kRows;
    const uint4 *rg0 = reinterpret_cast<const uint4 *>(p.wg + static_cast<size_t>(row0 + g) * D);
    const uint4 *rg8 = reinterpret_cast<const uint4 *>(p.wg + static_cast<size_t>(row0 + g + 8) * D);
    const uint4 *ru0 = reinterpret_cast<const uint4 *>(p.wu + static_cast<size_t>(row0 + g) * D);
    const uint4 *ru8 = reinterpret_cast<const uint4 *>(p.wu + static_cast<size_t>(row0 + g + 8) * D);
    const uint4 *xt[NT];
    bool tv[NT];
#pragma unroll
    for (int n = 0; n < NT; n++) {
        const int t = 8 * n + g;
        tv[n] = t < T;
        xt[n] = reinterpret_cast<const uint4 *>(p.x + static_cast<size_t>(tv[n] ? t : 0) * D);
    }
    float acc[2][NT][4];
#pragma unroll
    for (int m = 0; m < 2; m++)
#pragma unroll
        for (int n = 0; n < NT; n++)
#pragma unroll
            for (int i = 0; i < 4; i++) acc[m][n][i] = 0.0f;
    const int steps = D / 32;
    constexpr int kUnroll = NT > 4 ? 1 : 2;  // two steps of loads in flight while registers allow
#pragma unroll kUnroll
    for (int s = warp; s < steps; s += kWarps) {
        const int q = 4 * s + c;  // the thread's 16-byte chunk of each row
        const uint4 a0 = __ldcs(rg0 + q), a8 = __ldcs(rg8 + q), b0 = __ldcs(ru0 + q), b8 = __ldcs(ru8 + q);
        uint4 xv[NT];
#pragma unroll
        for (int n = 0; n < NT; n++) xv[n] = tv[n] ? __ldg(xt[n] + q) : make_uint4(0, 0, 0, 0);
        const uint32_t ga[2][4] = {{a0.x, a8.x, a0.y, a8.y}, {a0.z, a8.z, a0.w, a8.w}};
        const uint32_t ua[2][4] = {{b0.x, b8.x, b0.y, b8.y}, {b0.z, b8.z, b0.w, b8.w}};
#pragma unroll
        for (int h = 0; h < 2; h++)
#pragma unroll
            for (int n = 0; n < NT; n++) {
                const uint32_t bx0 = h ? xv[n].z : xv[n].x, bx1 = h ? xv[n].w : xv[n].y;
                mma_bf16(acc[0][n], ga[h], bx0, bx1);
                mma_bf16(acc[1][n], ua[h], bx0, bx1);
            }
    }
    // this warp's partial tiles: C[g][2c], C[g][2c+1], C[g+8][2c], C[g+8][2c+1] of each token tile
    constexpr int TT = NT * 8;
#pragma unroll
    for (int m = 0; m < 2; m++)
#pragma unroll
        for (int n = 0; n < NT; n++) {
            float *r = red + ((warp * 2 + m) * kRows) * TT + 8 * n + 2 * c;
            r[g * TT] = acc[m][n][0];
            r[g * TT + 1] = acc[m][n][1];
            r[(g + 8) * TT] = acc[m][n][2];
            r[(g + 8) * TT + 1] = acc[m][n][3];
        }
    __syncthreads();
    for (int i = threadIdx.x; i < T * kRows; i += kThreads) {
        const int t = i / kRows, r = i % kRows;  // consecutive threads: consecutive rows of one token
        float gs = 0.0f, us = 0.0f;
#pragma unroll 4
        for (int w = 0; w < kWarps; w++) {
            gs += red[((w * 2 + 0) * kRows + r) * TT + t];
            us += red[((w * 2 + 1) * kRows + r) * TT + t];
        }
        const float hv = swiglu(gs, us);
        if (!(fabsf(hv) <= 65504.0f)) *p.ovf_shared = 1;
        p.h16[static_cast<size_t>(t) * F + row0 + r] = __half_as_ushort(__float2half_rn(hv));
    }
}

template <int NT>
int launch_nt(const SharedParams &p, cudaStream_t s) {
    static int seen[64];
    const int smem = kWarps * 2 * kRows * NT * 8 * 4;
    const int err = ensure_smem(reinterpret_cast<const void *>(shared_up_kernel<NT>), smem, seen);
    if (err) return err;
    return launch_pdl(shared_up_kernel<NT>, dim3(p.F / kRows), dim3(kThreads), static_cast<size_t>(smem), s, p);
}

}  // namespace

int shared_small_max_tokens() { return kMaxTiles * 8; }

int launch_shared_up_small(const DeviceWeights &w, const Workspace &ws, const uint16_t *x, int T, int k,
                           void *stream) {
    SharedParams p;
    p.x = x;
    p.wg = w.sh_gate;
    p.wu = w.sh_up;
    p.h16 = ws.h16 + static_cast<size_t>(T) * k * w.F;  // rows P .. P+T-1
    p.T = T;
    p.D = w.D;
    p.F = w.F;
    p.ovf_shared = ws.ovf + w.E;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    switch ((T + 7) / 8) {
        case 1: return launch_nt<1>(p, s);
        case 2: return launch_nt<2>(p, s);
        case 3: return launch_nt<3>(p, s);
        case 4: return launch_nt<4>(p, s);
        case 5: return launch_nt<5>(p, s);
        default: return launch_nt<6>(p, s);
    }
}

}  // namespace ds4moe
