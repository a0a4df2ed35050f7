// ds4moe_expert_ffn_static: the expert FFN for callers that cannot allocate device memory.
//
// Its per-call intermediates (top-k arrays, grouping, h, y) live in one fixed region of
// device memory that the library reserves when it is loaded, instead of in the workspace
// that ds4moe_weights_create allocates. It runs the same kernels as ds4moe_expert_ffn with
// every expert group on the dequant-GEMV path. Nothing here calls cudaMalloc or cudaFree.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "internal.h"

using namespace ds4moe;

namespace {

constexpr size_t kStaticScratchBytes = size_t(3) << 20;  // 3 MiB on every device that loads the library

__device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
unsigned char *g_scratch_addr[kMaxDevices];  // device address of g_static_scratch, per device

// Device address of the static region on the current device, looked up once per device.
// In host code the symbol is only a host-side stand-in; cudaGetSymbolAddress gives the
// address that kernels may use.
int scratch_address(int dev, unsigned char **out) {
    if (dev < 0 || dev >= kMaxDevices) return DS4MOE_EUNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return DS4MOE_ECUDA;
        }
        g_scratch_addr[dev] = static_cast<unsigned char *>(p);
    }
    *out = g_scratch_addr[dev];
    return DS4MOE_OK;
}

size_t round256(size_t n) { return (n + 255) & ~size_t(255); }

// Carves the workspace of one call out of the static region; returns the bytes needed.
size_t carve(unsigned char *base, int T, int k, int E, int D, int F, Workspace *ws) {
    const size_t P = static_cast<size_t>(T) * k, rows = P + T;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        unsigned char *p = base ? base + off : nullptr;
        off += round256(bytes);
        return p;
    };
    ws->topk_idx = reinterpret_cast<int32_t *>(take(P * 4));
    ws->topk_w = reinterpret_cast<float *>(take(P * 4));
    ws->counts = reinterpret_cast<int32_t *>(take(static_cast<size_t>(E) * 4));
    ws->offsets = reinterpret_cast<int32_t *>(take((static_cast<size_t>(E) + 1) * 4));
    ws->perm = reinterpret_cast<int32_t *>(take(P * 4));
    ws->inv = reinterpret_cast<int32_t *>(take(P * 4));
    ws->gemv_list = reinterpret_cast<int32_t *>(take(static_cast<size_t>(E) * 4));
    ws->gemm_list = reinterpret_cast<int32_t *>(take(static_cast<size_t>(E) * 4));
    ws->meta = reinterpret_cast<GroupMeta *>(take(sizeof(GroupMeta)));
    ws->h32 = reinterpret_cast<float *>(take(rows * F * 4));
    ws->y = reinterpret_cast<float *>(take(rows * D * 4));
    ws->tile_prefix = nullptr;
    ws->tile_desc = nullptr;
    ws->single_list = nullptr;
    ws->h16 = nullptr;
    ws->x16 = nullptr;
    return off;
}

}  // namespace

extern "C" int ds4moe_expert_ffn_static(const uint16_t *x, const ds4moe_weights *h, const float *logits, int T, int k,
                                        int gate_mode, float *out, ds4moe_stream_t stream) {
    if (!h) return DS4MOE_EINVAL;
    if (h->pool.S) return DS4MOE_EUNSUPPORTED;  // the slot state lives in the handle's workspace
    if (h->dw.fmt != 0) return DS4MOE_EUNSUPPORTED;  // the 4-bit variant's GEMV needs the int16 token scratch
    const DeviceWeights &w = h->dw;
    if (T < 0 || k < 1 || k > 32 || k > w.E) return DS4MOE_EINVAL;
    if (gate_mode != DS4MOE_GATE_SOFTMAX && gate_mode != DS4MOE_GATE_SIGMOID) return DS4MOE_EINVAL;
    if (T == 0) return DS4MOE_OK;
    if (!x || !logits || !out || (reinterpret_cast<uintptr_t>(x) & 15u) || (reinterpret_cast<uintptr_t>(out) & 15u))
        return DS4MOE_EINVAL;
    Workspace ws{};
    if (carve(nullptr, T, k, w.E, w.D, w.F, &ws) > kStaticScratchBytes) return DS4MOE_EINVAL;  // too big for the region
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return DS4MOE_ECUDA;
    }
    if (dev != h->device) return DS4MOE_EINVAL;  // the handle's weights live on another device
    unsigned char *base = nullptr;
    const int rc0 = scratch_address(dev, &base);
    if (rc0 != DS4MOE_OK) return rc0;
    carve(base, T, k, w.E, w.D, w.F, &ws);
    ws.max_T = T;
    ws.max_k = k;
    ws.grid = h->ws.grid;      // read-only grid of the handle
    ws.status = h->ws.status;  // errors are reported through the handle, as for ds4moe_expert_ffn
    int rc = launch_route(logits, T, w.E, k, gate_mode, ws.topk_idx, ws.topk_w, stream);
    if (!rc)
        rc = launch_group(ws.topk_idx, T, k, w.E, 0, nullptr, ws.counts, ws.offsets, ws.perm, ws.inv, ws.gemv_list,
                          ws.gemm_list, nullptr, nullptr, nullptr, nullptr, ws.meta, ws.status, stream);
    if (!rc) rc = launch_gemv_up(w, ws, x, T, k, true, stream);
    if (!rc) rc = launch_gemv_down(w, ws, T, k, true, stream);
    if (!rc) rc = launch_combine(w, ws, T, k, 0, false, out, stream);
    return rc ? DS4MOE_ECUDA : DS4MOE_OK;
}
