// The C ABI: weights handle (validation, repack, upload, workspace), the device entry points
// and their launch sequence. Arguments are checked here, on the host, before any launch.
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "internal.h"

using namespace ds4moe;

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Test hook (ds4moe_test_fail_allocation): the n-th device allocation from now fails.
std::atomic<int> g_fail_countdown{0};

bool forced_failure() {
    int n = g_fail_countdown.load();
    while (n > 0 && !g_fail_countdown.compare_exchange_weak(n, n - 1)) {
    }
    return n == 1;
}

template <class T>
int dev_alloc(ds4moe_weights *h, T **p, size_t bytes) {
    *p = nullptr;
    if (h->n_allocs >= static_cast<int>(sizeof(h->allocs) / sizeof(h->allocs[0]))) return DS4MOE_ENOMEM;
    if (forced_failure()) return DS4MOE_ENOMEM;
    void *q = nullptr;
    if (cudaMalloc(&q, bytes ? bytes : 16) != cudaSuccess) {
        cudaGetLastError();
        return DS4MOE_ENOMEM;
    }
    h->allocs[h->n_allocs++] = q;
    *p = static_cast<T *>(q);
    return DS4MOE_OK;
}

void free_all(ds4moe_weights *h) {
    for (int i = 0; i < h->n_allocs; i++) cudaFree(h->allocs[i]);
    h->n_allocs = 0;
    for (int i = 0; i < h->n_host_allocs; i++) cudaFreeHost(h->host_allocs[i]);
    h->n_host_allocs = 0;
}

// Pinned host memory that the device can read (device-mapped); *dev receives its device address.
template <class T>
int host_alloc(ds4moe_weights *h, T **p, const uint8_t **dev, size_t bytes) {
    *p = nullptr;
    if (h->n_host_allocs >= static_cast<int>(sizeof(h->host_allocs) / sizeof(h->host_allocs[0]))) return DS4MOE_ENOMEM;
    void *q = nullptr, *d = nullptr;
    if (cudaHostAlloc(&q, bytes ? bytes : 16, cudaHostAllocMapped) != cudaSuccess) {
        cudaGetLastError();
        return DS4MOE_ENOMEM;
    }
    h->host_allocs[h->n_host_allocs++] = q;
    if (cudaHostGetDevicePointer(&d, q, 0) != cudaSuccess) {
        cudaGetLastError();
        return DS4MOE_ECUDA;
    }
    *p = static_cast<T *>(q);
    *dev = static_cast<const uint8_t *>(d);
    return DS4MOE_OK;
}

int cuda_status(int err) {
    if (err == 0) return DS4MOE_OK;
    return DS4MOE_ECUDA;
}

#define TRY(x)                        \
    do {                              \
        const int rc_ = (x);          \
        if (rc_ != DS4MOE_OK) {       \
            free_all(h);              \
            delete h;                 \
            return rc_;               \
        }                             \
    } while (0)

int upload(void *dst, const void *src, size_t bytes) {
    return cudaMemcpy(dst, src, bytes, cudaMemcpyHostToDevice) == cudaSuccess ? DS4MOE_OK : DS4MOE_ECUDA;
}

constexpr double kF16Max = 65504.0;

// Split IQ2-style blocks [rows][nb][66] into payload [rows][nb][64] and scales [rows][nb].
// amax: a bound on |weight| over the blocks (7 d).
bool repack_iq2(const uint8_t *src, size_t nblocks, uint8_t *qs, uint16_t *d, double *amax) {
    for (size_t b = 0; b < nblocks; b++) {
        const uint8_t *blk = src + b * 66;
        const uint16_t dv = static_cast<uint16_t>(blk[0] | (blk[1] << 8));
        if (!host_f16_finite(dv)) return false;
        const double bound = 7.0 * std::fabs(host_f16_value(dv));
        if (bound > *amax) *amax = bound;
        d[b] = dv;
        std::memcpy(qs + b * 64, blk + 2, 64);
    }
    return true;
}

// Split Q2_K-style blocks [rows][nb][84] into payload [rows][nb][80] and (d, dmin) pairs.
// amax: a bound on |weight| over the blocks (max(45 |d|, 15 |dmin|) + ...).
bool repack_q2k(const uint8_t *src, size_t nblocks, uint8_t *sq, uint32_t *dd, double *amax) {
    for (size_t b = 0; b < nblocks; b++) {
        const uint8_t *blk = src + b * 84;
        const uint16_t dv = static_cast<uint16_t>(blk[80] | (blk[81] << 8));
        const uint16_t mv = static_cast<uint16_t>(blk[82] | (blk[83] << 8));
        if (!host_f16_finite(dv) || !host_f16_finite(mv)) return false;
        const double bound = 45.0 * std::fabs(host_f16_value(dv)) + 15.0 * std::fabs(host_f16_value(mv));
        if (bound > *amax) *amax = bound;
        dd[b] = static_cast<uint32_t>(dv) | (static_cast<uint32_t>(mv) << 16);
        std::memcpy(sq + b * 80, blk, 80);
    }
    return true;
}

// bf16 bits -> fp16 bits, nearest-even (exact for values in fp16's normal range).
uint16_t bf16_to_f16(uint16_t b) {
    const uint32_t u = static_cast<uint32_t>(b) << 16;  // the binary32 value of the bf16
    const uint32_t sign = (u >> 16) & 0x8000u;
    const uint32_t mag = u & 0x7fffffffu;
    if (mag >= 0x7f800000u) return static_cast<uint16_t>(sign | (mag > 0x7f800000u ? 0x7e00u : 0x7c00u));
    const int e = static_cast<int>(mag >> 23) - 127;
    if (e > 15) return static_cast<uint16_t>(sign | 0x7c00u);
    if (e < -25) return static_cast<uint16_t>(sign);
    const uint32_t sig = (mag & 0x7fffffu) | 0x800000u;
    const int drop = e >= -14 ? 13 : 13 + (-14 - e);
    uint32_t q = sig >> drop;
    const uint32_t rem = sig & ((1u << drop) - 1u), half = 1u << (drop - 1);
    if (rem > half || (rem == half && (q & 1u))) q++;
    uint32_t h = e >= -14 ? (static_cast<uint32_t>(e + 15) << 10) + (q - 1024u) : q;
    if (h >= 0x7c00u) h = 0x7c00u;
    return static_cast<uint16_t>(sign | h);
}

// Every block of a handle's blobs must have finite fp16 scales; checked before anything is
// allocated, so a rejected blob costs no device call.
bool blobs_valid(const ds4moe_weights_desc *desc, int fmt) {
    const size_t nb_up = static_cast<size_t>(desc->d_ff) * (desc->d_model / 256);
    const size_t nb_down = static_cast<size_t>(desc->d_model) * (desc->d_ff / 256);
    auto ok = [](const uint8_t *blk, int at) {
        return host_f16_finite(static_cast<uint16_t>(blk[at] | (blk[at + 1] << 8)));
    };
    for (int e = 0; e < desc->n_experts; e++) {
        const uint8_t *mats[3] = {static_cast<const uint8_t *>(desc->gate_iq2[e]),
                                  static_cast<const uint8_t *>(desc->up_iq2[e]),
                                  static_cast<const uint8_t *>(desc->down_q2k[e])};
        for (int m = 0; m < 3; m++) {
            const size_t nb = m < 2 ? nb_up : nb_down;
            for (size_t b = 0; b < nb; b++) {
                if (fmt == 1) {  // Q4_K-style: d, dmin at bytes 0 and 2 of 144
                    const uint8_t *blk = mats[m] + b * 144;
                    if (!ok(blk, 0) || !ok(blk, 2)) return false;
                } else if (m < 2) {  // IQ2-style: d at byte 0 of 66
                    if (!ok(mats[m] + b * 66, 0)) return false;
                } else {  // Q2_K-style: d, dmin at bytes 80 and 82 of 84
                    const uint8_t *blk = mats[m] + b * 84;
                    if (!ok(blk, 80) || !ok(blk, 82)) return false;
                }
            }
        }
    }
    return true;
}

// Counts launches per stage and, when profiling, records an event at each stage start and
// one at the end of the call, all on the call's stream. Each stage is also an NVTX range
// ("ds4moe:<stage>") on the host thread that issues its launches, for timeline tools.
const char *const kStageNames[DS4MOE_N_STAGES] = {
    "ds4moe:route", "ds4moe:group", "ds4moe:gather", "ds4moe:up_gemv", "ds4moe:up_gemm",
    "ds4moe:down_gemv", "ds4moe:down_gemm", "ds4moe:combine", "ds4moe:step", "ds4moe:pool", "ds4moe:repair"};

struct StageClock {
    ds4moe_weights *h;
    cudaStream_t s;
    bool range_open = false;
    StageClock(ds4moe_weights *h_, ds4moe_stream_t s_) : h(h_), s(s_) {
        for (bool &r : h->stage_ran) r = false;
        h->events_recorded = false;
        h->n_stage_order = 0;
    }
    ~StageClock() { close_range(); }
    void close_range() {
        if (range_open) nvtxRangePop();
        range_open = false;
    }
    int stage(int i) {
        close_range();
        nvtxRangePushA(kStageNames[i]);
        range_open = true;
        h->stage_ran[i] = true;
        h->stage_order[h->n_stage_order++] = i;
        h->launches++;
        if (!h->profile) return 0;
        return static_cast<int>(cudaEventRecord(static_cast<cudaEvent_t>(h->events[i]), s));
    }
    int finish() {
        close_range();
        if (!h->profile) return 0;
        h->events_recorded = true;
        return static_cast<int>(cudaEventRecord(static_cast<cudaEvent_t>(h->events[DS4MOE_N_STAGES]), s));
    }
};

}  // namespace

extern "C" {

// n_slots = 0: every expert resident in device memory; otherwise a pooled handle (see
// ds4moe_weights_create_pooled) whose device weights are n_slots expert slots. fmt 1: the 4-bit
// variant (Q4_K-style blobs for all three projections, resident).
static int create_impl(const ds4moe_weights_desc *desc, int n_slots, int fmt, ds4moe_weights **out) {
    if (!desc || !out) return DS4MOE_EINVAL;
    *out = nullptr;
    const int D = desc->d_model, F = desc->d_ff, E = desc->n_experts;
    if (D <= 0 || F <= 0 || D % 256 || F % 256 || E < 1 || E > 1024) return DS4MOE_EINVAL;
    if (desc->max_tokens < 1 || desc->max_k < 1 || desc->max_k > 32 || desc->max_k > E) return DS4MOE_EINVAL;
    if (n_slots < 0 || (n_slots > 0 && (n_slots > E || n_slots < desc->max_k))) return DS4MOE_EINVAL;
    if (fmt == 1 && n_slots) return DS4MOE_EUNSUPPORTED;  // the 4-bit variant is resident only
    const int S = n_slots ? n_slots : E;  // experts held in device memory
    if (!desc->gate_iq2 || !desc->up_iq2 || !desc->down_q2k) return DS4MOE_EINVAL;
    for (int e = 0; e < E; e++)
        if (!desc->gate_iq2[e] || !desc->up_iq2[e] || !desc->down_q2k[e]) return DS4MOE_EINVAL;
    const int n_shared = (desc->shared_gate_bf16 != nullptr) + (desc->shared_up_bf16 != nullptr) +
                         (desc->shared_down_bf16 != nullptr);
    if (n_shared != 0 && n_shared != 3) return DS4MOE_EINVAL;
    const int64_t P = static_cast<int64_t>(desc->max_tokens) * desc->max_k;
    if (P > (int64_t(1) << 30)) return DS4MOE_EINVAL;
    if (!blobs_valid(desc, fmt)) return DS4MOE_EBADDATA;

    ds4moe_weights *h = new (std::nothrow) ds4moe_weights();
    if (!h) return DS4MOE_ENOMEM;
    if (cudaGetDevice(&h->device) != cudaSuccess) {
        cudaGetLastError();
        delete h;
        return DS4MOE_ECUDA;
    }
    h->gemm_min_tokens = -1;
    h->shared_gemm_min_tokens = 2;
    h->single_step = 1;
    h->small_groups = 1;
    h->gemm_pairs = 0;
    DeviceWeights &w = h->dw;
    w.D = D;
    w.F = F;
    w.E = S;
    w.nbD = D / 256;
    w.nbF = F / 256;
    w.has_shared = n_shared == 3;
    const size_t nb_up = static_cast<size_t>(F) * w.nbD;    // blocks per gate/up matrix
    const size_t nb_down = static_cast<size_t>(D) * w.nbF;  // blocks per down matrix
    const size_t up_bytes = nb_up * 132;       // gate + up of one expert, tiled (66 bytes per block each)
    const size_t down_bytes = nb_down * 84;    // down of one expert, tiled
    w.fmt = fmt;
    if (fmt == 1) {
        // the 4-bit variant: each expert's gate, up and down blocks as given, validated (finite
        // fp16 d and dmin in every block), in row order; never on the tensor-core path
        const size_t q4b = q4_expert_bytes(w);
        TRY(dev_alloc(h, &w.q4, E * q4b));
        TRY(dev_alloc(h, &w.iq2, 16));
        TRY(dev_alloc(h, &w.q2k, 16));
        TRY(dev_alloc(h, &w.tc_ok, E));
        const size_t gb = nb_up * 144, db = nb_down * 144;
        std::vector<uint8_t> ok(E);
        for (int e = 0; e < E; e++) {
            double amax = 0.0;  // a bound on |weight|: 63 * 15 |d| + 63 |dmin| per block
            const uint8_t *mats[3] = {static_cast<const uint8_t *>(desc->gate_iq2[e]),
                                      static_cast<const uint8_t *>(desc->up_iq2[e]),
                                      static_cast<const uint8_t *>(desc->down_q2k[e])};
            for (int m = 0; m < 3; m++) {
                const size_t nbk = m < 2 ? nb_up : nb_down;
                for (size_t b = 0; b < nbk; b++) {
                    const uint8_t *blk = mats[m] + b * 144;
                    const uint16_t dv = static_cast<uint16_t>(blk[0] | (blk[1] << 8));
                    const uint16_t mv = static_cast<uint16_t>(blk[2] | (blk[3] << 8));
                    if (!host_f16_finite(dv) || !host_f16_finite(mv)) TRY(DS4MOE_EBADDATA);
                    const double bound = 945.0 * std::fabs(host_f16_value(dv)) + 63.0 * std::fabs(host_f16_value(mv));
                    if (bound > amax) amax = bound;
                }
            }
            ok[e] = amax <= kF16Max ? 1 : 0;  // otherwise the expert stays on the GEMV path
            TRY(upload(w.q4 + e * q4b, mats[0], gb));
            TRY(upload(w.q4 + e * q4b + gb, mats[1], gb));
            TRY(upload(w.q4 + e * q4b + 2 * gb, mats[2], db));
        }
        TRY(upload(w.tc_ok, ok.data(), E));
    }
    if (fmt == 0) {
        TRY(dev_alloc(h, &w.iq2, S * up_bytes));
        TRY(dev_alloc(h, &w.q2k, S * down_bytes));
        TRY(dev_alloc(h, &w.tc_ok, S));
    }
    SlotPool &sp = h->pool;
    uint8_t *store_iq2 = nullptr, *store_q2k = nullptr, *store_ok = nullptr;  // pooled: host views of the store
    if (n_slots) {
        sp.S = S;
        sp.E = E;
        sp.up_bytes = up_bytes;
        sp.down_bytes = down_bytes;
        TRY(host_alloc(h, &store_iq2, &sp.host_iq2, E * up_bytes));
        TRY(host_alloc(h, &store_q2k, &sp.host_q2k, E * down_bytes));
        TRY(host_alloc(h, &store_ok, &sp.host_tc_ok, E));
        TRY(dev_alloc(h, &sp.slot_of, E * 4));
        TRY(dev_alloc(h, &sp.expert_of, S * 4));
        TRY(dev_alloc(h, &sp.stamp, S * 4));
        TRY(dev_alloc(h, &sp.ctr, 4 * 8));
        TRY(dev_alloc(h, &sp.miss, S * 8));
        // no expert resident yet; empty slots hold zero blocks (every weight 0)
        if (cudaMemset(sp.slot_of, 0xff, E * 4) != cudaSuccess || cudaMemset(sp.expert_of, 0xff, S * 4) != cudaSuccess ||
            cudaMemset(sp.stamp, 0, S * 4) != cudaSuccess || cudaMemset(sp.ctr, 0, 32) != cudaSuccess ||
            cudaMemset(sp.miss, 0, S * 8) != cudaSuccess || cudaMemset(w.iq2, 0, S * up_bytes) != cudaSuccess ||
            cudaMemset(w.q2k, 0, S * down_bytes) != cudaSuccess || cudaMemset(w.tc_ok, 0, S) != cudaSuccess)
            TRY(DS4MOE_ECUDA);
    }
    if (fmt == 0) {
        std::vector<uint8_t> qs(nb_up * 64), sq(nb_down * 80), ok(E), tiles(std::max(up_bytes, down_bytes));
        std::vector<uint16_t> dv(nb_up);
        std::vector<uint32_t> dd(nb_down);
        DeviceWeights w0 = w;  // offsets of expert 0: the host staging buffer holds one expert
        for (int e = 0; e < E; e++) {
            const void *mats[2] = {desc->gate_iq2[e], desc->up_iq2[e]};
            double amax = 0.0;
            for (int m = 0; m < 2; m++) {
                if (!repack_iq2(static_cast<const uint8_t *>(mats[m]), nb_up, qs.data(), dv.data(), &amax))
                    TRY(DS4MOE_EBADDATA);
                for (int r = 0; r < F; r++) {
                    const int swz = iq2_swz(w0, r);
                    for (int q = 0; q < 4 * w.nbD; q++)  // 16-byte chunks, permuted within the row
                        std::memcpy(tiles.data() + iq2_qs_offset(w0, m, 0, r) + static_cast<size_t>(q ^ swz) * 16,
                                    qs.data() + static_cast<size_t>(r) * w.nbD * 64 + static_cast<size_t>(q) * 16, 16);
                    std::memcpy(tiles.data() + iq2_d_offset(w0, m, 0, r), dv.data() + static_cast<size_t>(r) * w.nbD,
                                static_cast<size_t>(w.nbD) * 2);
                }
            }
            if (n_slots)
                std::memcpy(store_iq2 + e * up_bytes, tiles.data(), up_bytes);
            else
                TRY(upload(w.iq2 + e * up_bytes, tiles.data(), up_bytes));
            if (!repack_q2k(static_cast<const uint8_t *>(desc->down_q2k[e]), nb_down, sq.data(), dd.data(), &amax))
                TRY(DS4MOE_EBADDATA);
            for (int r = 0; r < D; r++) {
                std::memcpy(tiles.data() + q2k_sq_offset(w0, 0, r), sq.data() + static_cast<size_t>(r) * w.nbF * 80,
                            static_cast<size_t>(w.nbF) * 80);
                std::memcpy(tiles.data() + q2k_dd_offset(w0, 0, r), dd.data() + static_cast<size_t>(r) * w.nbF,
                            static_cast<size_t>(w.nbF) * 4);
            }
            if (n_slots)
                std::memcpy(store_q2k + e * down_bytes, tiles.data(), down_bytes);
            else
                TRY(upload(w.q2k + e * down_bytes, tiles.data(), down_bytes));
            ok[e] = amax <= kF16Max ? 1 : 0;  // otherwise the expert stays on the fp32 GEMV path
        }
        if (n_slots)
            std::memcpy(store_ok, ok.data(), E);
        else
            TRY(upload(w.tc_ok, ok.data(), E));
    }
    if (w.has_shared) {
        const size_t n = static_cast<size_t>(F) * D;
        TRY(dev_alloc(h, &w.sh_gate, n * 2));
        TRY(dev_alloc(h, &w.sh_up, n * 2));
        TRY(dev_alloc(h, &w.sh_down, n * 2));
        TRY(dev_alloc(h, &w.sh_down_f16, n * 2));
        TRY(upload(w.sh_gate, desc->shared_gate_bf16, n * 2));
        TRY(upload(w.sh_up, desc->shared_up_bf16, n * 2));
        TRY(upload(w.sh_down, desc->shared_down_bf16, n * 2));
        std::vector<uint16_t> f16(n);
        for (size_t i = 0; i < n; i++) f16[i] = bf16_to_f16(desc->shared_down_bf16[i]);
        TRY(upload(w.sh_down_f16, f16.data(), n * 2));
        // the tensor-core path holds the shared expert in fp16: only if every weight fits
        w.shared_tc_ok = true;
        const uint16_t *mats[3] = {desc->shared_gate_bf16, desc->shared_up_bf16, desc->shared_down_bf16};
        for (const uint16_t *m : mats)
            for (size_t i = 0; i < n && w.shared_tc_ok; i++)
                if ((m[i] & 0x7fffu) > 0x477fu) w.shared_tc_ok = false;  // |bf16| > 65280 (or inf/nan)
    }
    Workspace &ws = h->ws;
    ws.max_T = desc->max_tokens;
    ws.max_k = desc->max_k;
    const size_t rows = static_cast<size_t>(P) + desc->max_tokens;
    TRY(dev_alloc(h, &ws.topk_idx, P * 4));
    TRY(dev_alloc(h, &ws.topk_w, P * 4));
    TRY(dev_alloc(h, &ws.counts, E * 4));
    TRY(dev_alloc(h, &ws.offsets, (E + 1) * 4));
    TRY(dev_alloc(h, &ws.perm, P * 4));
    TRY(dev_alloc(h, &ws.inv, P * 4));
    TRY(dev_alloc(h, &ws.gemv_list, E * 4));
    TRY(dev_alloc(h, &ws.gemm_list, E * 4));
    TRY(dev_alloc(h, &ws.single_list, E * 4));
    TRY(dev_alloc(h, &ws.tile_prefix, (E + 1) * 4));
    TRY(dev_alloc(h, &ws.tile_desc, (E + P / kGemmBN + 1) * 16));
    TRY(dev_alloc(h, &ws.meta, sizeof(GroupMeta)));
    TRY(dev_alloc(h, &ws.meta2, sizeof(GroupMeta)));
    TRY(dev_alloc(h, &ws.ovf, (E + 1) * 4));
    TRY(dev_alloc(h, &ws.repair_list, E * 4));
    if (cudaMemset(ws.ovf, 0, (E + 1) * 4) != cudaSuccess) TRY(DS4MOE_ECUDA);
    TRY(dev_alloc(h, &ws.grid, 2048));
    TRY(dev_alloc(h, &ws.h32, rows * F * 4));
    const size_t rows_tc = std::max<size_t>(rows, kGemmBN);  // at least one full token box
    TRY(dev_alloc(h, &ws.h16, rows_tc * F * 2));
    TRY(dev_alloc(h, &ws.x16, rows_tc * D * 2));
    if (encode_token_maps(h->tmap_x16, ws.x16, static_cast<int>(rows_tc), D) ||
        encode_token_maps(h->tmap_h16, ws.h16, static_cast<int>(rows_tc), F))
        TRY(DS4MOE_ECUDA);
    TRY(dev_alloc(h, &ws.y, rows * D * 4));
    TRY(dev_alloc(h, &ws.status, 16));
    TRY(dev_alloc(h, &ws.gbar, 16));
    TRY(dev_alloc(h, &ws.hmax, 1024 * 8 * 4));
    TRY(dev_alloc(h, &ws.trace, 1024 * 6 * 8));
    TRY(dev_alloc(h, &ws.small_pos, P * 4));
    TRY(dev_alloc(h, &ws.xq, static_cast<size_t>(desc->max_tokens) * D * 2));
    TRY(dev_alloc(h, &ws.x8, static_cast<size_t>(desc->max_tokens) * (D / 32) * 4));
    TRY(dev_alloc(h, &ws.xsc, static_cast<size_t>(desc->max_tokens) * 16));
    if (fmt == 1) {  // the 4-bit variant's int16 h (calls of up to 64 tokens)
        const size_t P64 = static_cast<size_t>(std::min<int64_t>(P, 64 * desc->max_k));
        TRY(dev_alloc(h, &ws.hq4, P64 * F * 2));
        TRY(dev_alloc(h, &ws.hsum4, P64 * (F / 32) * 4));
        TRY(dev_alloc(h, &ws.hsc4, P64 * 4));
    }
    if (cudaMemset(ws.gbar, 0, 16) != cudaSuccess) TRY(DS4MOE_ECUDA);
    TRY(dev_alloc(h, &ws.grid_hi, 2048));
    {
        uint8_t g[2048], hb[2048];
        host_grid(g);
        for (int i = 0; i < 2048; i++) hb[i] = g[i] == 1 ? 0x3C : g[i] == 3 ? 0x42 : g[i] == 5 ? 0x45 : 0x47;
        TRY(upload(ws.grid, g, 2048));
        TRY(upload(ws.grid_hi, hb, 2048));
    }
    if (cudaMemset(ws.status, 0, 16) != cudaSuccess) TRY(DS4MOE_ECUDA);
    if (cudaDeviceSynchronize() != cudaSuccess) TRY(DS4MOE_ECUDA);
    *out = h;
    return DS4MOE_OK;
}

int ds4moe_weights_create(const ds4moe_weights_desc *desc, ds4moe_weights **out) { return create_impl(desc, 0, 0, out); }

int ds4moe_test_fail_allocation(int n) {
    if (n < 0) return DS4MOE_EINVAL;
    g_fail_countdown.store(n);
    return DS4MOE_OK;
}

int ds4moe_weights_create_q4(const ds4moe_weights_desc *desc, ds4moe_weights **out) { return create_impl(desc, 0, 1, out); }

int ds4moe_weights_create_pooled(const ds4moe_weights_desc *desc, int n_slots, ds4moe_weights **out) {
    if (n_slots < 1) {
        if (out) *out = nullptr;
        return DS4MOE_EINVAL;
    }
    return create_impl(desc, n_slots, 0, out);
}

int ds4moe_pool_info(ds4moe_weights *h, int *n_slots, uint64_t *hits, uint64_t *misses, int32_t *slot_expert) {
    if (!h || !h->pool.S) return DS4MOE_EINVAL;
    unsigned long long c[4] = {0, 0, 0, 0};
    if (cudaDeviceSynchronize() != cudaSuccess || cudaMemcpy(c, h->pool.ctr, sizeof c, cudaMemcpyDeviceToHost) != cudaSuccess ||
        (slot_expert && cudaMemcpy(slot_expert, h->pool.expert_of, static_cast<size_t>(h->pool.S) * 4,
                                   cudaMemcpyDeviceToHost) != cudaSuccess)) {
        cudaGetLastError();
        return DS4MOE_ECUDA;
    }
    if (n_slots) *n_slots = h->pool.S;
    if (hits) *hits = c[1];
    if (misses) *misses = c[2];
    return DS4MOE_OK;
}

void ds4moe_weights_destroy(ds4moe_weights *h) {
    if (!h) return;
    int cur = 0;
    cudaGetDevice(&cur);
    cudaSetDevice(h->device);
    cudaDeviceSynchronize();
    for (auto &ev : h->events)
        if (ev) cudaEventDestroy(static_cast<cudaEvent_t>(ev));
    free_all(h);
    cudaSetDevice(cur);
    delete h;
}

int ds4moe_set_option(ds4moe_weights *h, int option, int value) {
    if (!h || (value < 0 && !(option == DS4MOE_OPT_GEMM_MIN_TOKENS && value == -1))) return DS4MOE_EINVAL;
    switch (option) {
        case DS4MOE_OPT_GEMM_MIN_TOKENS: h->gemm_min_tokens = value; return DS4MOE_OK;
        case DS4MOE_OPT_SHARED_GEMM_MIN_TOKENS: h->shared_gemm_min_tokens = value; return DS4MOE_OK;
        case DS4MOE_OPT_SINGLE_STEP: h->single_step = value ? 1 : 0; return DS4MOE_OK;
        case DS4MOE_OPT_SMALL_GROUPS: h->small_groups = value ? 1 : 0; return DS4MOE_OK;
        case DS4MOE_OPT_TRACE: h->trace = value ? 1 : 0; return DS4MOE_OK;
        case DS4MOE_OPT_WAIT_TEST: h->wait_test = value > 0 ? 1 : 0; return DS4MOE_OK;
        case DS4MOE_OPT_GEMM_PAIRS: h->gemm_pairs = value ? 1 : 0; return DS4MOE_OK;
        case DS4MOE_OPT_PROFILE:
            if (value && !h->events[0]) {
                for (auto &ev : h->events) {
                    cudaEvent_t e;
                    if (cudaEventCreate(&e) != cudaSuccess) return DS4MOE_ECUDA;
                    ev = e;
                }
            }
            h->profile = value ? 1 : 0;
            return DS4MOE_OK;
        default: return DS4MOE_EINVAL;
    }
}

int ds4moe_weights_dequantize(const ds4moe_weights *h, int expert, int matrix, float *dst_f32, uint16_t *dst_f16,
                              ds4moe_stream_t stream) {
    if (!h || expert < 0 || expert >= h->dw.E || matrix < 0 || matrix > 2 || (!dst_f32 && !dst_f16))
        return DS4MOE_EINVAL;
    if (h->pool.S) return DS4MOE_EUNSUPPORTED;  // a pooled handle's slots change from call to call
    if (h->dw.fmt == 1 && dst_f16) return DS4MOE_EUNSUPPORTED;  // the 4-bit variant has no fp16 operand path
    int rc = 0;
    if (dst_f32) rc = launch_dequant(h->dw, h->ws.grid, expert, matrix, dst_f32, nullptr, stream);
    // the fp16 values are the tensor-core path's own operand bytes, from its producers
    if (!rc && dst_f16) rc = launch_producer_dump(h->dw, h->ws.grid, expert, matrix, dst_f16, stream);
    return cuda_status(rc);
}

int ds4moe_router_logits(const void *x, const void *w_router, const float *bias, int T, int D, int E,
                         float *logits, ds4moe_stream_t stream) {
    if (T < 0 || D <= 0 || D % 256 || D > 8192 || E < 8 || E % 8 || E > 1024) return DS4MOE_EINVAL;
    if (T == 0) return DS4MOE_OK;
    if (!x || !w_router || !logits || !aligned16(x) || !aligned16(w_router)) return DS4MOE_EINVAL;
    if (reinterpret_cast<uintptr_t>(logits) % 4 || (bias && reinterpret_cast<uintptr_t>(bias) % 4)) return DS4MOE_EINVAL;
    return cuda_status(launch_router(static_cast<const uint16_t *>(x), static_cast<const uint16_t *>(w_router), bias, T,
                                     D, E, logits, stream));
}

int ds4moe_router_last_status(ds4moe_stream_t stream) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) {
        cudaGetLastError();
        return DS4MOE_ECUDA;
    }
    int st = 0;
    if (router_read_status(&st)) {
        cudaGetLastError();
        return DS4MOE_ECUDA;
    }
    return (st & ST_TIMEOUT) ? DS4MOE_ETIMEOUT : DS4MOE_OK;
}

int ds4moe_route(const float *logits, int T, int E, int k, int gate_mode, int32_t *topk_idx, float *topk_w,
                 ds4moe_stream_t stream) {
    if (T < 0 || E < 1 || E > 1024 || k < 1 || k > 32 || k > E) return DS4MOE_EINVAL;
    if (gate_mode != DS4MOE_GATE_SOFTMAX && gate_mode != DS4MOE_GATE_SIGMOID) return DS4MOE_EINVAL;
    if (T == 0) return DS4MOE_OK;
    if (!logits || !topk_idx || !topk_w) return DS4MOE_EINVAL;
    return cuda_status(launch_route(logits, T, E, k, gate_mode, topk_idx, topk_w, stream));
}

int ds4moe_group(const int32_t *topk_idx, int T, int k, int E, int32_t *counts, int32_t *offsets, int32_t *perm,
                 int32_t *inv, ds4moe_stream_t stream) {
    if (T < 0 || E < 1 || E > 1024 || k < 1 || k > 32) return DS4MOE_EINVAL;
    if (static_cast<int64_t>(T) * k > (int64_t(1) << 30)) return DS4MOE_EINVAL;
    if (!counts || !offsets || (T > 0 && (!topk_idx || !perm || !inv))) return DS4MOE_EINVAL;
    return cuda_status(launch_group(topk_idx, T, k, E, 0, nullptr, counts, offsets, perm, inv, nullptr, nullptr,
                                    nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, stream));
}

int ds4moe_expert_ffn(const uint16_t *x, ds4moe_weights *h, const float *logits, int T, int k, int gate_mode,
                      float *out, ds4moe_stream_t stream) {
    if (!h) return DS4MOE_EINVAL;
    if (T < 0 || T > h->ws.max_T || k < 1 || k > h->ws.max_k || k > h->dw.E) return DS4MOE_EINVAL;
    if (gate_mode != DS4MOE_GATE_SOFTMAX && gate_mode != DS4MOE_GATE_SIGMOID) return DS4MOE_EINVAL;
    if (T == 0) return DS4MOE_OK;
    if (!x || !logits || !out || !aligned16(x) || !aligned16(out)) return DS4MOE_EINVAL;
    const DeviceWeights &w = h->dw;
    const Workspace &ws = h->ws;
    StageClock clk(h, stream);
    const bool pooled = h->pool.S > 0;
    const int E_route = pooled ? h->pool.E : w.E;  // the experts the logits route over
    int rc = 0;
    if (pooled) {
        // a pooled handle routes first: slots for the touched experts, the missing ones copied
        // in, the top-k indices rewritten to slots (the fused kernel maps its own top-k)
        rc = clk.stage(DS4MOE_STAGE_ROUTE);
        if (!rc) rc = launch_route(logits, T, E_route, k, gate_mode, ws.topk_idx, ws.topk_w, stream);
        if (!rc) rc = clk.stage(DS4MOE_STAGE_POOL);
        if (!rc) rc = launch_pool_assign(h->pool, ws.topk_idx, T * k, ws.status, stream);
        if (!rc) rc = launch_pool_fill(h->pool, w, decode_step_ctas(), stream);
        h->launches++;
        if (rc) return cuda_status(rc);
    }
    if (T == 1 && h->single_step && decode_step_supported(w, k) &&
        !(h->gemm_min_tokens == 1 || (w.has_shared && h->shared_gemm_min_tokens == 1))) {
        // one token: routing, both expert phases and the combine in one cooperative kernel
        rc = clk.stage(DS4MOE_STAGE_STEP);
        if (!rc)
            rc = launch_decode_step(w, ws, x, logits, k, gate_mode, out, h->trace ? ws.trace : nullptr, E_route,
                                    pooled ? h->pool.slot_of : nullptr, static_cast<unsigned int>(h->wait_test), stream);
        if (!rc) {
            rc = clk.finish();
            h->calls++;
            return cuda_status(rc);
        }
        // the cooperative launch was refused (e.g. the SMs are shared): the separate kernels
        cudaGetLastError();
        h->stage_ran[DS4MOE_STAGE_STEP] = false;
        h->launches--;
        rc = 0;
    }
    // A group holds at most T tokens, so the tensor-core path can only be needed when
    // T reaches the threshold; the device decides per group after routing.
    const bool q4 = w.fmt == 1;  // the 4-bit variant: groups below the threshold on the dequant-GEMV kernels
    const bool sg_fits = !q4 && h->small_groups && small_groups_supported(w);
    // (the 4-bit variant has no small-group kernels: from 2 tokens its groups are cheaper on the
    // tensor cores than on the GEMV, measured on prefill_t2048_q4)
    // (without the small-group kernels, above 64 tokens even one-token groups are cheaper on the
    // tensor cores than on the single-token decode kernels: prefill_t8192_d7168 has ~30 of them)
    const int gm = h->gemm_min_tokens >= 0 ? h->gemm_min_tokens
                   : q4 ? (T <= 64 ? 0 : 2) : sg_fits ? (T <= 64 ? 0 : 7) : (T <= 64 ? 2 : 1);
    const int gemm_min = (gm > 0 && T >= gm) ? gm : 0;
    const bool shared_tc = w.has_shared && w.shared_tc_ok && h->shared_gemm_min_tokens > 0 &&
                           T >= h->shared_gemm_min_tokens;
    const bool any_tc = gemm_min > 0 || shared_tc;
    // The small-group kernels take every routed group below the threshold; the shared expert
    // must then be on the tensor cores, or (T = 1) on the single-token decode kernels.
    const bool sg = sg_fits && (!w.has_shared || shared_tc || T == 1);
    // With few tokens the shared expert's gate/up runs on its own warp-MMA kernel (one CTA per 16
    // rows) and only its down projection on the tensor-core kernel.
    // (Not when the caller forces everything onto the tensor cores with a threshold of 1.)
    const bool shared_up_small = sg && shared_tc && T <= shared_small_max_tokens() && h->gemm_min_tokens != 1 &&
                                 h->shared_gemm_min_tokens != 1;
    const bool up_tc = gemm_min > 0 || (shared_tc && !shared_up_small);
    if (!pooled) {  // (a pooled handle has routed already)
        rc = clk.stage(DS4MOE_STAGE_ROUTE);
        if (!rc) rc = launch_route(logits, T, w.E, k, gate_mode, ws.topk_idx, ws.topk_w, stream);
    }
    if (!rc) rc = clk.stage(DS4MOE_STAGE_GROUP);
    if (!rc)
        rc = launch_group(ws.topk_idx, T, k, w.E, gemm_min, w.tc_ok, ws.counts, ws.offsets, ws.perm, ws.inv,
                          ws.gemv_list, ws.gemm_list, (sg || q4) ? nullptr : ws.single_list, ws.tile_prefix, ws.tile_desc,
                          sg ? ws.small_pos : nullptr, ws.meta, ws.status, stream, ws.ovf);
    if (up_tc) {
        if (!rc) rc = clk.stage(DS4MOE_STAGE_GATHER);
        if (!rc) rc = launch_gather(w, ws, x, T, k, gemm_min, shared_tc && !shared_up_small, stream);
    }
    // Without the small-group kernels: one-token groups (every group at T = 1) run on the
    // decode kernels; groups of 2 .. gemm_min-1 tokens on the multi-token GEMV kernels, which
    // are launched only when such groups can exist; larger groups on the tensor cores.
    const bool multi_gemv = q4 || (!sg && (gemm_min == 0 ? T > 1 : gemm_min > 2));
    // (the 4-bit variant takes its shared expert into the GEMV launches at every T)
    const bool shared_single = w.has_shared && !shared_tc && T == 1 && !q4;
    const bool shared_multi = w.has_shared && !shared_tc && (T > 1 || q4);
    // (with a threshold of 1 every routed group is on the tensor cores: no one-token groups)
    const bool decode_kernels = !sg && !q4 && (gemm_min != 1 || shared_single);
    if (sg || q4 || decode_kernels || multi_gemv || shared_multi) {
        if (!rc) rc = clk.stage(DS4MOE_STAGE_UP_GEMV);
        if (!sg && !q4 && !decode_kernels) h->launches--;  // the stage's kernel is the GEMV below
    }
    if (sg) {
        if (!rc) rc = launch_prep_x(ws, x, T, w.D, stream);
        if (!rc) rc = launch_small_up(w, ws, T, k, stream);
        h->launches++;
        if (shared_single) {  // T = 1: the decode kernels take the shared expert alone (no single list)
            if (!rc) rc = launch_decode_up(w, ws, x, T, k, true, stream);
            h->launches++;
        }
    } else if (decode_kernels) {
        if (!rc) rc = launch_decode_up(w, ws, x, T, k, shared_single, stream);
    } else if (q4) {  // the 4-bit variant: the tokens as int16 dp2a pairs for its GEMV
        if (!rc) rc = launch_prep_x(ws, x, T, w.D, stream);
    }
    if (multi_gemv || shared_multi) {
        if (!rc) rc = launch_gemv_up(w, ws, x, T, k, shared_multi, stream);
        h->launches++;
    }
    if (shared_up_small) {
        if (!rc) rc = clk.stage(DS4MOE_STAGE_UP_GEMM);
        if (!rc) rc = launch_shared_up_small(w, ws, x, T, k, stream);
    }
    if (up_tc) {
        if (!rc && !shared_up_small) rc = clk.stage(DS4MOE_STAGE_UP_GEMM);
        else h->launches++;
        if (!rc) rc = launch_gemm_up(w, ws, h->tmap_x16, T, k, shared_tc && !shared_up_small, h->gemm_pairs != 0, stream);
    }
    if (sg || q4 || decode_kernels || multi_gemv || shared_multi) {
        if (!rc) rc = clk.stage(DS4MOE_STAGE_DOWN_GEMV);
        if (!sg && !q4 && !decode_kernels) h->launches--;  // the stage's kernel is the GEMV below
    }
    if (sg) {
        if (!rc) rc = launch_small_down(w, ws, T, k, stream);
        if (shared_single) {
            if (!rc) rc = launch_decode_down(w, ws, T, k, true, stream);
            h->launches++;
        }
    } else if (decode_kernels) {
        if (!rc) rc = launch_decode_down(w, ws, T, k, shared_single, stream);
    } else if (!q4) {
    } else if (T <= 64) {  // the 4-bit variant: each pair's h as int16 for its down GEMV
        if (!rc) rc = launch_prep_h(ws, T * k, w.F, stream);
    } else {
        h->launches--;  // the stage's kernel is the GEMV below, counted there
    }
    if (multi_gemv || shared_multi) {
        if (!rc) rc = launch_gemv_down(w, ws, T, k, shared_multi, stream, q4 && T <= 64);
        h->launches++;
    }
    if (any_tc) {
        if (!rc) rc = clk.stage(DS4MOE_STAGE_DOWN_GEMM);
        if (!rc) rc = launch_gemm_down(w, ws, h->tmap_h16, T, k, shared_tc, h->gemm_pairs != 0, stream);
        // Groups (and the shared expert) whose token, h or y values overflowed fp16 on the tensor
        // cores are flagged by those kernels; they are recomputed here in fp32 on the GEMV kernels
        // (which find nothing to do when no flag is set), and the combine reads their fp32 rows.
        Workspace wr = ws;
        wr.gemv_list = ws.repair_list;
        wr.meta = ws.meta2;
        const int32_t *shared_flag = ws.ovf + w.E;
        if (!rc) rc = clk.stage(DS4MOE_STAGE_REPAIR);
        if (!rc) rc = launch_repair_list(w, ws, gemm_min, stream);
        if (!rc) rc = launch_gemv_up(w, wr, x, T, k, shared_tc, stream, shared_flag);
        if (!rc) rc = launch_gemv_down(w, wr, T, k, shared_tc, stream, false, shared_flag);
        h->launches += 2;
    }
    if (!rc) rc = clk.stage(DS4MOE_STAGE_COMBINE);
    if (!rc) rc = launch_combine(w, ws, T, k, gemm_min, shared_tc, out, stream);
    if (!rc) rc = clk.finish();
    h->calls++;
    return cuda_status(rc);
}

int ds4moe_get_stats(ds4moe_weights *h, ds4moe_stats *out) {
    if (!h || !out) return DS4MOE_EINVAL;
    std::memset(out, 0, sizeof *out);
    out->calls = h->calls;
    out->launches = h->launches;
    if (!h->events_recorded) return DS4MOE_OK;
    if (cudaEventSynchronize(static_cast<cudaEvent_t>(h->events[DS4MOE_N_STAGES])) != cudaSuccess) {
        cudaGetLastError();
        return DS4MOE_ECUDA;
    }
    for (int n = 0; n < h->n_stage_order; n++) {
        const int i = h->stage_order[n];
        if (!h->stage_ran[i]) continue;  // a stage taken back (the fused kernel's refused launch)
        // the next stage recorded in this call ends this one, the call's end event the last
        int j = DS4MOE_N_STAGES;
        for (int m = n + 1; m < h->n_stage_order; m++)
            if (h->stage_ran[h->stage_order[m]]) {
                j = h->stage_order[m];
                break;
            }
        float ms = 0.0f;
        if (cudaEventElapsedTime(&ms, static_cast<cudaEvent_t>(h->events[i]),
                                 static_cast<cudaEvent_t>(h->events[j])) != cudaSuccess) {
            cudaGetLastError();
            return DS4MOE_ECUDA;
        }
        out->stage_ms[i] = ms;
    }
    return DS4MOE_OK;
}

int ds4moe_step_trace(ds4moe_weights *h, uint64_t *out, int max_values, int *n_values) {
    if (!h || !out || !n_values || max_values < 0) return DS4MOE_EINVAL;
    const int n = std::min(max_values, decode_step_ctas() * 6);
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpy(out, h->ws.trace, static_cast<size_t>(n) * 8, cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return DS4MOE_ECUDA;
    }
    *n_values = n;
    return DS4MOE_OK;
}

int ds4moe_last_status(ds4moe_weights *h, ds4moe_stream_t stream) {
    if (!h) return DS4MOE_EINVAL;
    if (cudaStreamSynchronize(stream) != cudaSuccess) {
        cudaGetLastError();
        return DS4MOE_ECUDA;
    }
    int st = 0;
    if (cudaMemcpy(&st, h->ws.status, sizeof st, cudaMemcpyDeviceToHost) != cudaSuccess) return DS4MOE_ECUDA;
    if (cudaMemset(h->ws.status, 0, sizeof st) != cudaSuccess) return DS4MOE_ECUDA;
    if (st & ST_RANGE) return DS4MOE_ERANGE;
    if (st & ST_TIMEOUT) return DS4MOE_ETIMEOUT;
    if (st & ST_BADIDX) return DS4MOE_EINVAL;
    if (st & ST_CAPACITY) return DS4MOE_ECAPACITY;
    return DS4MOE_OK;
}

}  // extern "C"
