// Internal declarations shared by the library's translation units (not part of the ABI).
#pragma once

#include <cstddef>
#include <cstdint>

#include "../../include/ds4moe.h"

namespace ds4moe {

constexpr int kGemmBN = 256;  // token rows per tensor-core tile
constexpr int kTokenBoxes = 5; // TMA box heights 16, 32, 64, 128, 256 rows

void host_grid(uint8_t out[2048]);
bool host_f16_finite(uint16_t h);
double host_f16_value(uint16_t h);

// Device status bits, OR-ed by kernels into the handle's status word.
enum : int {
    ST_RANGE = 1,    // a value overflowed fp16 on the tensor-core path
    ST_TIMEOUT = 2,  // a bounded wait gave up
    ST_BADIDX = 4,   // an expert index outside [0, E) reached the grouping kernel
    ST_CAPACITY = 8, // a call touched more experts than a pooled handle's slots
};

// Resident, repacked expert weights. Each IQ2-style row keeps its 64-byte block payloads
// (8 sub-blocks x 8 bytes) contiguous, 16-byte aligned, and the fp16 block scales in a
// separate plane; each Q2_K-style row keeps 80-byte payloads (16 B scales + 64 B codes)
// and a plane of (d, dmin) fp16 pairs. Row-major within an expert, experts back to back.
struct DeviceWeights {
    int D, F, E;
    int nbD, nbF;           // blocks per row of gate/up (D/256) and of down (F/256)
    uint8_t *iq2;              // gate and up, tiled: see iq2_qs_row
    uint8_t *q2k;              // down, tiled: see q2k_sq_row
    uint16_t *sh_gate, *sh_up; // [F][D] bf16, or null
    uint16_t *sh_down;         // [D][F] bf16, or null
    uint16_t *sh_down_f16;     // [D][F] fp16 copy for the tensor-core path, or null
    uint8_t *tc_ok;            // [E] 1 if every dequantised weight of the expert fits fp16
    int fmt;                   // 0: IQ2-style gate/up + Q2_K-style down; 1: the 4-bit variant (q4)
    uint8_t *q4;               // fmt 1: Q4_K-style rows, see q4_row
    bool has_shared;
    bool shared_tc_ok;         // the shared expert's weights fit fp16
};

// Tiled device layout of the routed experts' packed weights: the rows that one single-token
// step streams together are one contiguous range, so each is fetched with one bulk copy.
//   gate/up: expert e, rows 16t .. 16t+15 form one tile of 16 * nbD * 132 bytes:
//            [gate qs: 16 x nbD x 64][up qs: 16 x nbD x 64][gate d: 16 x nbD fp16][up d: 16 x nbD fp16]
//   down:    expert e, rows 4t .. 4t+3 form one tile of 4 * nbF * 84 bytes:
//            [sq: 4 x nbF x 80 (scales, codes)][dd: 4 x nbF x u32 (d | dmin << 16)]
// Within a tile each row's blocks stay together, so kernels index a row pointer by block; the
// 16-byte chunks of a row's codes are permuted by iq2_swz (below).
#ifdef __CUDACC__
#define DS4MOE_HD __host__ __device__
#else
#define DS4MOE_HD
#endif

// The 4-bit variant: expert e holds its gate rows, then its up rows (F rows of nbD blocks each),
// then its down rows (D rows of nbF blocks), 144-byte Q4_K-style blocks in row order.
DS4MOE_HD inline size_t q4_expert_bytes(const DeviceWeights &w) {
    return (2 * static_cast<size_t>(w.F) * w.nbD + static_cast<size_t>(w.D) * w.nbF) * 144;
}
// Row r of gate (m = 0), up (m = 1) or down (m = 2) of expert e.
DS4MOE_HD inline size_t q4_row_offset(const DeviceWeights &w, int m, int e, int r) {
    const size_t base = static_cast<size_t>(e) * q4_expert_bytes(w);
    if (m < 2) return base + (static_cast<size_t>(m) * w.F + r) * w.nbD * 144;
    return base + 2 * static_cast<size_t>(w.F) * w.nbD * 144 + static_cast<size_t>(r) * w.nbF * 144;
}

constexpr int kIq2TileRows = 16;
constexpr int kQ2kTileRows = 4;

DS4MOE_HD inline size_t iq2_tile_bytes(int nbD) { return static_cast<size_t>(kIq2TileRows) * nbD * 132; }
DS4MOE_HD inline size_t q2k_tile_bytes(int nbF) { return static_cast<size_t>(kQ2kTileRows) * nbF * 84; }
DS4MOE_HD inline size_t iq2_tile_offset(const DeviceWeights &w, int e, int r) {
    return (static_cast<size_t>(e) * (w.F / kIq2TileRows) + r / kIq2TileRows) * iq2_tile_bytes(w.nbD);
}
DS4MOE_HD inline size_t q2k_tile_offset(const DeviceWeights &w, int e, int d) {
    return (static_cast<size_t>(e) * (w.D / kQ2kTileRows) + d / kQ2kTileRows) * q2k_tile_bytes(w.nbF);
}
// Row r of gate (m = 0) or up (m = 1) of expert e: nbD blocks of 64 code bytes, and their nbD scales d.
DS4MOE_HD inline size_t iq2_qs_offset(const DeviceWeights &w, int m, int e, int r) {
    return iq2_tile_offset(w, e, r) + static_cast<size_t>(m * kIq2TileRows + r % kIq2TileRows) * w.nbD * 64;
}
DS4MOE_HD inline size_t iq2_d_offset(const DeviceWeights &w, int m, int e, int r) {
    return iq2_tile_offset(w, e, r) + static_cast<size_t>(2 * kIq2TileRows) * w.nbD * 64 +
           static_cast<size_t>(m * kIq2TileRows + r % kIq2TileRows) * w.nbD * 2;
}
// Row d of down of expert e: nbF blocks of 80 bytes (scales, codes), and their nbF d | dmin words.
DS4MOE_HD inline size_t q2k_sq_offset(const DeviceWeights &w, int e, int d) {
    return q2k_tile_offset(w, e, d) + static_cast<size_t>(d % kQ2kTileRows) * w.nbF * 80;
}
DS4MOE_HD inline size_t q2k_dd_offset(const DeviceWeights &w, int e, int d) {
    return q2k_tile_offset(w, e, d) + static_cast<size_t>(kQ2kTileRows) * w.nbF * 80 +
           static_cast<size_t>(d % kQ2kTileRows) * w.nbF * 4;
}
// Within a row, the 16-byte chunks of codes (two 32-weight sub-blocks each) are stored permuted:
// chunk q at position q ^ iq2_swz(w, r). The rows of a tile are 64 * nbD bytes apart (a multiple of
// 128 when nbD is even), so without it the 16 rows of a tile read at one chunk index would all hit
// the same shared-memory banks; with it, eight consecutive rows cover all eight 16-byte bank groups,
// and a row read chunk by chunk still covers each aligned group of eight chunks once.
DS4MOE_HD inline int iq2_swz(const DeviceWeights &w, int r) { return r & ((w.nbD & 1) ? 3 : 7); }
DS4MOE_HD inline const uint8_t *q4_row(const DeviceWeights &w, int m, int e, int r) { return w.q4 + q4_row_offset(w, m, e, r); }
DS4MOE_HD inline const uint8_t *iq2_qs_row(const DeviceWeights &w, int m, int e, int r) {
    return w.iq2 + iq2_qs_offset(w, m, e, r);
}
DS4MOE_HD inline const uint16_t *iq2_d_row(const DeviceWeights &w, int m, int e, int r) {
    return reinterpret_cast<const uint16_t *>(w.iq2 + iq2_d_offset(w, m, e, r));
}
DS4MOE_HD inline const uint8_t *q2k_sq_row(const DeviceWeights &w, int e, int d) {
    return w.q2k + q2k_sq_offset(w, e, d);
}
DS4MOE_HD inline const uint32_t *q2k_dd_row(const DeviceWeights &w, int e, int d) {
    return reinterpret_cast<const uint32_t *>(w.q2k + q2k_dd_offset(w, e, d));
}

// Per-call grouping metadata written on the device by the grouping kernel.
struct GroupMeta {
    int n_gemv;    // experts with 0 < n_e < gemm_min (n_e > 1 when singles are split off), in gemv_list
    int n_gemm;    // experts with n_e >= gemm_min, listed in gemm_list in expert order
    int n_single;  // experts with exactly one token (when split off), listed in single_list
    int n_small_pairs;  // pairs of the gemv_list experts (positions listed in small_pos when requested)
    int n_tiles;   // tensor-core token tiles of the gemm_list experts (ceil(n_e / kGemmBN) each)
    int n_full;    // of which full (kGemmBN tokens): tile_desc holds them first, then the ragged ones,
                   // largest first
};

// Streamed experts (pooled handles): the host store and the slot state. The store holds every
// expert in the device layout (gate/up tiles, then down tiles); the device pool (DeviceWeights
// with E = S) holds S of them.
struct SlotPool {
    int S;                       // slots, 0 for a resident handle
    int E;                       // experts in the store
    size_t up_bytes, down_bytes; // one expert's gate/up and down ranges
    const uint8_t *host_iq2;     // [E][up_bytes]   device-mapped pinned host memory
    const uint8_t *host_q2k;     // [E][down_bytes]
    const uint8_t *host_tc_ok;   // [E]
    int32_t *slot_of;            // [E] slot of each expert, -1 if not resident
    int32_t *expert_of;          // [S] expert of each slot, -1 if empty
    uint32_t *stamp;             // [S] number of the last call that used the slot, 0 if none
    unsigned long long *ctr;     // [4] calls, hits, misses, misses of the last call
    int32_t *miss;               // [S][2] the last call's misses: expert, slot
};

struct Workspace {
    int max_T, max_k;
    int32_t *topk_idx;  // [T*k]
    float *topk_w;      // [T*k]
    int32_t *counts;    // [E]
    int32_t *offsets;   // [E+1]
    int32_t *perm;      // [P]
    int32_t *inv;       // [P]
    int32_t *gemv_list; // [E]
    int32_t *gemm_list; // [E]
    int32_t *single_list; // [E]
    int32_t *tile_prefix; // [E+1] exclusive prefix of ceil(n_e / kGemmBN) over gemm_list
    int32_t *tile_desc;   // [E + P/kGemmBN][4] per tensor-core token tile: expert, first row, tokens, 0
                          // (full tiles first, then the ragged ones by decreasing size)
    GroupMeta *meta;
    uint8_t *grid;      // [256][8] IQ2-style grid
    uint8_t *grid_hi;   // [256][8] the grid's magnitudes as fp16 high bytes (1, 3, 5, 7 -> 3C, 42, 45, 47)
    float *h32;         // [P+T][F] fp32 intermediate of the GEMV path (rows P.. = shared expert)
    uint16_t *h16;      // [P+T][F] fp16 intermediate of the tensor-core path
    uint16_t *x16;      // [P+T][D] fp16 tokens gathered per group for the tensor-core path
    float *y;           // [P+T][D] per-pair expert outputs (rows P.. = shared expert); the tensor-core
                        // down GEMM writes its rows as D fp16 values in the first half of the row
    int *status;        // device status word
    unsigned *gbar;     // grid barrier of the single-token kernel: count, generation
    float *hmax;        // [1024][8] per-CTA maxima of the single-token kernel
    uint64_t *trace;    // [1024][6] timestamps of the single-token kernel
    int32_t *small_pos; // [P] positions of the small-group pairs (expert order)
    uint32_t *xq;       // [T][D/8][4] tokens as int16 pairs for the small-group kernels (dp2a order)
    int32_t *x8;        // [T][D/32] 8 x the sum of each 32-column sub-block of xq
    float *xsc;         // [T][4] dequantisation factor of xq (element 0; the rest pad to 16 bytes)
    uint32_t *hq4;      // 4-bit variant handles: [P][F/8][4] h as int16 dp2a pairs (prep_h)
    int *hsum4;         // [P][F/32] sum of each 32-column sub-block of hq4
    float *hsc4;        // [P] factor from hq4 back to h
    int32_t *ovf;       // [E+1] per call: the expert's (E: the shared expert's) tensor-core result
                        // overflowed fp16 and is recomputed in fp32 before the combine
    int32_t *repair_list; // [E] the experts to recompute
    GroupMeta *meta2;   // their count (n_gemv; the other fields 0)
};

}  // namespace ds4moe

struct ds4moe_weights {
    int device;
    ds4moe::DeviceWeights dw;
    ds4moe::Workspace ws;
    int gemm_min_tokens;
    int shared_gemm_min_tokens;
    int profile;
    int single_step;  // T = 1 calls use the fused single-token kernel when it supports the shape
    int trace;        // record the single-token kernel's per-CTA timestamps
    int small_groups; // groups below the tensor-core threshold run on the small-group kernels
    int wait_test;    // DS4MOE_OPT_WAIT_TEST
    int gemm_pairs;   // DS4MOE_OPT_GEMM_PAIRS
    void *events[DS4MOE_N_STAGES + 1];  // cudaEvent_t: start of each stage, end of the call
    bool stage_ran[DS4MOE_N_STAGES];
    bool events_recorded;
    uint64_t calls, launches;
    alignas(64) unsigned char tmap_x16[128 * ds4moe::kTokenBoxes];  // CUtensorMaps of x16 [rows][D]
    alignas(64) unsigned char tmap_h16[128 * ds4moe::kTokenBoxes];  // CUtensorMaps of h16 [rows][F]
    int stage_order[DS4MOE_N_STAGES];  // stages in the order the last call recorded them
    int n_stage_order;
    ds4moe::SlotPool pool;            // pool.S > 0: a pooled handle
    void *host_allocs[4];             // pinned host memory of the pool's store
    int n_host_allocs;
    void *allocs[64];
    int n_allocs;
};

namespace ds4moe {

// Launchers (return a cudaError_t as int; 0 = success).
int launch_router(const uint16_t *x, const uint16_t *w, const float *bias, int T, int D, int E, float *logits,
                  void *stream);
// The tensor-core router (router_tc.cu): calls of at least 64 tokens with E a multiple of 128.
bool router_tc_supported(int T, int D, int E);
int launch_router_tc(const uint16_t *x, const uint16_t *w, const float *bias, int T, int D, int E, float *logits,
                     void *stream);
// Reads and clears the tensor-core router's status bits (ST_TIMEOUT); 0 on success.
int router_read_status(int *st);
int launch_route(const float *logits, int T, int E, int k, int gate_mode, int32_t *idx, float *w,
                 void *stream);
int launch_pool_assign(const SlotPool &sp, int32_t *idx, int P, int *status, void *stream);
int launch_pool_fill(const SlotPool &sp, const DeviceWeights &w, int n_sms, void *stream);
// ovf (may be null): the call's overflow flags [E+1], cleared here
int launch_group(const int32_t *idx, int T, int k, int E, int gemm_min, const uint8_t *tc_ok,
                 int32_t *counts, int32_t *offsets, int32_t *perm, int32_t *inv, int32_t *gemv_list,
                 int32_t *gemm_list, int32_t *single_list, int32_t *tile_prefix, int32_t *tile_desc, int32_t *small_pos, GroupMeta *meta,
                 int *status, void *stream, int32_t *ovf = nullptr);
bool small_groups_supported(const DeviceWeights &w);
int launch_prep_x(const Workspace &ws, const uint16_t *x, int T, int D, void *stream);
int launch_small_up(const DeviceWeights &w, const Workspace &ws, int T, int k, void *stream);
int launch_small_down(const DeviceWeights &w, const Workspace &ws, int T, int k, void *stream);
int shared_small_max_tokens();
int launch_shared_up_small(const DeviceWeights &w, const Workspace &ws, const uint16_t *x, int T, int k,
                           void *stream);
int launch_gather(const DeviceWeights &w, const Workspace &ws, const uint16_t *x, int T, int k, int gemm_min,
                  bool shared, void *stream);
// pairs: run on clusters of two CTAs (cta_group::2) where the shape allows
int launch_gemm_up(const DeviceWeights &w, const Workspace &ws, const void *tmap_x16, int T, int k, bool shared,
                   bool pairs, void *stream);
int launch_gemm_down(const DeviceWeights &w, const Workspace &ws, const void *tmap_h16, int T, int k, bool shared,
                     bool pairs, void *stream);
int encode_token_map(void *map_out, void *base, int rows, int cols, int box_rows);
int encode_token_maps(void *maps_out, void *base, int rows, int cols);
int launch_producer_dump(const DeviceWeights &w, const uint8_t *grid, int expert, int matrix, uint16_t *dst16,
                         void *stream);
int launch_decode_up(const DeviceWeights &w, const Workspace &ws, const uint16_t *x, int T, int k, bool shared,
                     void *stream);
int launch_decode_down(const DeviceWeights &w, const Workspace &ws, int T, int k, bool shared, void *stream);
bool decode_step_supported(const DeviceWeights &w, int k);
// E_route: experts the logits route over; slot_of: null, or a pooled handle's expert -> slot map
int launch_decode_step(const DeviceWeights &w, const Workspace &ws, const uint16_t *x, const float *logits, int k,
                       int gate_mode, float *out, uint64_t *trace, int E_route, const int32_t *slot_of,
                       unsigned int bar_extra, void *stream);
int decode_step_ctas();
// shared_flag: non-null for a repair (launch_repair_list): the shared expert only when *shared_flag
int launch_gemv_up(const DeviceWeights &w, const Workspace &ws, const uint16_t *x, int T, int k,
                   bool shared_on_gemv, void *stream, const int32_t *shared_flag = nullptr);
// int16_h: the 4-bit variant's down rows on int16 h (launch_prep_h first)
int launch_gemv_down(const DeviceWeights &w, const Workspace &ws, int T, int k, bool shared_on_gemv, void *stream,
                     bool int16_h = false, const int32_t *shared_flag = nullptr);
// After the tensor-core GEMMs: the experts whose tensor-core results overflowed fp16 (ovf, set by
// the gather and the GEMM epilogues) into repair_list and meta2->n_gemv, for the GEMV kernels to
// recompute in fp32 (ovf[E] is the shared expert's flag).
int launch_repair_list(const DeviceWeights &w, const Workspace &ws, int gemm_min, void *stream);
int launch_prep_h(const Workspace &ws, int rows, int F, void *stream);
// gemm_min > 0: the pairs of groups of at least gemm_min tokens (tc_ok experts) ran on the
// tensor-core down GEMM and their y rows hold fp16; shared_f16: so does the shared expert's.
int launch_combine(const DeviceWeights &w, const Workspace &ws, int T, int k, int gemm_min, bool shared_f16,
                   float *out, void *stream);
int launch_dequant(const DeviceWeights &w, const uint8_t *grid, int expert, int matrix, float *dst32,
                   uint16_t *dst16, void *stream);

}  // namespace ds4moe
