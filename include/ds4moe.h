/*
 * ds4moe.h -- C ABI of the routed-MoE expert FFN over 2-bit block-quantised experts,
 * for one NVIDIA GB300 GPU (sm_103a).
 *
 * What it computes. One routed mixture-of-experts layer's expert FFN, the hot path of a
 * DeepSeek-V4-style engine: per token, top-k routing over router logits, grouping of the
 * (token, slot) pairs by expert, a SwiGLU expert per pair (h = silu(W_gate x) * (W_up x),
 * y = W_down h), an always-on bf16 shared expert, and the gate-weighted sum added into the
 * residual. Sources: "DwarfStar" (ds4 README), section "模型权重" (only routed experts are
 * quantised: up/gate to IQ2_XXS, down to Q2_K; shared expert, projections and router stay
 * unquantised); "DwarfStar 深度解析" §2.1 (per-token dynamic expert choice, irregular
 * compute) and §3.4.3 (the quantisation split, the router kept at full precision);
 * "Part 5: 服务层" §6 "会话批处理" (several sessions' decode steps in one batched kernel).
 * The block layouts are this library's own IQ2-style, Q2_K-style and Q4_K-style formats
 * (the pages name the formats but print no layout; the library's format notes fix them).
 * Where a declaration below says "library reading", the pages are silent on that point.
 *
 * Conventions.
 *   - Every function returns a status (DS4MOE_OK = 0) and never throws or aborts.
 *   - Host functions are synchronous and thread-safe.
 *   - Device functions are asynchronous on the given stream; their pointers are device
 *     memory owned by the caller, and all argument checks happen on the host before any
 *     launch. Errors a kernel detects are recorded in a device status word of the weights
 *     handle and returned by ds4moe_last_status().
 *   - A weights handle owns its workspace, so calls that use one handle must not overlap
 *     (issue them on one stream, or order them with events).
 *   - bf16 and fp16 values are passed as their 16-bit patterns (uint16_t).
 */
#ifndef DS4MOE_H
#define DS4MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *ds4moe_stream_t;

enum ds4moe_status {
    DS4MOE_OK = 0,
    DS4MOE_EINVAL = 1,       /* bad argument (null pointer, size, alignment, k > E, ...) */
    DS4MOE_ENOMEM = 2,       /* device or host allocation failed */
    DS4MOE_ECUDA = 3,        /* a CUDA runtime call failed (no device, launch error, ...) */
    DS4MOE_EBADDATA = 4,     /* input data rejected (non-finite weights, bad packed scale) */
    DS4MOE_ETIMEOUT = 5,     /* a bounded device-side wait gave up */
    DS4MOE_EUNSUPPORTED = 6, /* shape or device not supported by the library */
    DS4MOE_ERANGE = 7,       /* not returned by this version: tensor-core groups whose fp16 values
                                overflow are recomputed in fp32 within the call */
    DS4MOE_ECAPACITY = 8     /* a call touched more experts than a pooled handle's slots */
};

/* Gate weights over the k selected logits l_0 >= ... >= l_{k-1} (a NaN logit counts as -inf).
 * Library reading of "DwarfStar 深度解析" §2.1 (the pages name no gate function): a term whose
 * logit equals l_0 counts as exp(0) = 1 also when both are infinite (the limit of equal logits),
 * so an all -inf selection gets 1/k each and a +inf logit takes the weight of every finite one. */
enum ds4moe_gate_mode {
    DS4MOE_GATE_SOFTMAX = 0, /* g_s = exp(l_s - l_0) / sum_j exp(l_j - l_0) over the k selected */
    DS4MOE_GATE_SIGMOID = 1  /* g_s = sigmoid(l_s) / sum_j sigmoid(l_j) over the k selected,
                                evaluated as the softmax rule over log sigmoid(l_s) (same ratio) */
};

/* Matrices of one expert, for ds4moe_weights_dequantize(). */
enum ds4moe_matrix { DS4MOE_GATE = 0, DS4MOE_UP = 1, DS4MOE_DOWN = 2 };

/* Options of a weights handle, for ds4moe_set_option(). */
enum ds4moe_option {
    /* Expert groups with at least this many tokens run on the tcgen05 tensor-core path;
     * smaller groups run on the small-group kernels (DS4MOE_OPT_SMALL_GROUPS) or on the fused
     * dequant-GEMV kernels. 0 means never use tensor cores; 1 means always; -1 (the default)
     * chooses: with the small-group kernels, no tensor cores for calls of at most 64 tokens
     * and 7 above that; without them, 2. */
    DS4MOE_OPT_GEMM_MIN_TOKENS = 0,
    /* Same threshold for the bf16 shared expert (by token count T). Default 2. */
    DS4MOE_OPT_SHARED_GEMM_MIN_TOKENS = 1,
    /* 1: record CUDA events around each stage of ds4moe_expert_ffn on its stream, so that
     * ds4moe_get_stats() can report per-stage device times. Default 0. */
    DS4MOE_OPT_PROFILE = 2,
    /* 1: a call with T = 1 runs as one cooperative kernel (routing, both expert phases and
     * the combine; d_ff = 2048, k <= 8, d_model <= 8192); 0: as the separate kernels.
     * Default 1. */
    DS4MOE_OPT_SINGLE_STEP = 3,
    /* 1: the single-token kernel records per-CTA timestamps, read by ds4moe_step_trace(). */
    DS4MOE_OPT_TRACE = 4,
    /* 1: expert groups below the tensor-core threshold run on the small-group kernels, which
     * decode each 2-bit weight group once for all the tokens of its group (up to 6 at a time)
     * and take the down projection pair by pair; used when d_model <= 4096 and d_ff <= 2048
     * and the bf16 shared expert, if any, is on the tensor cores (or T = 1). 0: the fused
     * dequant-GEMV kernels. Default 1. */
    DS4MOE_OPT_SMALL_GROUPS = 5,
    /* Tests of the bounded device waits: value > 0 makes the single-token kernel's grid barrier
     * wait for an arrival that never comes, so the wait runs out (about 2 s), every CTA finishes
     * through its abort path, and ds4moe_last_status reports DS4MOE_ETIMEOUT; the handle stays
     * usable. Default 0. */
    DS4MOE_OPT_WAIT_TEST = 6,
    /* 1: the tensor-core kernels run on pairs of CTAs (clusters of two, one MMA over both CTAs'
     * shared memory: 256 weight rows per MMA, each CTA holding half of the token tile) where the
     * shape allows (d_ff a multiple of 256 for the first GEMM, d_model a multiple of 512 for the
     * down GEMM); 0: one CTA per tile. Library reading, no passage. */
    DS4MOE_OPT_GEMM_PAIRS = 7
};

/* Stages of ds4moe_expert_ffn, in launch order (indices into ds4moe_stats.stage_ms). */
enum ds4moe_stage {
    DS4MOE_STAGE_ROUTE = 0,     /* top-k routing */
    DS4MOE_STAGE_GROUP = 1,     /* grouping of pairs by expert */
    DS4MOE_STAGE_GATHER = 2,    /* fp16 token gather for the tensor-core path */
    DS4MOE_STAGE_UP_GEMV = 3,   /* dequant-GEMV gate/up + SwiGLU */
    DS4MOE_STAGE_UP_GEMM = 4,   /* tensor-core gate/up + SwiGLU */
    DS4MOE_STAGE_DOWN_GEMV = 5, /* dequant-GEMV down */
    DS4MOE_STAGE_DOWN_GEMM = 6, /* tensor-core down */
    DS4MOE_STAGE_COMBINE = 7,   /* gate-weighted combine into the residual */
    DS4MOE_STAGE_STEP = 8,      /* the single-token kernel: the whole call */
    DS4MOE_STAGE_POOL = 9,      /* pooled handles: slot assignment and the copies of missing experts */
    DS4MOE_STAGE_REPAIR = 10,   /* tensor-core groups whose fp16 values overflowed, recomputed in fp32 */
    DS4MOE_N_STAGES = 11
};

typedef struct {
    uint64_t calls;     /* ds4moe_expert_ffn calls since creation */
    uint64_t launches;  /* kernels launched by those calls */
    float stage_ms[DS4MOE_N_STAGES]; /* device time per stage of the last profiled call, 0 if
                                        the stage did not run or profiling is off */
} ds4moe_stats;

/* Human-readable text of a status code (static storage). Library reading, no passage. */
const char *ds4moe_strerror(int status);

/* ------------------------------------------------------------------ host: formats */

/* Bytes of a packed [rows x cols] matrix: rows * cols/256 * 84 (Q2_K-style) or * 66
 * (IQ2-style). 0 if rows < 0, cols <= 0 or cols % 256 != 0. The block sizes follow the formats
 * the pages name ("DwarfStar" README, "模型权重": Q2_K and IQ2_XXS, 256-weight super-blocks);
 * the exact byte counts are the library's layouts (library reading). */
size_t ds4moe_q2k_bytes(int64_t rows, int64_t cols);
size_t ds4moe_iq2_bytes(int64_t rows, int64_t cols);
/* The 4-bit variant's Q4_K-style blocks ("DwarfStar" README, "模型权重": the q4 build; the
 * 144-byte layout is the library's reading): rows * cols/256 * 144 bytes. */
size_t ds4moe_q4k_bytes(int64_t rows, int64_t cols);

/* The IQ2-style grid: 256 entries x 8 magnitudes in {1, 3, 5, 7}, entry-major, into out[2048]
 * (entry 0 all ones, the rest drawn by splitmix64 from the library's fixed seed; library reading
 * of the codebook format the pages name in "DwarfStar" README, "模型权重"). */
int ds4moe_iq2_grid(uint8_t *out);

/* Quantise a row-major fp32 matrix w [rows x cols] (cols % 256 == 0) into dst (dst_bytes
 * at least the size above) with the library's quantisers (plain min/max affine for the Q2_K-style
 * blocks; an exhaustive scale and grid search for the IQ2-style blocks; fp64 decisions, ties to
 * the lowest index); the output is byte-identical to any implementation that follows them. Runs
 * on all host cores. EINVAL: bad sizes or null pointers; EBADDATA: a non-finite weight or an fp16
 * scale overflow (dst is then unspecified). Source: "DwarfStar" README, "模型权重" (up/gate in
 * IQ2_XXS, down in Q2_K); the quantisers themselves are the library's reading. */
int ds4moe_quantize_q2k(const float *w, int64_t rows, int64_t cols, void *dst, size_t dst_bytes);
int ds4moe_quantize_iq2(const float *w, int64_t rows, int64_t cols, void *dst, size_t dst_bytes);
/* The 4-bit variant ("DwarfStar" README, "模型权重": the q4 build keeps every routed-expert
 * projection in 4 bits; the Q4_K-style block layout and its min/max quantiser are the library's
 * reading). */
int ds4moe_quantize_q4k(const float *w, int64_t rows, int64_t cols, void *dst, size_t dst_bytes);

/* Host dequantisation to fp32 (each weight's exact value in the library's formats), for tests
 * and tools. Library reading of the formats named in "DwarfStar" README, "模型权重". */
int ds4moe_dequantize_q2k(const void *src, int64_t rows, int64_t cols, float *dst);
int ds4moe_dequantize_iq2(const void *src, int64_t rows, int64_t cols, float *dst);
int ds4moe_dequantize_q4k(const void *src, int64_t rows, int64_t cols, float *dst);

/* ------------------------------------------------------------------ weights handle */

typedef struct ds4moe_weights ds4moe_weights;

typedef struct {
    int d_model;   /* D, a multiple of 256 */
    int d_ff;      /* F, a multiple of 256 */
    int n_experts; /* E, 1..1024 */
    /* Host pointers, one per expert: gate and up are IQ2-style [d_ff x d_model] blobs of
     * ds4moe_iq2_bytes(d_ff, d_model) bytes; down is a Q2_K-style [d_model x d_ff] blob of
     * ds4moe_q2k_bytes(d_model, d_ff) bytes. Copied; the caller keeps ownership. */
    const void *const *gate_iq2;
    const void *const *up_iq2;
    const void *const *down_q2k;
    /* Host bf16 shared expert, or all three NULL for none: gate/up [d_ff x d_model],
     * down [d_model x d_ff], row-major. Copied. */
    const uint16_t *shared_gate_bf16;
    const uint16_t *shared_up_bf16;
    const uint16_t *shared_down_bf16;
    int max_tokens; /* largest T of any later call, >= 1 */
    int max_k;      /* largest k of any later call, 1..min(32, n_experts) */
} ds4moe_weights_desc;

/* Create a handle on the current CUDA device: validates the blobs (finite fp16 scales, before
 * any device call), repacks them into the device layout, uploads them and allocates the
 * workspace for max_tokens x max_k pairs. Synchronous. EBADDATA names a non-finite fp16 scale;
 * ENOMEM a failed device allocation (nothing is kept). Source: "DwarfStar" README, "模型权重" (the
 * routed experts are held quantised, the shared expert unquantised); holding them resident in
 * device memory, the layout and the workspace are the library's reading. */
int ds4moe_weights_create(const ds4moe_weights_desc *desc, ds4moe_weights **out);

/* A handle of the 4-bit variant: the three per-expert pointers of desc hold Q4_K-style blobs
 * (gate and up [d_ff x d_model], down [d_model x d_ff], ds4moe_q4k_bytes each). Its routed
 * groups run on the dequant-GEMV kernels, and in calls of more than 64 tokens those of 2 or
 * more tokens on the tensor-core kernels (not on the fused single-token or the small-group
 * kernels); the bf16 shared expert keeps its usual kernels.
 * ds4moe_weights_dequantize gives their fp32 values (dst_f16 is EUNSUPPORTED);
 * ds4moe_expert_ffn_static is EUNSUPPORTED for them. Otherwise as ds4moe_weights_create.
 * Source: "DwarfStar" README, "模型权重" (the q4 build, and the q2-q4 mix). */
int ds4moe_weights_create_q4(const ds4moe_weights_desc *desc, ds4moe_weights **out);

/* A handle whose routed experts stream from host memory into a pool of n_slots expert slots
 * in device memory ("DwarfStar" README, "运行大于 RAM 的模型": a model larger than memory
 * keeps its routed experts outside and loads the ones each token routes to). The packed
 * experts are kept in pinned, device-mapped host memory in the device layout, which the GPU
 * reads directly (over NVLink-C2C on Grace systems). Each call, after routing and in stream
 * order (no host synchronisation):
 *   - every expert the call touches gets a slot: a resident expert keeps its slot (a hit);
 *     each missing expert, in increasing expert order, takes the slot not used by this call
 *     that was used least recently (empty slots first, then the oldest last use, ties to the
 *     lower slot), evicting its expert, and is copied in (a miss);
 *   - the experts then run on the same kernels as a resident handle's, over slot indices
 *     (a call of one token on the fused single-token kernel, through its expert-to-slot
 *     map), with results identical bit for bit to a resident handle's.
 * A call that touches more than n_slots experts records DS4MOE_ECAPACITY in the status word
 * (ds4moe_last_status), changes no slot and leaves out unspecified.
 * max_k <= n_slots <= n_experts. Other arguments and errors as ds4moe_weights_create. */
int ds4moe_weights_create_pooled(const ds4moe_weights_desc *desc, int n_slots, ds4moe_weights **out);

/* Pool state of a pooled handle (synchronises the device): its slot count, the hits and
 * misses since creation, and (slot_expert: n_slots ints, may be NULL) the expert held by each
 * slot or -1. Any output pointer may be NULL. EINVAL for a handle that is not pooled.
 * Library reading, no passage (a diagnostic of the streamed-expert pool above). */
int ds4moe_pool_info(ds4moe_weights *w, int *n_slots, uint64_t *hits, uint64_t *misses, int32_t *slot_expert);

/* Test hook for failure handling: the n-th device allocation that any handle creation makes from
 * now on fails as if the device were out of memory (the creation then returns DS4MOE_ENOMEM and
 * frees what it had allocated); n = 0 turns the hook off. Process-wide. EINVAL for n < 0.
 * Library reading, no passage. */
int ds4moe_test_fail_allocation(int n);

/* Free a handle (NULL is allowed). Synchronises the device first. Library reading, no passage. */
void ds4moe_weights_destroy(ds4moe_weights *w);

/* Set one of the options above on a handle. EINVAL for an unknown option or a negative value
 * (except -1 for DS4MOE_OPT_GEMM_MIN_TOKENS). Library reading, no passage. */
int ds4moe_set_option(ds4moe_weights *w, int option, int value);

/* Dequantise one resident expert matrix on the device, through the device decode the
 * kernels use: fp32 values (the GEMV path's weights) into dst_f32 (rows*cols floats, may be
 * NULL), and into dst_f16 (may be NULL) the fp16 operand bytes exactly as the tensor-core
 * producers write them, which are RN-even of the fp32 values. Asynchronous. EINVAL for a bad
 * expert or matrix or two NULL outputs; EUNSUPPORTED for a pooled handle. A test entry point:
 * library reading, no passage (the formats it decodes: "DwarfStar" README, "模型权重"). */
int ds4moe_weights_dequantize(const ds4moe_weights *w, int expert, int matrix, float *dst_f32,
                              uint16_t *dst_f16, ds4moe_stream_t stream);

/* ------------------------------------------------------------------ device: the hot path */

/* Router logits, the step in front of routing: logits[t][e] = sum_d x[t][d] * w_router[e][d]
 * + bias[e]. x bf16 [T x D] and w_router bf16 [E x D] row-major, 16-byte aligned; bias fp32 [E]
 * or NULL; logits fp32 [T x E]. D a multiple of 256 (<= 8192), E a multiple of 8 (<= 1024),
 * T >= 0 (T = 0 is a no-op). Device pointers, asynchronous on the stream.
 * The fp32 order is fixed for a given (T, D, E), so the top-k after it is reproducible run to
 * run. T < 64, or E not a multiple of 128 (CUDA cores): the columns are cut into segments of 1024
 * (the last one shorter when D is not a multiple); per (t, e) and segment, 32 partial sums p_l,
 * each adding in increasing d the products of the segment's columns d with (d / 8) % 32 == l (each
 * bf16 x bf16 product is exact in fp32; one FMA per product), then p_l += p_(l xor o) for
 * o = 16, 8, 4, 2, 1; the segment sums are added in increasing segment order, then bias[e]; every
 * addition rounds to nearest even. T >= 64 and E a multiple of 128 (tensor cores): the products of
 * 16 consecutive columns are added to an fp32 accumulator in increasing column blocks (the order
 * within a block is the hardware's), then bias[e]. A bounded wait that gives up (no completion of
 * a copy or an MMA within about 2 s) leaves that CTA's logits unwritten and is reported by
 * ds4moe_router_last_status().
 * Source: "DwarfStar" README, "模型权重", and "DwarfStar 深度解析" §3.4.3 (the router stays
 * unquantised; bf16 weights and an fp32 bias are this library's reading). */
int ds4moe_router_logits(const void *x, const void *w_router, const float *bias, int T, int D, int E,
                         float *logits, ds4moe_stream_t stream);

/* Synchronises the stream and reports whether a tensor-core router call since the last query had
 * a bounded wait give up: DS4MOE_ETIMEOUT (then clears it), DS4MOE_OK, or DS4MOE_ECUDA. The state
 * is per process (the router takes no handle). */
int ds4moe_router_last_status(ds4moe_stream_t stream);

/* Top-k routing: per token t, the k experts with the largest logits (ties to the lower
 * expert index; NaN orders as -inf), in that order, and their gate weights (mode above).
 * logits fp32 [T x E] row-major; topk_idx int32 [T x k]; topk_w fp32 [T x k].
 * 1 <= k <= min(E, 32), E <= 1024, T >= 0 (T = 0 is a no-op).
 * Source: "DwarfStar 深度解析" §2.1 (per-token dynamic expert choice) and §3.4.3
 * (router at full precision); tie rule and gate modes are this library's reading. */
int ds4moe_route(const float *logits, int T, int E, int k, int gate_mode, int32_t *topk_idx,
                 float *topk_w, ds4moe_stream_t stream);

/* Group the T*k (token, slot) pairs by expert: a stable counting sort in (token, slot)
 * order. counts int32 [E]; offsets int32 [E+1] (exclusive scan, offsets[E] = T*k);
 * perm int32 [T*k] (pair id t*k+s at each grouped position); inv int32 [T*k] (grouped
 * position of pair t*k+s). Deterministic. An index outside [0, E) is grouped as expert 0 (inside
 * ds4moe_expert_ffn it is also recorded, and ds4moe_last_status reports EINVAL). Device pointers,
 * asynchronous; EINVAL for bad sizes or null pointers. Source: "Part 5: 服务层" §6 "会话批处理"
 * (read-only weight work done once for the whole batch: each expert's tokens gathered so its
 * weights stream once) and "DwarfStar 深度解析" §2.1 (per-token expert choice makes MoE compute
 * irregular); the stable order is the library's reading. */
int ds4moe_group(const int32_t *topk_idx, int T, int k, int E, int32_t *counts, int32_t *offsets,
                 int32_t *perm, int32_t *inv, ds4moe_stream_t stream);

/* The expert FFN: out[t] += y_shared[t] + sum_s g[t,s] * y_{idx[t,s]}(x[t]), for t < T.
 *   x         bf16 [T x d_model], 16-byte aligned;
 *   logits    fp32 [T x n_experts] (router logits, bias already added);
 *   gate_mode DS4MOE_GATE_SOFTMAX or DS4MOE_GATE_SIGMOID (above);
 *   out       fp32 [T x d_model] residual, updated in place, 16-byte aligned.
 * Routing, grouping, the SwiGLU experts and the combine all run on the device with no
 * host synchronisation; results are bit-reproducible run to run. T <= max_tokens and
 * k <= max_k of the handle. EINVAL on bad arguments; device-side errors are reported by
 * ds4moe_last_status(). A group on the tensor-core path (and the shared expert there) whose token,
 * h or y values overflow fp16 is recomputed in fp32 on the GEMV kernels within the same call. Source: "DwarfStar" README, "模型权重" (routed up/gate in IQ2_XXS, down
 * in Q2_K, the shared expert unquantised) and "DwarfStar 深度解析" §2.1 and §3.4.3 (the routed
 * MoE layer and its expert tree). Library readings: T added to the signature, gate_mode (the
 * pages name no gate function), SwiGLU as the activation, the shared expert at weight 1, and out
 * an fp32 residual updated in place. */
int ds4moe_expert_ffn(const uint16_t *x, ds4moe_weights *w, const float *logits, int T, int k,
                      int gate_mode, float *out, ds4moe_stream_t stream);

/* Counters of the handle, and (when DS4MOE_OPT_PROFILE is on) the per-stage device times of
 * the last call, read from its CUDA events (waits for them). Library reading, no passage. */
int ds4moe_get_stats(ds4moe_weights *w, ds4moe_stats *out);

/* Diagnostics of the single-token kernel (with DS4MOE_OPT_TRACE on; library reading, no
 * passage): synchronises the device
 * and copies up to max_values timestamps of the last call into out: per CTA six globaltimer
 * values in ns -- start, prologue done, gate/up phase done, grid barrier passed, h staged,
 * down phase done. *n_values receives the number copied (6 per CTA). */
int ds4moe_step_trace(ds4moe_weights *w, uint64_t *out, int max_values, int *n_values);

/* Synchronise the stream, then return and clear the handle's device status word
 * (DS4MOE_OK when no kernel reported an error since the last call). Library reading, no
 * passage (how device-side errors reach the host). */
int ds4moe_last_status(ds4moe_weights *w, ds4moe_stream_t stream);

/* The expert FFN without any device allocation, for callers that cannot allocate device
 * memory while they run: for example a plug-in whose host framework owns and budgets every
 * device allocation, or a serving loop that must not call cudaMalloc (it can synchronise the
 * device and can fail under memory pressure). Such a caller creates the weights handle once
 * at load time -- it may ask for the smallest workspace, max_tokens = 1 and max_k = 1 -- and
 * runs its decode batches through this entry point. The pages have no counterpart: this is
 * a deployment variant of ds4moe_expert_ffn, not a step of the method.
 *
 * Same arguments and result as ds4moe_expert_ffn (out += the expert FFN of x), computed with
 * every expert group on the dequant-GEMV path. The per-call intermediates (top-k arrays,
 * grouping, h and y) live in one static 3 MiB region of device memory that every GPU which
 * loads the library holds until the process exits; the handle's own workspace is not used,
 * so T and k are not limited by the handle's max_tokens and max_k, only by the region:
 * calls needing more than 3 MiB (about T*(k+1)*(d_model + d_ff)*4 bytes, e.g. more than 9
 * tokens at top-8 with d_model 7168 and d_ff 2048) return DS4MOE_EINVAL without launching.
 * The current device must be the handle's. The first call on a device looks up the region's
 * device address (cudaGetSymbolAddress) and keeps it for the life of the process; make that
 * first call before any stream capture. The kept address does not survive a reset of the device
 * (cudaDeviceReset): after one, this entry point must not be called again in that process.
 * All calls share the region: calls that overlap on the GPU (other streams, other threads,
 * other handles) race and must be ordered by the caller. Device-side errors are reported
 * through the handle, by ds4moe_last_status(). Nothing here calls cudaMalloc or cudaFree. */
int ds4moe_expert_ffn_static(const uint16_t *x, const ds4moe_weights *w, const float *logits, int T, int k,
                             int gate_mode, float *out, ds4moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DS4MOE_H */
