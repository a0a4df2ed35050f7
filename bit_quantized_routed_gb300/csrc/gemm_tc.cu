// Tensor-core grouped GEMM for prefill-sized expert groups (tcgen05 + TMEM, sm_103a).
//
// "DwarfStar" README, "速度" and "基准测试": prefill runs in chunks of thousands of tokens
// and is compute-rich; with many tokens per expert the expert FFN is a dense contraction,
// so it runs on the 5th-generation tensor cores. Per (expert, 128 weight rows, up to 256
// tokens) tile -- for the down GEMM (expert, 256 weight rows, up to 256 tokens), so that each
// token tile copied in feeds two MMAs per K step in both GEMMs:
//   * sixteen producer warps stream the packed weight rows from HBM (each thread one half of
//     a row's columns per stage, with a ring of register prefetches and L2 prefetches ahead of
//     it), decode them to fp16 (RN-even of the exact fp32 value) and write them into shared
//     memory in the canonical K-major SWIZZLE_128B layout (128-row x 64-column atom columns);
//   * one warp issues TMA loads of the group's token rows (fp16, gathered per group) into
//     the same layout;
//   * one thread issues tcgen05.mma (M=128, N=tokens rounded up to 16, K=16) into fp32
//     accumulators in tensor memory: gate and up side by side for the first GEMM, the two
//     128-row halves side by side for the down GEMM;
//   * the producer warps then read the accumulators back with tcgen05.ld (four warps per
//     TMEM lane quarter) and apply the epilogue: h = silu(gate) * up (fp16 out) for the
//     first GEMM, y (fp16 out, into the first half of the row's fp32 slot) for the down GEMM.
// Swap-AB: weights are the M side and tokens the N side, so groups of a few dozen tokens
// still fill MMAs. Every wait on an mbarrier is bounded: after ~2 s it records
// DS4MOE_ETIMEOUT in the handle's status word and the CTA drains its copies, frees its
// tensor memory and exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "ptx.cuh"

namespace ds4moe {
namespace {

constexpr int BM = 128;   // weight rows per tile (MMA M)
constexpr int BN = kGemmBN;  // token rows per tile (MMA N at most)
constexpr int BK = 64;    // K elements per stage: one 128-byte swizzle atom
constexpr int kThreads = 576;  // warp 0 TMA, warp 1 MMA (+ TMEM alloc), warps 2..17 producers/epilogue
constexpr int kProducers = 512;
constexpr int kTableBytes = 256 * 16 * 8;  // replicated lookup table (grid or code selectors)

enum { UP = 0, DOWN = 1 };

// PAIR: the kernel runs on clusters of two CTAs (cta_group::2): each MMA covers 256 weight rows
// (128 in each CTA's shared memory) and each CTA holds half of the token tile, so per SM a stage
// carries half the token bytes and four stages fit where one CTA alone holds three.
template <int KIND, bool PAIR>
struct Cfg {
    static constexpr int NA = 2;  // first GEMM: gate and up; down GEMM: two 128-row weight tiles
    static constexpr int STAGES = PAIR ? 4 : 3;
    static constexpr int TMEM_COLS = 512;
    static constexpr int CTAS = PAIR ? 2 : 1;
    static constexpr int BROWS = PAIR ? kGemmBN / 2 : kGemmBN;  // token rows of a stage in one CTA
};

constexpr int A_BYTES = BM * BK * 2;  // 16 KB

// Shared-memory matrix descriptor (K-major, SWIZZLE_128B, 8-row atoms 1024 bytes apart) as two words:
// the low word holds the start address >> 4 (14 bits) and the leading-byte offset 1; the high word,
// the same for every operand, the 1024-byte stride, the descriptor version bit and the swizzle mode.
// A start address 16 * n bytes further is the low word + n (shared addresses stay below 2^18).
__device__ __forceinline__ uint32_t sw128_desc_lo(uint32_t saddr) { return ((saddr >> 4) & 0x3FFFu) | (1u << 16); }
constexpr uint32_t kSw128DescHi = (1024u >> 4) | (1u << (46 - 32)) | (2u << (61 - 32));

// Instruction descriptor of kind::f16: fp16 A and B (K-major), fp32 accumulate, M x N.
__device__ __forceinline__ uint32_t idesc_f16(int M, int N) {
    return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// Byte offset of 16-byte chunk c of row r in a 128-row, 128-byte-wide SWIZZLE_128B tile.
__device__ __forceinline__ uint32_t sw128_off(int r, int c) {
    return static_cast<uint32_t>((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// Bits 15 and 31 of the result: set for an fp16 half of hp that is +-inf or NaN (its magnitude
// bits at or above 0x7c00; adding 0x0400 to each 15-bit magnitude carries into bit 15 exactly then).
__device__ __forceinline__ uint32_t f16x2_overflow(uint32_t hp) { return ((hp & 0x7fff7fffu) + 0x04000400u) & 0x80008000u; }

__device__ __forceinline__ void st_shared16(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// ------------------------------------------------------------------ tiles

struct GemmParams {
    DeviceWeights w;
    const int4 *tile_desc;
    const GroupMeta *meta;
    const uint8_t *grid;
    uint16_t *h16;  // UP output, [rows][F]
    uint16_t *y16;  // DOWN output: row r's fp16 values at y16 + 2 * D * r (the first half of the
                    // row's fp32 slot in the y buffer, which the GEMV paths fill in fp32)
    int T, P, shared;
    int *status;
    int32_t *ovf;  // [E+1] an fp16 overflow of a tile's h or y flags its expert (E: the shared expert)
};

struct Tile {
    int shared;  // 1: the shared expert (bf16/fp16 rows), 0: a routed expert
    int e;       // routed expert
    int row0;    // first token row (x16 / h16 / y row)
    int ntok;    // token rows in the tile (1..BN)
    int m;       // weight-row tile (128 rows of gate and up for the first GEMM, 256 down rows)
};

// Tiles t = nt * m_tiles + m: token tile nt, weight-row tile m. The token tiles go longest
// first: the routed experts' full tiles (tile_desc[0, n_full)), the shared expert's, then the
// routed ragged tiles by decreasing size (tile_desc[n_full, routed)). routed = meta->n_tiles.
__device__ __forceinline__ int n_tiles_total(const GemmParams &p, int m_tiles, int routed) {
    const int sh = p.shared ? (p.T + BN - 1) / BN : 0;
    return (routed + sh) * m_tiles;
}

__device__ __forceinline__ Tile decode_tile(const GemmParams &p, int t, int m_tiles, int n_full) {
    Tile ti;
    ti.m = t % m_tiles;
    int nt = t / m_tiles;
    const int sh = p.shared ? (p.T + BN - 1) / BN : 0;
    if (nt >= n_full && nt < n_full + sh) {
        const int lt = nt - n_full;
        ti.shared = 1;
        ti.e = -1;
        ti.row0 = p.P + lt * BN;
        ti.ntok = min(BN, p.T - lt * BN);
    } else {
        if (nt >= n_full) nt -= sh;
        const int4 d = __ldg(p.tile_desc + nt);  // expert, first row, tokens
        ti.shared = 0;
        ti.e = d.x;
        ti.row0 = d.y;
        ti.ntok = d.z;
    }
    return ti;
}

// ------------------------------------------------------------------ producers
//
// Each of the 512 producer threads owns one 32-column half of one tile row per stage (thread u:
// row (u >> 1) & 127 of A tile u >> 8, half u & 1, so two neighbouring lanes read the two halves
// of one 16-byte chunk). The first GEMM's two A tiles are the same 128 rows of gate and of up; the
// down GEMM's are two consecutive 128-row tiles, so one token tile feeds 256 output rows. A format
// fetches the packed data of a stage into registers (a ring of PF stages in flight hides the HBM
// latency) and emits it as fp16 into the swizzled A tile. Every fp16 value is RN-even of the
// weight's exact fp32 value.

__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }
__device__ __forceinline__ void prefetch_l2(const void *a) { asm volatile("prefetch.global.L2 [%0];" ::"l"(a)); }
__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }

// fp16 high byte of magnitude m in {1, 3, 5, 7}: their low bytes are zero.
__device__ __forceinline__ uint32_t mag_hibyte(uint32_t m) {
    return m == 1u ? 0x3Cu : m == 3u ? 0x42u : m == 5u ? 0x45u : 0x47u;
}

// IQ2-style rows: one 32-weight sub-block (4 groups of 8) per stage.
struct IQ2Fmt {
    static constexpr int PF = 4;
    static constexpr int PD = 16;  // L2 prefetch distance (stages), every 8 stages (one 128-byte line of chunks)
    static constexpr int PE = 8;
    struct Data {
        uint2 q;  // index word, sign/scale word
        uint32_t d;
    };
    const uint8_t *qs;   // this row's code blocks
    const uint16_t *dp;  // this row's block scales
    const uint2 *gt;  // grid as fp16 high bytes, this lane's replica
    int swz;          // the row's chunk permutation (iq2_swz)
    int sb;           // which sub-block of the stage's 16-byte chunk
    __device__ __forceinline__ Data fetch(int kb) const {
        Data v;
        v.q = __ldg(reinterpret_cast<const uint2 *>(qs) + 2 * (kb ^ swz) + sb);  // chunk kb = 4 * block + part
        v.d = __ldg(dp + (kb >> 2));
        return v;
    }
    __device__ __forceinline__ void prefetch(int kb) const { prefetch_l2(qs + 16 * (kb ^ swz)); }
    __device__ __forceinline__ void emit(const Data &v, uint32_t tile, int r, int = 0) const {
        const __half2 dh = u2h(v.d | (v.d << 16));
        const uint32_t iw = v.q.x, sw = v.q.y;
        // (s+1)/16, exact in fp16; G*(s+1)/16 is then exact and one multiply by d rounds once
        const __half2 c16 = __float2half2_rn(static_cast<float>((sw >> 28) + 1u) * 0.0625f);
#pragma unroll
        for (int g = 0; g < 4; g++) {
            const uint2 ent = gt[((iw >> (8 * g)) & 255u) << 4];
            const uint32_t s7 = (sw >> (7 * g)) & 127u;
            const uint32_t lo = ent.x ^ ((s7 * 0x10204080u) & 0x80808080u);
            const uint32_t hi = ent.y ^ ((s7 * 0x01020408u + (__popc(s7) << 31)) & 0x80808080u);
            uint4 o;
            o.x = h2u(__hmul2(__hmul2(u2h(__byte_perm(lo, 0u, 0x1404)), c16), dh));
            o.y = h2u(__hmul2(__hmul2(u2h(__byte_perm(lo, 0u, 0x3424)), c16), dh));
            o.z = h2u(__hmul2(__hmul2(u2h(__byte_perm(hi, 0u, 0x1404)), c16), dh));
            o.w = h2u(__hmul2(__hmul2(u2h(__byte_perm(hi, 0u, 0x3424)), c16), dh));
            st_shared16(tile + sw128_off(r, sb * 4 + g), o);
        }
    }
};

// Q2_K-style rows, half row: two 16-weight sub-blocks per stage. The 4 possible values of a
// sub-block, RN-even(fp32(d*sc*q - dmin*m)) for q = 0..3, are formed once; each code byte then
// selects its four values with two byte permutations (selectors from a table).
struct Q2KFmt {
    static constexpr int PF = 4;
    static constexpr int PD = 8;  // L2 prefetch distance (stages), every 4 stages (one 80-byte block)
    static constexpr int PE = 4;
    struct Data {
        uint2 q;      // 2 x 16 codes
        uint32_t sc;  // two scale bytes (low 4 bits sc, high 4 bits m)
        uint32_t dd;
    };
    const uint8_t *sq;    // this row's blocks (scales, codes)
    const uint32_t *ddp;  // this row's d | dmin words
    int half;             // which half of the stage's 64 columns
    const uint2 *st;  // code byte -> two byte_perm selectors, this lane's replica
    __device__ __forceinline__ Data fetch(int kb) const {
        const int b = kb >> 2, part = kb & 3;
        const uint8_t *blk = sq + b * 80;
        Data v;
        v.q = __ldg(reinterpret_cast<const uint2 *>(blk + 16 + 16 * part + 8 * half));
        v.sc = __ldg(reinterpret_cast<const uint16_t *>(blk + 4 * part + 2 * half));
        v.dd = __ldg(ddp + b);
        return v;
    }
    __device__ __forceinline__ void prefetch(int kb) const {
        const uint8_t *blk = sq + (kb >> 2) * 80;
        prefetch_l2(blk);
        prefetch_l2(blk + 79);
    }
    __device__ __forceinline__ void emit(const Data &v, uint32_t tile, int r, int = 0) const {
        const float d = f16_to_f32(static_cast<uint16_t>(v.dd & 0xffffu));
        const float dmin = f16_to_f32(static_cast<uint16_t>(v.dd >> 16));
#pragma unroll
        for (int j = 0; j < 2; j++) {  // sub-block 2 * half + j of the stage
            const uint32_t sc = v.sc >> (8 * j);
            const uint32_t q = j ? v.q.y : v.q.x;
            const float ds = __fmul_rn(d, static_cast<float>(sc & 15u));
            const float dm = __fmul_rn(dmin, static_cast<float>((sc >> 4) & 15u));
            const uint32_t p01 = pack_h2(q2k_weight(ds, dm, 0u), q2k_weight(ds, dm, 1u));
            const uint32_t p23 = pack_h2(q2k_weight(ds, dm, 2u), q2k_weight(ds, dm, 3u));
#pragma unroll
            for (int hh = 0; hh < 2; hh++) {
                const uint2 s0 = st[((q >> (16 * hh)) & 255u) << 4];
                const uint2 s1 = st[((q >> (16 * hh + 8)) & 255u) << 4];
                uint4 o;
                o.x = __byte_perm(p01, p23, s0.x);
                o.y = __byte_perm(p01, p23, s0.y);
                o.z = __byte_perm(p01, p23, s1.x);
                o.w = __byte_perm(p01, p23, s1.y);
                st_shared16(tile + sw128_off(r, 4 * half + 2 * j + hh), o);
            }
        }
    }
};

// The 4-bit variant (Q4_K-style rows, 144-byte blocks of 8 sub-blocks of 32): each weight is
// computed as its exact fp32 value (one rounding of d sc q - dmin m) and then RN-even to fp16,
// as for the Q2_K-style rows. fetch keeps the block's d | dmin word and the two words that hold
// the sub-block's scale and min bits.
__device__ __forceinline__ void q4_scales(uint32_t dd, uint32_t lo_word, uint32_t hi_word, int sub, float &ds, float &dm) {
    const uint32_t low = (lo_word >> (8 * (sub & 3))) & 0xffu;
    const uint32_t high = (hi_word >> (8 * (sub >> 1) + 4 * (sub & 1))) & 15u;
    ds = __fmul_rn(f16_to_f32(static_cast<uint16_t>(dd & 0xffffu)), static_cast<float>((low & 15u) | ((high & 3u) << 4)));
    dm = __fmul_rn(f16_to_f32(static_cast<uint16_t>(dd >> 16)), static_cast<float>((low >> 4) | ((high >> 2) << 4)));
}

// Eight codes of a u32 (weight i in bits 4i..4i+3) as four fp16 pairs.
__device__ __forceinline__ uint4 q4_to_f16x8(uint32_t word, float ds, float dm) {
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; i++) v[i] = q2k_weight(ds, dm, (word >> (4 * i)) & 15u);
    return make_uint4(pack_h2(v[0], v[1]), pack_h2(v[2], v[3]), pack_h2(v[4], v[5]), pack_h2(v[6], v[7]));
}

// Rows of the 4-bit variant (gate, up or down), half row: one 32-weight sub-block per stage.
struct Q4Fmt {
    static constexpr int PF = 2;
    static constexpr int PD = 8;  // L2 prefetch distance (stages), once per 144-byte block (4 stages)
    static constexpr int PE = 4;
    struct Data {
        uint4 q;
        uint32_t dd, lo, hi;
    };
    const uint8_t *row;
    int part;
    __device__ __forceinline__ Data fetch(int kb) const {
        const int b = kb >> 2, sub = 2 * (kb & 3) + part;
        const uint8_t *blk = row + b * 144;
        Data v;
        v.q = __ldg(reinterpret_cast<const uint4 *>(blk + 16) + sub);
        v.dd = __ldg(reinterpret_cast<const uint32_t *>(blk));
        v.lo = __ldg(reinterpret_cast<const uint32_t *>(blk + 4) + (sub >> 2));
        v.hi = __ldg(reinterpret_cast<const uint32_t *>(blk + 12));
        return v;
    }
    __device__ __forceinline__ void prefetch(int kb) const {
        const uint8_t *blk = row + (kb >> 2) * 144;
        prefetch_l2(blk);
        prefetch_l2(blk + 143);
    }
    __device__ __forceinline__ void emit(const Data &v, uint32_t tile, int r, int kb) const {
        float ds, dm;
        q4_scales(v.dd, v.lo, v.hi, 2 * (kb & 3) + part, ds, dm);
        st_shared16(tile + sw128_off(r, 4 * part + 0), q4_to_f16x8(v.q.x, ds, dm));
        st_shared16(tile + sw128_off(r, 4 * part + 1), q4_to_f16x8(v.q.y, ds, dm));
        st_shared16(tile + sw128_off(r, 4 * part + 2), q4_to_f16x8(v.q.z, ds, dm));
        st_shared16(tile + sw128_off(r, 4 * part + 3), q4_to_f16x8(v.q.w, ds, dm));
    }
};

// bf16 rows (shared gate/up), half row: 32 columns per stage -> fp16.
struct BF16Fmt {
    static constexpr int PF = 1;
    static constexpr int PD = 0;  // no L2 prefetch
    static constexpr int PE = 1;
    struct Data {
        uint4 v[4];
    };
    const uint16_t *row;
    int half;
    __device__ __forceinline__ Data fetch(int kb) const {
        Data d;
        const uint4 *src = reinterpret_cast<const uint4 *>(row + kb * BK + 32 * half);
#pragma unroll
        for (int c = 0; c < 4; c++) d.v[c] = __ldg(src + c);
        return d;
    }
    __device__ __forceinline__ void prefetch(int) const {}
    __device__ __forceinline__ void emit(const Data &d, uint32_t tile, int r, int = 0) const {
#pragma unroll
        for (int c = 0; c < 4; c++) {
            const uint4 v = d.v[c];
            st_shared16(tile + sw128_off(r, 4 * half + c),
                        make_uint4(pack_h2(bf16_lo(v.x), bf16_hi(v.x)), pack_h2(bf16_lo(v.y), bf16_hi(v.y)),
                                   pack_h2(bf16_lo(v.z), bf16_hi(v.z)), pack_h2(bf16_lo(v.w), bf16_hi(v.w))));
        }
    }
};

// fp16 rows (shared down), half row: 32 columns per stage -> copied.
struct F16Fmt {
    static constexpr int PF = 1;
    static constexpr int PD = 0;
    static constexpr int PE = 1;
    struct Data {
        uint4 v[4];
    };
    const uint16_t *row;
    int half;
    __device__ __forceinline__ Data fetch(int kb) const {
        Data d;
        const uint4 *src = reinterpret_cast<const uint4 *>(row + kb * BK + 32 * half);
#pragma unroll
        for (int c = 0; c < 4; c++) d.v[c] = __ldg(src + c);
        return d;
    }
    __device__ __forceinline__ void prefetch(int) const {}
    __device__ __forceinline__ void emit(const Data &d, uint32_t tile, int r, int = 0) const {
#pragma unroll
        for (int c = 0; c < 4; c++) st_shared16(tile + sw128_off(r, 4 * half + c), d.v[c]);
    }
};

struct Pipe {  // the producers' view of the stage ring
    uint64_t *bars;
    int S;
    int stage;
    uint32_t phase;
    volatile int *abort_flag;
    int *status;
};

// Produces the A operand of K stages [kb_begin, kb_end) of one tile (num_kb stages) for this
// thread's row (slice).
template <class Fmt>
__device__ __forceinline__ bool produce_tile(const Fmt &f, int kb_begin, int kb_end, int num_kb, uint8_t *smem,
                                             int stage_bytes, int a_off, int r, Pipe &pp) {
    constexpr int PF = Fmt::PF;
    typename Fmt::Data ring[PF];
#pragma unroll
    for (int i = 0; i < PF; i++)
        if (kb_begin + i < kb_end) ring[i] = f.fetch(kb_begin + i);
    for (int kb0 = kb_begin; kb0 < kb_end; kb0 += PF) {
#pragma unroll
        for (int i = 0; i < PF; i++) {
            const int kb = kb0 + i;
            if (kb >= kb_end) break;
            const typename Fmt::Data cur = ring[i];
            if (kb + PF < kb_end) ring[i] = f.fetch(kb + PF);
            if (Fmt::PD > 0 && kb % Fmt::PE == 0 && kb + Fmt::PD < num_kb) f.prefetch(kb + Fmt::PD);
            if (!mbar_wait(smem_u32(pp.bars + 2 * pp.S + pp.stage), pp.phase ^ 1u, pp.abort_flag, pp.status))
                return false;
            f.emit(cur, smem_u32(smem + pp.stage * stage_bytes + a_off), r, kb);
            fence_proxy_async();
            mbar_arrive(smem_u32(pp.bars + pp.stage));
            if (++pp.stage == pp.S) {
                pp.stage = 0;
                pp.phase ^= 1u;
            }
        }
    }
    return true;
}

// ------------------------------------------------------------------ the kernel

// Tensor maps of one token operand with box heights 16, 32, 64, 128 and 256 rows: a tile
// loads only the smallest box that covers its tokens.
struct TokenMaps {
    CUtensorMap m[kTokenBoxes];
};

__device__ __forceinline__ int box_index(int ntok) {
    int i = 0;
    while ((16 << i) < ntok) i++;
    return i;
}

// FMT 0: IQ2-style gate/up, Q2_K-style down; FMT 1: the 4-bit variant's rows. PAIR: see Cfg.
// Roles: warp 0 lane 0 issues the token-tile copies; warp 1 allocates tensor memory and one lane
// issues the MMAs (in a pair, only rank 0 does; rank 1's lane forwards its stages' readiness and
// its epilogue's release of the accumulators to rank 0); warps 2..17 produce and then read back.
template <int KIND, int FMT, bool PAIR>
__global__ void __launch_bounds__(kThreads, 1) gemm_kernel(const __grid_constant__ TokenMaps maps, GemmParams p) {
    pdl_wait();
    using C = Cfg<KIND, PAIR>;
    constexpr int S = C::STAGES;
    constexpr int NA = C::NA;
    constexpr int CTAS = C::CTAS;
    constexpr int B_BYTES = C::BROWS * BK * 2;
    constexpr int STAGE_BYTES = NA * A_BYTES + B_BYTES;
    extern __shared__ uint8_t smem_raw[];
    // align by an integer offset so that every pointer below stays a shared-memory pointer (the
    // offset is the same in both CTAs of a pair, as the pair's MMAs require)
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint2 *table = reinterpret_cast<uint2 *>(smem + S * STAGE_BYTES);  // [256][16] replicated lookup table
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S * STAGE_BYTES + kTableBytes);
    // bars: full_a[S], full_b[S], empty[S], acc_full, acc_empty, spare, (pairs) peer_full[S], peer_acc
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + 4 * S + 4);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int D = p.w.D, F = p.w.F;
    // weight rows per m-tile, over the pair: the first GEMM's 128 (per CTA) rows of gate and of up,
    // the down GEMM's two 128-row tiles (per CTA)
    constexpr int MR = (KIND == UP ? BM : BM * NA) * CTAS;
    const uint32_t crank = PAIR ? cluster_ctarank() : 0u;  // rank in the pair (0 issues the MMAs)
    const int unit = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
    const int units = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
    const int m_tiles = (KIND == UP ? F : D) / MR;
    const int routed = p.meta->n_tiles;
    const int n_full = p.meta->n_full;
    const int total = n_tiles_total(p, m_tiles, routed);
    // (a pair never leaves early: both CTAs take part in the joint allocation and the cluster barriers)
    if (!PAIR && unit >= total) return;  // uniform over the CTA, before any allocation
    const int num_kb = (KIND == UP ? D : F) / BK;

    auto full_a = [&](int s) { return smem_u32(bars + s); };
    auto full_b = [&](int s) { return smem_u32(bars + S + s); };
    auto empty = [&](int s) { return smem_u32(bars + 2 * S + s); };
    const uint32_t acc_full = smem_u32(bars + 3 * S), acc_empty = smem_u32(bars + 3 * S + 1);
    const uint32_t spare = smem_u32(bars + 3 * S + 2);
    auto a_tile = [&](int s, int a) { return smem_u32(smem + s * STAGE_BYTES + a * A_BYTES); };
    auto b_tile = [&](int s) { return smem_u32(smem + s * STAGE_BYTES + NA * A_BYTES); };
    // pairs: rank 1's lane of warp 1 forwards, for each stage, that its half (producers' rows
    // and token copy) is in (peer_full on rank 0), and for each tile, that its epilogue has read
    // the accumulators (peer_acc on rank 0)
    auto peer_full = [&](int s) { return smem_u32(bars + 3 * S + 3 + s); };
    const uint32_t peer_acc = smem_u32(bars + 4 * S + 3);
    auto wait = [&](uint32_t bar, uint32_t parity) { return mbar_wait(bar, parity, abort_flag, p.status); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; s++) {
            mbar_init(full_a(s), kProducers);
            mbar_init(full_b(s), 1);
            mbar_init(empty(s), 1);
            mbar_init(peer_full(s), 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, kProducers);
        mbar_init(spare, 1);
        mbar_init(peer_acc, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // lookup table, replicated 16 times so that the 16 lanes of a half-warp never share a bank
    for (int i = threadIdx.x; i < 256 * 16; i += kThreads) {
        const uint32_t e = static_cast<uint32_t>(i >> 4);
        uint2 v;
        if (KIND == UP) {  // grid entry e as fp16 high bytes
            const uint8_t *g = p.grid + 8 * e;
            v.x = mag_hibyte(g[0]) | (mag_hibyte(g[1]) << 8) | (mag_hibyte(g[2]) << 16) | (mag_hibyte(g[3]) << 24);
            v.y = mag_hibyte(g[4]) | (mag_hibyte(g[5]) << 8) | (mag_hibyte(g[6]) << 16) | (mag_hibyte(g[7]) << 24);
        } else {  // code byte e: selectors of values q0, q1 and q2, q3 (value q at bytes 2q, 2q+1)
            uint32_t sel[4];
#pragma unroll
            for (int i2 = 0; i2 < 4; i2++) sel[i2] = (e >> (2 * i2)) & 3u;
            v.x = (2 * sel[0]) | ((2 * sel[0] + 1) << 4) | ((2 * sel[1]) << 8) | ((2 * sel[1] + 1) << 12);
            v.y = (2 * sel[2]) | ((2 * sel[2] + 1) << 4) | ((2 * sel[3]) << 8) | ((2 * sel[3] + 1) << 12);
        }
        table[i] = v;
    }
    if (warp == 1) {
        if (PAIR) {  // one warp of each CTA of the pair allocates, jointly
            asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_holder)),
                         "r"(C::TMEM_COLS)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
        } else {
            asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_holder)),
                         "r"(C::TMEM_COLS)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        }
    }
    tc_fence_before();
    __syncthreads();
    if (PAIR) cluster_sync();  // both CTAs' barriers are initialised before any remote arrive
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    // token rows of a tile: MMA N = tokens rounded up to 16 per CTA's half (a pair's N is at least 32)
    auto mma_n = [](int ntok) { return PAIR ? max(32, (ntok + 31) & ~31) : max(16, (ntok + 15) & ~15); };

    if (warp == 0) {
        // ---------------------------------------------------------- TMA: token tiles (this CTA's half)
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int issued_parity[S];
#pragma unroll
            for (int s = 0; s < S; s++) issued_parity[s] = -1;
            bool ok = true;
            for (int t = unit; t < total && ok; t += units) {
                const Tile ti = decode_tile(p, t, m_tiles, n_full);
                const int half = mma_n(ti.ntok) / CTAS;
                const int bi = box_index(half);
                const CUtensorMap *map = &maps.m[bi];
                const uint32_t bytes = static_cast<uint32_t>(16 << bi) * BK * 2;
                const int row = ti.row0 + static_cast<int>(crank) * half;
                for (int kb = 0; kb < num_kb; kb++) {
                    if (!wait(empty(stage), phase ^ 1u)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(full_b(stage), bytes);
                    tma_load_2d(b_tile(stage), map, kb * BK, row, full_b(stage));
                    issued_parity[stage] = static_cast<int>(phase);
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok)  // let copies still in flight land before the CTA exits
                for (int s = 0; s < S; s++)
                    if (issued_parity[s] >= 0) mbar_drain(full_b(s), static_cast<uint32_t>(issued_parity[s]));
        }
    } else if (warp == 1 && crank == 0) {
        // ---------------------------------------------------------- MMA issue (one thread)
        if (lane == 0) {
            const uint32_t peer_acc_full = PAIR ? map_shared(acc_full, 1u) : 0u;
            int stage = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true, issued = false;
            for (int t = unit; t < total && ok; t += units) {
                const Tile ti = decode_tile(p, t, m_tiles, n_full);
                // both CTAs' epilogues have read the previous tile's accumulators
                if (!wait(acc_empty, acc_phase ^ 1u) || (PAIR && !wait(peer_acc, acc_phase ^ 1u))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t idesc = idesc_f16(BM * CTAS, mma_n(ti.ntok));
                // one stage: wait for both halves (producers' rows, token copy; tested together
                // first), the MMAs, the commit that frees the stage
                auto stage_mmas = [&](int st, uint32_t ph, int kb) -> bool {
                    if ((!mbar_test2(full_a(st), full_b(st), ph) && (!wait(full_a(st), ph) || !wait(full_b(st), ph))) ||
                        (PAIR && !wait(peer_full(st), ph)))
                        return false;
                    tc_fence_after();
                    // one add per operand descriptor: this thread shares its issue slots with producers
                    const uint32_t a_lo = sw128_desc_lo(a_tile(st, 0)), b_lo = sw128_desc_lo(b_tile(st));
#pragma unroll
                    for (int a = 0; a < NA; a++)
#pragma unroll
                        for (int k = 0; k < BK / 16; k++) {
                            const uint32_t ad = a_lo + static_cast<uint32_t>((a * A_BYTES + k * 32) >> 4);
                            const uint32_t bd = b_lo + static_cast<uint32_t>((k * 32) >> 4);
                            if (PAIR)
                                tc_mma_pair(tmem + a * BN, ad, bd, kSw128DescHi, idesc, (kb | k) != 0);
                            else
                                tc_mma(tmem + a * BN, ad, bd, kSw128DescHi, idesc, (kb | k) != 0);
                        }
                    issued = true;
                    if (PAIR) {  // the stage is free in both CTAs once these MMAs are done
                        tc_commit_pair(empty(st));
                        tc_commit_pair(map_shared(empty(st), 1u));
                    } else {
                        tc_commit(empty(st));
                    }
                    return true;
                };
                auto advance = [&]() {
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                };
                // stages up to the ring's start, then whole turns of the ring with the stage index
                // known at compile time (fewer instructions between stages), then the rest
                int kb = 0;
                for (; ok && kb < num_kb && stage != 0; kb++, advance()) ok = stage_mmas(stage, phase, kb);
                for (; ok && kb + S <= num_kb; kb += S) {
#pragma unroll
                    for (int st = 0; st < S; st++)
                        if (ok) ok = stage_mmas(st, phase, kb + st);
                    phase ^= 1u;
                }
                for (; ok && kb < num_kb; kb++, advance()) ok = stage_mmas(stage, phase, kb);
                if (!ok) break;
                if (PAIR) {
                    tc_commit_pair(acc_full);
                    tc_commit_pair(peer_acc_full);
                } else {
                    tc_commit(acc_full);
                }
                acc_phase ^= 1u;
            }
            if (!ok && issued) {  // wait for the MMAs in flight before the memory goes away
                if (PAIR)
                    tc_commit_pair(spare);
                else
                    tc_commit(spare);
                mbar_drain(spare, 0);
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- a pair's rank 1: forward readiness
        if (PAIR && lane == 0) {
            int stage = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int t = unit; t < total && ok; t += units) {
                for (int kb = 0; kb < num_kb; kb++) {
                    if (!wait(full_a(stage), phase) || !wait(full_b(stage), phase)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_remote(map_shared(peer_full(stage), 0u));  // this CTA's half of the stage is in
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                // this CTA's epilogue of the tile has read its accumulators: rank 0 may start the next tile
                if (!ok || !wait(acc_empty, acc_phase)) break;
                mbar_arrive_remote(map_shared(peer_acc, 0u));
                acc_phase ^= 1u;
            }
        }
    } else {
        // ---------------------------------------------------------- producers, then epilogue
        const int u = (warp - 2) * 32 + lane;  // 0..511
        // row (u >> 1) & 127 of A tile u >> 8 (gate / up, or the first / second 128 down rows), half u & 1
        const int r = (u >> 1) & 127;  // tile row
        const int sel = u >> 8;
        const int part = u & 1;
        const int q = warp & 3;                // TMEM lane quarter this warp may access
        const int colq = (warp - 2) >> 2;      // epilogue: which 16-column chunks (one of four)
        const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
        const uint2 *tab = table + (lane & 15);
        // first row of this CTA's A tile a within the m-tile
        auto tile_row0 = [&](int a) {
            return (KIND == DOWN ? a * BM * CTAS : 0) + static_cast<int>(crank) * BM;
        };
        Pipe pp{bars, S, 0, 0u, abort_flag, p.status};
        // K stages [kb_begin, kb_end) of tile tt's A operand, in the tile's weight format
        auto produce = [&](const Tile &tt, int kb_begin, int kb_end) -> bool {
            const int wrow = tt.m * MR + tile_row0(sel) + r;
            const int a_off = sel * A_BYTES;
            if (KIND == UP) {
                if (tt.shared) {
                    BF16Fmt f{(sel ? p.w.sh_up : p.w.sh_gate) + static_cast<size_t>(wrow) * D, part};
                    return produce_tile(f, kb_begin, kb_end, num_kb, smem, STAGE_BYTES, a_off, r, pp);
                } else if (FMT == 1) {
                    Q4Fmt f{q4_row(p.w, sel, tt.e, wrow), part};
                    return produce_tile(f, kb_begin, kb_end, num_kb, smem, STAGE_BYTES, a_off, r, pp);
                } else {
                    IQ2Fmt f{iq2_qs_row(p.w, sel, tt.e, wrow), iq2_d_row(p.w, sel, tt.e, wrow), tab, iq2_swz(p.w, wrow),
                             part};
                    return produce_tile(f, kb_begin, kb_end, num_kb, smem, STAGE_BYTES, a_off, r, pp);
                }
            } else {
                if (tt.shared) {
                    F16Fmt f{p.w.sh_down_f16 + static_cast<size_t>(wrow) * F, part};
                    return produce_tile(f, kb_begin, kb_end, num_kb, smem, STAGE_BYTES, a_off, r, pp);
                } else if (FMT == 1) {
                    Q4Fmt f{q4_row(p.w, 2, tt.e, wrow), part};
                    return produce_tile(f, kb_begin, kb_end, num_kb, smem, STAGE_BYTES, a_off, r, pp);
                } else {
                    Q2KFmt f{q2k_sq_row(p.w, tt.e, wrow), q2k_dd_row(p.w, tt.e, wrow), part, tab};
                    return produce_tile(f, kb_begin, kb_end, num_kb, smem, STAGE_BYTES, a_off, r, pp);
                }
            }
        };
        uint32_t acc_phase = 0;
        bool ok = true;
        for (int t = unit; t < total && ok; t += units) {
            const Tile ti = decode_tile(p, t, m_tiles, n_full);
            ok = produce(ti, 0, num_kb);
            if (!ok) break;
            // epilogue: accumulators -> registers -> global; four warps per TMEM lane quarter
            if (!wait(acc_full, acc_phase)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // overflow bits of the tile's fp16 results: bit 15 / 31 of f16x2_overflow for a half that is
            // +-inf or NaN (the value is beyond fp16's range after rounding)
            uint32_t bad = 0;
            bool range_ok_down = true;  // the down GEMM's per-value test (its register budget prefers it)
            static_assert(NA == 2, "the epilogue reads two accumulators");
            for (int c0 = 16 * colq; c0 < ti.ntok; c0 += 64) {
                // 16 columns of both accumulators (gate and up, or the two down tiles), one wait
                uint32_t v0[16], v1[16];
                tmem_ld16_start(tmem + lane_addr + c0, v0);
                tmem_ld16_start(tmem + lane_addr + BN + c0, v1);
                tmem_wait_ld(v0, v1);
                // two columns (tokens) per conversion: one packed fp32 -> fp16x2 round-to-nearest-even;
                // a chunk of 16 valid tokens (all but a ragged tile's last) takes no per-token checks
                const int nv = min(16, ti.ntok - c0);  // valid tokens of the chunk, uniform over the warp
                if (KIND == UP) {
                    uint16_t *dst = p.h16 + static_cast<size_t>(ti.row0 + c0) * F + ti.m * MR + tile_row0(0) + q * 32 + lane;
                    if (nv == 16) {
#pragma unroll
                        for (int j = 0; j < 16; j += 2) {
                            const uint32_t hp = pack_h2(swiglu_fast(__uint_as_float(v0[j]), __uint_as_float(v1[j])),
                                                        swiglu_fast(__uint_as_float(v0[j + 1]), __uint_as_float(v1[j + 1])));
                            bad |= f16x2_overflow(hp);
                            dst[static_cast<size_t>(j) * F] = static_cast<uint16_t>(hp & 0xffffu);
                            dst[static_cast<size_t>(j + 1) * F] = static_cast<uint16_t>(hp >> 16);
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 16; j += 2) {
                            const uint32_t hp = pack_h2(swiglu_fast(__uint_as_float(v0[j]), __uint_as_float(v1[j])),
                                                        swiglu_fast(__uint_as_float(v0[j + 1]), __uint_as_float(v1[j + 1])));
                            if (j < nv) {
                                bad |= f16x2_overflow(hp) & (j + 1 < nv ? 0x80008000u : 0x00008000u);
                                dst[static_cast<size_t>(j) * F] = static_cast<uint16_t>(hp & 0xffffu);
                            }
                            if (j + 1 < nv) dst[static_cast<size_t>(j + 1) * F] = static_cast<uint16_t>(hp >> 16);
                        }
                    }
                } else {
#pragma unroll 1
                    for (int a = 0; a < NA; a++) {  // the two 128-row tiles
                        uint16_t *dst = p.y16 + static_cast<size_t>(ti.row0 + c0) * (2 * D) + ti.m * MR + tile_row0(a) +
                                        q * 32 + lane;
#pragma unroll
                        for (int j = 0; j < 16; j += 2) {
                            const float y0 = __uint_as_float(a ? v1[j] : v0[j]);
                            const float y1 = __uint_as_float(a ? v1[j + 1] : v0[j + 1]);
                            const uint32_t yp = pack_h2(y0, y1);
                            if (c0 + j < ti.ntok) {
                                range_ok_down &= fabsf(y0) <= 65504.0f;
                                dst[static_cast<size_t>(j) * (2 * D)] = static_cast<uint16_t>(yp & 0xffffu);
                            }
                            if (c0 + j + 1 < ti.ntok) {
                                range_ok_down &= fabsf(y1) <= 65504.0f;
                                dst[static_cast<size_t>(j + 1) * (2 * D)] = static_cast<uint16_t>(yp >> 16);
                            }
                        }
                    }
                }
            }
            const bool range_ok = bad == 0 && range_ok_down;
            if (!range_ok) p.ovf[ti.shared ? p.w.E : ti.e] = 1;  // recomputed in fp32 before the combine
            tc_fence_before();
            mbar_arrive(acc_empty);
            acc_phase ^= 1u;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (PAIR) cluster_sync();  // neither CTA leaves while the pair's MMAs may still touch its memory
    if (warp == 1) {
        tc_fence_after();
        if (PAIR)
            asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS) : "memory");
        else
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS) : "memory");
    }
}

// The A operand as the producers write it, for tests: one 128-row x 64-column stage per CTA,
// decoded by the same formats into a swizzled shared-memory tile, then un-swizzled into
// dst16 [rows][cols] (fp16 bits).
__global__ void __launch_bounds__(kProducers) producer_dump_kernel(DeviceWeights w, const uint8_t *grid, int expert,
                                                            int matrix, uint16_t *dst16) {
    __shared__ __align__(1024) uint8_t tile[A_BYTES];
    __shared__ uint2 table[256 * 16];
    const int lane = threadIdx.x & 31;
    // the GEMM producers' slices of one A tile: row (u >> 1) & 127, half u & 1 for u < 256
    const int u = threadIdx.x;
    const bool down = matrix == DS4MOE_DOWN;
    const int r = (u >> 1) & 127;
    for (int i = threadIdx.x; i < 256 * 16; i += blockDim.x) {
        const uint32_t e = static_cast<uint32_t>(i >> 4);
        uint2 v;
        if (!down) {
            const uint8_t *g = grid + 8 * e;
            v.x = mag_hibyte(g[0]) | (mag_hibyte(g[1]) << 8) | (mag_hibyte(g[2]) << 16) | (mag_hibyte(g[3]) << 24);
            v.y = mag_hibyte(g[4]) | (mag_hibyte(g[5]) << 8) | (mag_hibyte(g[6]) << 16) | (mag_hibyte(g[7]) << 24);
        } else {
            uint32_t c[4];
            for (int i2 = 0; i2 < 4; i2++) c[i2] = (e >> (2 * i2)) & 3u;
            v.x = (2 * c[0]) | ((2 * c[0] + 1) << 4) | ((2 * c[1]) << 8) | ((2 * c[1] + 1) << 12);
            v.y = (2 * c[2]) | ((2 * c[2] + 1) << 4) | ((2 * c[3]) << 8) | ((2 * c[3] + 1) << 12);
        }
        table[i] = v;
    }
    __syncthreads();
    const int rows = down ? w.D : w.F, cols = down ? w.F : w.D;
    const int m = blockIdx.x, kb = blockIdx.y;
    const int wrow = m * BM + r;
    const uint32_t t = smem_u32(tile);
    const uint2 *tab = table + (lane & 15);
    if (down && u < 256) {
        Q2KFmt f{q2k_sq_row(w, expert, wrow), q2k_dd_row(w, expert, wrow), u & 1, tab};
        f.emit(f.fetch(kb), t, r);
    } else if (u < 256) {
        const int m = matrix == DS4MOE_GATE ? 0 : 1;
        IQ2Fmt f{iq2_qs_row(w, m, expert, wrow), iq2_d_row(w, m, expert, wrow), tab, iq2_swz(w, wrow), u & 1};
        f.emit(f.fetch(kb), t, r);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < BM * 8; i += blockDim.x) {  // 8 chunks of 16 bytes per row
        const int rr = i >> 3, c = i & 7;
        const uint4 v = *reinterpret_cast<const uint4 *>(tile + sw128_off(rr, c));
        if (m * BM + rr < rows)
            *reinterpret_cast<uint4 *>(dst16 + static_cast<size_t>(m * BM + rr) * cols + kb * BK + 8 * c) = v;
    }
}

// x (bf16) -> x16 (fp16) for rows of tensor-core groups and of the shared expert, one warp per
// token: lane j < k resolves the row of the token's j-th pair (or that its group is not on the
// tensor cores), and the shared expert's row is P + token; the warp then reads the token's D values once, 32
// columns x 8 per lane and group of four steps, and writes each group to every destination row. A
// value beyond fp16's range flags each destination's expert (ovf[E]: the shared expert), whose
// results are then recomputed in fp32.
__global__ void __launch_bounds__(256, 4) gather_kernel(const uint16_t *__restrict__ x, const int32_t *__restrict__ inv,
                                                     const int32_t *__restrict__ topk_idx,
                                                     const int32_t *__restrict__ counts,
                                                     const uint8_t *__restrict__ tc_ok, int gemm_min, int k, int D,
                                                     int P, int T, int shared, uint16_t *__restrict__ x16,
                                                     int32_t *__restrict__ ovf, int E) {
    pdl_wait();
    constexpr int G = 4;  // 16-byte steps per lane held at once
    const int D8 = D / 8;
    const int lane = threadIdx.x & 31;
    const int warps = gridDim.x * (blockDim.x >> 5);
    for (int tok = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); tok < T; tok += warps) {
        int row = -1, owner = E;  // this lane's destination row (routed pair j = lane) and its expert
        if (lane < k) {
            const int pair = tok * k + lane;
            const int e = topk_idx[pair];
            owner = e;
            if (gemm_min > 0 && counts[e] >= gemm_min && tc_ok[e]) row = inv[pair];
        }
        const unsigned rows = __ballot_sync(0xffffffffu, row >= 0);
        if (!rows && !shared) continue;
        bool range_ok = true;
        const uint4 *src = reinterpret_cast<const uint4 *>(x + static_cast<size_t>(tok) * D);
        for (int c0 = 0; c0 < D8; c0 += 32 * G) {
            uint4 v[G];
#pragma unroll
            for (int g = 0; g < G; g++) {
                const int c = c0 + 32 * g + lane;
                if (c < D8) {
                    const uint4 b = __ldg(src + c);
                    const float f[8] = {bf16_lo(b.x), bf16_hi(b.x), bf16_lo(b.y), bf16_hi(b.y),
                                        bf16_lo(b.z), bf16_hi(b.z), bf16_lo(b.w), bf16_hi(b.w)};
#pragma unroll
                    for (int j = 0; j < 8; j++) range_ok &= fabsf(f[j]) <= 65504.0f;
                    v[g] = make_uint4(pack_h2(f[0], f[1]), pack_h2(f[2], f[3]), pack_h2(f[4], f[5]), pack_h2(f[6], f[7]));
                }
            }
            for (unsigned m = rows; m; m &= m - 1) {
                const int dl = __ffs(m) - 1;
                const int r = __shfl_sync(0xffffffffu, row, dl);
                uint4 *dst = reinterpret_cast<uint4 *>(x16 + static_cast<size_t>(r) * D);
#pragma unroll
                for (int g = 0; g < G; g++) {
                    const int c = c0 + 32 * g + lane;
                    if (c < D8) dst[c] = v[g];
                }
            }
            if (shared) {
                uint4 *dst = reinterpret_cast<uint4 *>(x16 + static_cast<size_t>(P + tok) * D);
#pragma unroll
                for (int g = 0; g < G; g++) {
                    const int c = c0 + 32 * g + lane;
                    if (c < D8) dst[c] = v[g];
                }
            }
        }
        if (!__all_sync(0xffffffffu, range_ok)) {
            if (row >= 0) ovf[owner] = 1;
            if (shared && lane == 0) ovf[E] = 1;
        }
    }
}

int sm_count_tc() {
    static int n = 0;
    if (!n) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 148;
    }
    return n;
}

template <int KIND, int FMT, bool PAIR>
int launch_gemm_fmt(const TokenMaps &maps, const GemmParams &p, cudaStream_t s) {
    using C = Cfg<KIND, PAIR>;
    const size_t smem = 1024 + static_cast<size_t>(C::STAGES) * (C::NA * A_BYTES + C::BROWS * BK * 2) + kTableBytes + 256;
    static int seen[64];
    const void *fn = reinterpret_cast<const void *>(gemm_kernel<KIND, FMT, PAIR>);
    const int err = ensure_smem(fn, static_cast<int>(smem), seen);
    if (err) return err;
    if (!PAIR) return launch_pdl(gemm_kernel<KIND, FMT, PAIR>, dim3(sm_count_tc()), dim3(kThreads), smem, s, maps, p);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(sm_count_tc() & ~1));  // one CTA per SM, in pairs
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see pdl_wait
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return static_cast<int>(cudaLaunchKernelEx(&cfg, gemm_kernel<KIND, FMT, PAIR>, maps, p));
}

// CTA pairs when the weight rows split into 256-row (first GEMM) or 512-row (down GEMM) m-tiles.
template <int KIND>
int launch_gemm(const TokenMaps &maps, const GemmParams &p, bool pairs, cudaStream_t s) {
    const bool pair = pairs && (KIND == UP ? p.w.F % 256 == 0 : p.w.D % 512 == 0);
    if (p.w.fmt == 1)
        return pair ? launch_gemm_fmt<KIND, 1, true>(maps, p, s) : launch_gemm_fmt<KIND, 1, false>(maps, p, s);
    return pair ? launch_gemm_fmt<KIND, 0, true>(maps, p, s) : launch_gemm_fmt<KIND, 0, false>(maps, p, s);
}

GemmParams make_params(const DeviceWeights &w, const Workspace &ws, int T, int k, bool shared) {
    GemmParams p;
    p.w = w;
    p.tile_desc = reinterpret_cast<const int4 *>(ws.tile_desc);
    p.meta = ws.meta;
    p.grid = ws.grid;
    p.h16 = ws.h16;
    p.y16 = reinterpret_cast<uint16_t *>(ws.y);
    p.T = T;
    p.P = T * k;
    p.shared = shared ? 1 : 0;
    p.status = ws.status;
    p.ovf = ws.ovf;
    return p;
}

}  // namespace

int launch_gather(const DeviceWeights &w, const Workspace &ws, const uint16_t *x, int T, int k, int gemm_min,
                  bool shared, void *stream) {
    const int P = T * k;
    const int blocks = std::min((T + 7) / 8, sm_count_tc() * 4);  // a warp per token, 8 tokens per CTA
    return launch_pdl(gather_kernel, dim3(blocks), dim3(256), 0, static_cast<cudaStream_t>(stream), x,
                      static_cast<const int32_t *>(ws.inv), static_cast<const int32_t *>(ws.topk_idx),
                      static_cast<const int32_t *>(ws.counts), static_cast<const uint8_t *>(w.tc_ok), gemm_min,
                      k, w.D, P, T, shared ? 1 : 0, ws.x16, ws.ovf, w.E);
}

int launch_producer_dump(const DeviceWeights &w, const uint8_t *grid, int expert, int matrix, uint16_t *dst16,
                         void *stream) {
    const bool down = matrix == DS4MOE_DOWN;
    const int rows = down ? w.D : w.F, cols = down ? w.F : w.D;
    dim3 g(rows / BM, cols / BK);
    producer_dump_kernel<<<g, kProducers, 0, static_cast<cudaStream_t>(stream)>>>(w, grid, expert, matrix, dst16);
    return static_cast<int>(cudaGetLastError());
}

int launch_gemm_up(const DeviceWeights &w, const Workspace &ws, const void *tmap_x16, int T, int k, bool shared,
                   bool pairs, void *stream) {
    return launch_gemm<UP>(*static_cast<const TokenMaps *>(tmap_x16), make_params(w, ws, T, k, shared), pairs,
                           static_cast<cudaStream_t>(stream));
}

int launch_gemm_down(const DeviceWeights &w, const Workspace &ws, const void *tmap_h16, int T, int k, bool shared,
                     bool pairs, void *stream) {
    return launch_gemm<DOWN>(*static_cast<const TokenMaps *>(tmap_h16), make_params(w, ws, T, k, shared), pairs,
                             static_cast<cudaStream_t>(stream));
}

// Tensor maps of an fp16 token operand [rows][cols] (row-major, SWIZZLE_128B): boxes of 64
// columns and 16, 32, 64, 128, 256 rows, written to maps_out (kTokenBoxes maps of 128 bytes).
int encode_token_maps(void *maps_out, void *base, int rows, int cols) {
    for (int i = 0; i < kTokenBoxes; i++)
        if (encode_token_map(static_cast<CUtensorMap *>(maps_out) + i, base, rows, cols, 16 << i)) return 1;
    return 0;
}

// One tensor map: 64 x box_rows boxes.
int encode_token_map(void *map_out, void *base, int rows, int cols, int box_rows) {
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
    const cuuint32_t box[2] = {BK, static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = encode(static_cast<CUtensorMap *>(map_out), CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, base, dims,
                              strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? 0 : 1;
}

}  // namespace ds4moe
