// Device helpers of the dp2a kernels (the fused single-token kernel and the small-group kernels):
// exact integer dot products of the 2-bit codes with int16 activations, the shared-memory lookup
// tables of the IQ2-style codebook and signs, and the mbarrier hand-shakes they share.
//
// IQ2-style group of 8 weights as nibbles: the codebook word of entry e holds, per element, m - 1
// (m in {1, 3, 5, 7}, so m - 1 is even), elements 2b in byte b's low nibble and 2b + 1 in its high
// nibble; the sign word of a 7-bit pattern s holds 0x9 (keep) or 0x7 (negate) per element, the 8th
// sign being the parity of the 7. Their XOR is, per nibble, the signed weight plus 8 with no carry
// between nibbles (m - 1 ^ 9 = m + 8, m - 1 ^ 7 = 8 - m), so one mask gives the even weights plus 8
// as bytes and another 16 x (the odd weights plus 8), ready for dp2a against int16 pairs.
#pragma once

#include "common.cuh"
#include "ptx.cuh"

namespace ds4moe {

// v rounded to the nearest integer (ties to even), for |v| <= 2^22, as the low bits of the result:
// adding 1.5 * 2^23 leaves the rounded integer in the mantissa (two full-rate operations).
__device__ __forceinline__ uint32_t round_to_int_bits(float v) {
    return static_cast<uint32_t>(__float_as_int(__fadd_rn(v, 12582912.0f)) - 0x4B400000);
}

// Exact int -> float for |v| < 2^22 with two full-rate operations (no conversion unit).
__device__ __forceinline__ float small_int_to_float(int v) { return __int_as_float(0x4B400000 + v) - 12582912.0f; }

// d = c + a.lo16 * b.byte0 + a.hi16 * b.byte1 (lo) or with bytes 2, 3 (hi): signed 16-bit a,
// unsigned bytes b.
__device__ __forceinline__ int dp2a_lo_su(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp2a.lo.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp2a_hi_su(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp2a.hi.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// The codebook word of a grid entry (its 8 magnitude bytes, elements 0..3 in g.x).
__device__ __forceinline__ uint32_t iq2_nibble_word(uint2 g) {
    const uint32_t lo = g.x - 0x01010101u, hi = g.y - 0x01010101u;  // bytes m - 1
    // bytes (e0, e1, e2, e3), (e4, e5, e6, e7) -> bytes (e0 | e1 << 4, e2 | e3 << 4, ...)
    const uint32_t ev = __byte_perm(lo, hi, 0x6420), od = __byte_perm(lo, hi, 0x7531);
    return ev | (od << 4);
}

// The sign word of a 7-bit stored sign pattern (the 8th sign is the parity of the 7): the 8 sign
// bits spread to one per nibble (bit e at 4 e), then 0x9 ^ 0xE = 0x7 where a sign is set.
__device__ __forceinline__ uint32_t iq2_sign_word(uint32_t s7) {
    uint32_t v = s7 | ((__popc(s7) & 1u) << 7);
    v = (v | (v << 12)) & 0x000F000Fu;  // signs 0-3 at bits 0-3, 4-7 at bits 16-19
    v = (v | (v << 6)) & 0x03030303u;   // two per byte
    v = (v | (v << 3)) & 0x11111111u;   // one per nibble
    return 0x99999999u ^ (v * 0xEu);
}

// The lookup table: 256 slots of 256 bytes. Slot e holds codebook word e in its first 128 bytes and
// sign word e (e < 128) in its second 128 bytes, one u32 replica per lane, so any index a lane
// looks up sits in that lane's own bank. Built by 16 warps (warp16 = 0..15): each word is computed
// once per warp (lane l < 16: codebook word of entry warp16 + 16 l, from its grid entry gown that
// the caller loaded early; lane 16 + j: sign word of pattern warp16 + 16 j) and handed to every lane
// by a shuffle.
__device__ __forceinline__ void iq2_table_store(uint8_t *tab, uint2 gown, int warp16, int lane) {
    const uint32_t mine = lane < 16 ? iq2_nibble_word(gown) : iq2_sign_word(static_cast<uint32_t>(warp16 + 16 * (lane & 7)));
#pragma unroll
    for (int j = 0; j < 16; j++)
        *reinterpret_cast<uint32_t *>(tab + (warp16 + 16 * j) * 256 + lane * 4) = __shfl_sync(0xffffffffu, mine, j);
#pragma unroll
    for (int j = 0; j < 8; j++)
        *reinterpret_cast<uint32_t *>(tab + (warp16 + 16 * j) * 256 + 128 + lane * 4) = __shfl_sync(0xffffffffu, mine, 16 + j);
}

// Byte offsets in the table of group g's codebook and sign words of a sub-block whose index word
// is qx and sign/scale word qy, for the lane with lane4 = 4 * lane.
__device__ __forceinline__ uint32_t iq2_cb_off(uint32_t qx, int g, uint32_t lane4) {
    return __byte_perm(lane4, qx, 0x1140u + 0x10u * g);  // lane4 | byte g of qx << 8
}
__device__ __forceinline__ uint32_t iq2_sg_off(uint32_t qy, int g, uint32_t lane4) {
    const uint32_t f = g == 0 ? (qy << 8) : g == 1 ? (qy << 1) : (qy >> (7 * g - 8));  // signs 7g..7g+6 at bit 8
    return (f & 0x7F00u) | lane4 | 128u;
}

// Sixteen Q2_K-style 2-bit codes (one u32: byte b holds weights 4b..4b+3) dotted with 16 int16 h
// stored as hp[2j] = (h_j, h_4+j), hp[2j+1] = (h_8+j, h_12+j).
__device__ __forceinline__ int q2k_idot(uint32_t qw, const uint32_t *hp) {
    int a = 0;  // one accumulation chain: the callers have several rows in flight
#pragma unroll
    for (int j = 0; j < 4; j++) {
        const int c = static_cast<int>((qw >> (2 * j)) & 0x03030303u);  // weights j, 4+j, 8+j, 12+j
        a = __dp2a_hi(static_cast<int>(hp[2 * j + 1]), c, __dp2a_lo(static_cast<int>(hp[2 * j]), c, a));
    }
    return a;
}

// Position of h element r (0..15) of a 16-column sub-block in the order q2k_idot reads it.
__device__ __forceinline__ int q2k_h_pos(int r) { return 4 * (r & 3) + (r >> 2); }

// Bounded wait with the common case (phase already complete) inline.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int *abort_flag, int *status) {
    return mbar_test(bar, parity) || mbar_wait(bar, parity, abort_flag, status);
}

__device__ __forceinline__ void bar_sync(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }

// Sums eight per-lane values over the warp; afterwards lane l holds the total of value (l >> 2) & 7.
__device__ __forceinline__ float reduce8(const float v[8], int lane) {
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
    float a[4], c[2];
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const float keep = b4 ? v[4 + i] : v[i], send = b4 ? v[i] : v[4 + i];
        a[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
#pragma unroll
    for (int i = 0; i < 2; i++) {
        const float keep = b3 ? a[2 + i] : a[i], send = b3 ? a[i] : a[2 + i];
        c[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
    float d = (b2 ? c[1] : c[0]) + __shfl_xor_sync(0xffffffffu, b2 ? c[0] : c[1], 4);
    d += __shfl_xor_sync(0xffffffffu, d, 2);
    d += __shfl_xor_sync(0xffffffffu, d, 1);
    return d;
}

}  // namespace ds4moe
