/*
 * oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 CPU restatement of the routed-MoE expert FFN over 2-bit experts:
 * the block formats, their quantisers and dequantisers, top-k routing and the stable
 * grouping of (token, slot) pairs by expert. The FFN itself is in oracle/moe.py (numpy fp64).
 * Only tests, the smoke check and the CPU-baseline leg of the benchmark may load this
 * file's library; the product path never does, and this file shares no code with it.
 *
 * Sources. "DwarfStar" (the ds4 README), section "模型权重": only the routed experts are
 * quantised, up/gate to IQ2_XXS and down to Q2_K; shared expert, projections and router
 * stay unquantised. "DwarfStar 深度解析" §3.4.3 draws the same split. The pages name the
 * formats but print no table; the byte layouts, the grid and the quantisers here are the
 * library's fixed readings (every such choice is a reading, not a page fact).
 *
 * Numerics. Every decision is an fp64 operation in the written order. Build with
 * -ffp-contract=off so that no multiply-add is fused.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ binary16 <-> fp64 */

/* IEEE-754 binary16 to double, exact. */
double or_half_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int m = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24); /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25); /* (1 + m/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* double to binary16, round half to even, subnormals kept, overflow to inf. */
uint16_t or_double_to_half(double x) {
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (isnan(x)) return 0x7e00;
    if (a >= 65520.0) return sign | 0x7c00; /* 65520 is the tie between 65504 and 2^16 */
    if (a < ldexp(1.0, -14)) {              /* subnormal range, quantum 2^-24 */
        double q = nearbyint(a * 16777216.0);
        return sign | (uint16_t)q; /* q == 1024 is the smallest normal, same bits */
    }
    int e;
    double f = frexp(a, &e);             /* a = f * 2^e, f in [0.5, 1) */
    double M = nearbyint(ldexp(f, 11));  /* 11-bit significand in [1024, 2048] */
    if (M == 2048.0) {
        M = 1024.0;
        e += 1;
    }
    int E = e - 1 + 15;
    if (E >= 31) return sign | 0x7c00;
    return sign | (uint16_t)(E << 10) | (uint16_t)((int)M - 1024);
}

/* ------------------------------------------------------------------ the IQ2 grid */

#define OR_IQ2_GRID_SEED 0x6473346D6F654951ULL

/* splitmix64 (Steele, Lea, Flood 2014): add the golden-gamma, then two xor-shift-multiply
 * rounds and a final xor-shift. */
uint64_t or_splitmix64_next(uint64_t *state) {
    uint64_t z = (*state += 0x9E3779B97F4A7C15ULL);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* Grid of 256 entries x 8 magnitudes: entry 0 all ones, then distinct draws in order. */
void or_iq2_grid(uint8_t grid[256 * 8]) {
    uint64_t st = OR_IQ2_GRID_SEED;
    for (int i = 0; i < 8; i++) grid[i] = 1;
    int n = 1;
    while (n < 256) {
        uint64_t r = or_splitmix64_next(&st);
        uint8_t cand[8];
        for (int i = 0; i < 8; i++) cand[i] = (uint8_t)(2 * ((r >> (2 * i)) & 3) + 1);
        int dup = 0;
        for (int m = 0; m < n && !dup; m++)
            if (memcmp(grid + 8 * m, cand, 8) == 0) dup = 1;
        if (!dup) {
            memcpy(grid + 8 * n, cand, 8);
            n++;
        }
    }
}

/* ------------------------------------------------------------------ Q2_K-style block */

static double clampd(double v, double lo, double hi) { return v < lo ? lo : (v > hi ? hi : v); }

/* Quantise 256 weights into one 84-byte block. Returns 0, or -1 on non-finite input or an
 * fp16 overflow of d/dmin. */
int or_q2k_quantize_block(const float *w, uint8_t *out) {
    double a[16], b[16];
    for (int i = 0; i < 256; i++)
        if (!isfinite(w[i])) return -1;
    double amax_a = 0.0, amax_b = 0.0;
    for (int j = 0; j < 16; j++) {
        double mn = w[16 * j], mx = w[16 * j];
        for (int i = 1; i < 16; i++) {
            double v = w[16 * j + i];
            if (v < mn) mn = v;
            if (v > mx) mx = v;
        }
        double lo = mn < 0.0 ? mn : 0.0;
        double hi = mx > lo ? mx : lo;
        a[j] = (hi - lo) / 3.0;
        b[j] = 0.0 - lo;
        if (a[j] > amax_a) amax_a = a[j];
        if (b[j] > amax_b) amax_b = b[j];
    }
    uint16_t dh = or_double_to_half(amax_a / 15.0);
    uint16_t mh = or_double_to_half(amax_b / 15.0);
    if (((dh >> 10) & 31) == 31 || ((mh >> 10) & 31) == 31) return -1;
    double d = or_half_to_double(dh), dmin = or_half_to_double(mh);
    memset(out, 0, 84);
    for (int j = 0; j < 16; j++) {
        int sc = d > 0.0 ? (int)clampd(nearbyint(a[j] / d), 0.0, 15.0) : 0;
        int m = dmin > 0.0 ? (int)clampd(nearbyint(b[j] / dmin), 0.0, 15.0) : 0;
        out[j] = (uint8_t)(sc | (m << 4));
        double den = d * (double)sc;
        double off = dmin * (double)m;
        for (int i = 0; i < 16; i++) {
            int k = 16 * j + i;
            int q = den > 0.0 ? (int)clampd(nearbyint(((double)w[k] + off) / den), 0.0, 3.0) : 0;
            out[16 + k / 4] |= (uint8_t)(q << (2 * (k % 4)));
        }
    }
    out[80] = (uint8_t)(dh & 0xff);
    out[81] = (uint8_t)(dh >> 8);
    out[82] = (uint8_t)(mh & 0xff);
    out[83] = (uint8_t)(mh >> 8);
    return 0;
}

/* One block back to 256 fp32 values: w = d*sc*q - dmin*m, rounded once to fp32. */
void or_q2k_dequant_block(const uint8_t *in, float *out) {
    double d = or_half_to_double((uint16_t)(in[80] | (in[81] << 8)));
    double dmin = or_half_to_double((uint16_t)(in[82] | (in[83] << 8)));
    for (int k = 0; k < 256; k++) {
        int j = k / 16;
        int sc = in[j] & 15, m = in[j] >> 4;
        int q = (in[16 + k / 4] >> (2 * (k % 4))) & 3;
        out[k] = (float)(d * (double)sc * (double)q - dmin * (double)m);
    }
}

/* ------------------------------------------------------------------ Q4_K-style block */

/* The 6-bit scale and min of sub-block j of a 144-byte block. */
static void q4k_scale_min(const uint8_t *blk, int j, int *sc, int *m) {
    int lo = blk[4 + j], hi = (blk[12 + j / 2] >> (4 * (j % 2))) & 15;
    *sc = (lo & 15) | ((hi & 3) << 4);
    *m = (lo >> 4) | ((hi >> 2) << 4);
}

/* Quantise 256 weights into one 144-byte Q4_K-style block (the 4-bit variant's layout). Returns 0, or -1 on
 * non-finite input or an fp16 overflow of d/dmin. */
int or_q4k_quantize_block(const float *w, uint8_t *out) {
    double a[8], b[8];
    for (int i = 0; i < 256; i++)
        if (!isfinite(w[i])) return -1;
    double amax_a = 0.0, amax_b = 0.0;
    for (int j = 0; j < 8; j++) {
        double mn = w[32 * j], mx = w[32 * j];
        for (int i = 1; i < 32; i++) {
            double v = w[32 * j + i];
            if (v < mn) mn = v;
            if (v > mx) mx = v;
        }
        double lo = mn < 0.0 ? mn : 0.0;
        double hi = mx > lo ? mx : lo;
        a[j] = (hi - lo) / 15.0;
        b[j] = 0.0 - lo;
        if (a[j] > amax_a) amax_a = a[j];
        if (b[j] > amax_b) amax_b = b[j];
    }
    uint16_t dh = or_double_to_half(amax_a / 63.0);
    uint16_t mh = or_double_to_half(amax_b / 63.0);
    if (((dh >> 10) & 31) == 31 || ((mh >> 10) & 31) == 31) return -1;
    double d = or_half_to_double(dh), dmin = or_half_to_double(mh);
    memset(out, 0, 144);
    out[0] = (uint8_t)(dh & 0xff);
    out[1] = (uint8_t)(dh >> 8);
    out[2] = (uint8_t)(mh & 0xff);
    out[3] = (uint8_t)(mh >> 8);
    for (int j = 0; j < 8; j++) {
        int sc = d > 0.0 ? (int)clampd(nearbyint(a[j] / d), 0.0, 63.0) : 0;
        int m = dmin > 0.0 ? (int)clampd(nearbyint(b[j] / dmin), 0.0, 63.0) : 0;
        out[4 + j] = (uint8_t)((sc & 15) | ((m & 15) << 4));
        out[12 + j / 2] |= (uint8_t)(((sc >> 4) | ((m >> 4) << 2)) << (4 * (j % 2)));
        double den = d * (double)sc;
        double off = dmin * (double)m;
        for (int i = 0; i < 32; i++) {
            int k = 32 * j + i;
            int q = den > 0.0 ? (int)clampd(nearbyint(((double)w[k] + off) / den), 0.0, 15.0) : 0;
            out[16 + k / 2] |= (uint8_t)(q << (4 * (k % 2)));
        }
    }
    return 0;
}

/* One block back to 256 fp32 values: w = d*sc*q - dmin*m, rounded once to fp32. */
void or_q4k_dequant_block(const uint8_t *in, float *out) {
    double d = or_half_to_double((uint16_t)(in[0] | (in[1] << 8)));
    double dmin = or_half_to_double((uint16_t)(in[2] | (in[3] << 8)));
    for (int k = 0; k < 256; k++) {
        int sc, m;
        q4k_scale_min(in, k / 32, &sc, &m);
        int q = (in[16 + k / 2] >> (4 * (k % 2))) & 15;
        out[k] = (float)(d * (double)sc * (double)q - dmin * (double)m);
    }
}

/* ------------------------------------------------------------------ IQ2-style block */

int or_iq2_quantize_block(const float *w, const uint8_t *grid, uint8_t *out) {
    double amax = 0.0;
    for (int i = 0; i < 256; i++) {
        if (!isfinite(w[i])) return -1;
        double v = fabs((double)w[i]);
        if (v > amax) amax = v;
    }
    uint16_t dh = or_double_to_half(amax / 7.0);
    if (((dh >> 10) & 31) == 31) return -1;
    memset(out, 0, 66);
    out[0] = (uint8_t)(dh & 0xff);
    out[1] = (uint8_t)(dh >> 8);
    double d = or_half_to_double(dh);
    if (d == 0.0) return 0;

    double nrm[256];
    for (int e = 0; e < 256; e++) {
        double n = 0.0;
        for (int i = 0; i < 8; i++) n += (double)grid[8 * e + i] * (double)grid[8 * e + i];
        nrm[e] = n;
    }
    for (int j = 0; j < 8; j++) {
        double a[4][8];
        uint32_t signs = 0;
        /* signs with even parity per group */
        for (int g = 0; g < 4; g++) {
            const float *wg = w + 32 * j + 8 * g;
            int neg[8], nneg = 0;
            for (int i = 0; i < 8; i++) {
                neg[i] = wg[i] < 0.0f;
                nneg += neg[i];
            }
            if (nneg & 1) {
                int im = 0;
                for (int i = 1; i < 8; i++)
                    if (fabs((double)wg[i]) < fabs((double)wg[im])) im = i;
                neg[im] = !neg[im];
            }
            for (int i = 0; i < 8; i++) a[g][i] = neg[i] ? -(double)wg[i] : (double)wg[i];
            for (int i = 0; i < 7; i++)
                if (neg[i]) signs |= 1u << (7 * g + i);
        }
        /* p_e = <a, G_e> in index order, per group */
        double p[4][256];
        for (int g = 0; g < 4; g++)
            for (int e = 0; e < 256; e++) {
                double s = 0.0;
                for (int i = 0; i < 8; i++) s += a[g][i] * (double)grid[8 * e + i];
                p[g][e] = s;
            }
        double best_cost = INFINITY;
        int best_s = 0, best_idx[4] = {0, 0, 0, 0};
        for (int s = 0; s < 16; s++) {
            double c = d * (double)(s + 1) / 16.0;
            double cost = 0.0;
            int idx[4];
            for (int g = 0; g < 4; g++) {
                double bestE = INFINITY;
                int bi = 0;
                for (int e = 0; e < 256; e++) {
                    double E = c * nrm[e] - 2.0 * p[g][e];
                    if (E < bestE) {
                        bestE = E;
                        bi = e;
                    }
                }
                idx[g] = bi;
                cost += c * bestE;
            }
            if (cost < best_cost) {
                best_cost = cost;
                best_s = s;
                for (int g = 0; g < 4; g++) best_idx[g] = idx[g];
            }
        }
        uint8_t *sb = out + 2 + 8 * j;
        for (int g = 0; g < 4; g++) sb[g] = (uint8_t)best_idx[g];
        uint32_t u = signs | ((uint32_t)best_s << 28);
        sb[4] = (uint8_t)(u & 0xff);
        sb[5] = (uint8_t)((u >> 8) & 0xff);
        sb[6] = (uint8_t)((u >> 16) & 0xff);
        sb[7] = (uint8_t)(u >> 24);
    }
    return 0;
}

/* One block back to 256 fp32 values: w = d*(s+1)/16*G[idx][i]*(+-1), exact in fp32. */
void or_iq2_dequant_block(const uint8_t *in, const uint8_t *grid, float *out) {
    double d = or_half_to_double((uint16_t)(in[0] | (in[1] << 8)));
    for (int j = 0; j < 8; j++) {
        const uint8_t *sb = in + 2 + 8 * j;
        uint32_t u = (uint32_t)sb[4] | ((uint32_t)sb[5] << 8) | ((uint32_t)sb[6] << 16) |
                     ((uint32_t)sb[7] << 24);
        int s = (int)(u >> 28);
        for (int g = 0; g < 4; g++) {
            uint32_t s7 = (u >> (7 * g)) & 127;
            int par = 0;
            for (int i = 0; i < 7; i++) par ^= (int)((s7 >> i) & 1);
            for (int i = 0; i < 8; i++) {
                int neg = i < 7 ? (int)((s7 >> i) & 1) : par;
                double v = d * (double)(s + 1) / 16.0 * (double)grid[8 * sb[g] + i];
                out[32 * j + 8 * g + i] = (float)(neg ? -v : v);
            }
        }
    }
}

/* ------------------------------------------------------------------ matrices */

int or_q2k_quantize(const float *w, int64_t rows, int64_t cols, uint8_t *dst) {
    int64_t nb = cols / 256;
    for (int64_t r = 0; r < rows; r++)
        for (int64_t b = 0; b < nb; b++)
            if (or_q2k_quantize_block(w + r * cols + 256 * b, dst + (r * nb + b) * 84)) return -1;
    return 0;
}

int or_iq2_quantize(const float *w, int64_t rows, int64_t cols, const uint8_t *grid, uint8_t *dst) {
    int64_t nb = cols / 256;
    for (int64_t r = 0; r < rows; r++)
        for (int64_t b = 0; b < nb; b++)
            if (or_iq2_quantize_block(w + r * cols + 256 * b, grid, dst + (r * nb + b) * 66))
                return -1;
    return 0;
}

int or_q4k_quantize(const float *w, int64_t rows, int64_t cols, uint8_t *dst) {
    int64_t nb = cols / 256;
    for (int64_t r = 0; r < rows; r++)
        for (int64_t b = 0; b < nb; b++)
            if (or_q4k_quantize_block(w + r * cols + 256 * b, dst + (r * nb + b) * 144)) return -1;
    return 0;
}

void or_q4k_dequant(const uint8_t *src, int64_t rows, int64_t cols, float *dst) {
    int64_t nb = cols / 256;
    for (int64_t r = 0; r < rows; r++)
        for (int64_t b = 0; b < nb; b++) or_q4k_dequant_block(src + (r * nb + b) * 144, dst + r * cols + 256 * b);
}

void or_q2k_dequant(const uint8_t *src, int64_t rows, int64_t cols, float *dst) {
    int64_t nb = cols / 256;
    for (int64_t r = 0; r < rows; r++)
        for (int64_t b = 0; b < nb; b++)
            or_q2k_dequant_block(src + (r * nb + b) * 84, dst + r * cols + 256 * b);
}

void or_iq2_dequant(const uint8_t *src, int64_t rows, int64_t cols, const uint8_t *grid, float *dst) {
    int64_t nb = cols / 256;
    for (int64_t r = 0; r < rows; r++)
        for (int64_t b = 0; b < nb; b++)
            or_iq2_dequant_block(src + (r * nb + b) * 66, grid, dst + r * cols + 256 * b);
}

/* ------------------------------------------------------------------ routing */

/* Routing ("DwarfStar 深度解析" §2.1: every token picks its experts from the router's logits).
 * Readings of this library, where the pages are silent:
 *   - order: logit descending, ties to the lower expert index; a NaN logit counts as -inf;
 *   - gate weights over the k selected logits v_0 >= ... >= v_{k-1} (NaN taken as -inf):
 *     mode 0 (softmax) g_s = exp(v_s - v_0) / sum_j exp(v_j - v_0), where a term with v_s equal to
 *     v_0 counts as exp(0) = 1 also when both are infinite (the limit of equal logits): an all -inf
 *     selection gets 1/k each, and a +inf logit takes the weight from every finite one;
 *     mode 1 (sigmoid) g_s = sigmoid(v_s) / sum_j sigmoid(v_j), evaluated as the mode-0 rule over
 *     log sigmoid(v) = min(v, 0) - log1p(exp(-|v|)) (the same ratio, with no underflow to 0/0). */
static double route_key(float v) { return isnan(v) ? -INFINITY : (double)v; }

/* 1 if expert a is ranked before expert b in the logits l of one token. */
static int route_before(const float *l, int a, int b) {
    const double ka = route_key(l[a]), kb = route_key(l[b]);
    if (ka != kb) return ka > kb;
    return a < b;
}

static double log_sigmoid(double v) { return fmin(v, 0.0) - log1p(exp(-fabs(v))); }

/* exp(v - top), with exp(0) = 1 where v equals top (infinities included). */
static double gate_term(double v, double top) { return v == top ? 1.0 : exp(v - top); }

/* Top-k per token and its gate weights: idx [T,k] and g [T,k] in the selection order. */
void or_route(const float *logits, int T, int E, int k, int mode, int32_t *idx, double *g) {
    int *order = (int *)malloc(sizeof(int) * (size_t)E);
    double *v = (double *)malloc(sizeof(double) * (size_t)k);
    for (int t = 0; t < T; t++) {
        const float *l = logits + (int64_t)t * E;
        /* insertion sort of the expert indices by route_before */
        for (int e = 0; e < E; e++) {
            int pos = e;
            while (pos > 0 && route_before(l, e, order[pos - 1])) {
                order[pos] = order[pos - 1];
                pos--;
            }
            order[pos] = e;
        }
        for (int s = 0; s < k; s++) {
            v[s] = route_key(l[order[s]]);
            if (mode != 0) v[s] = log_sigmoid(v[s]);
        }
        double den = 0.0;
        for (int s = 0; s < k; s++) den += gate_term(v[s], v[0]);
        for (int s = 0; s < k; s++) {
            idx[(int64_t)t * k + s] = order[s];
            g[(int64_t)t * k + s] = gate_term(v[s], v[0]) / den;
        }
    }
    free(v);
    free(order);
}

/* Counting sort of the T*k pairs by expert, stable in (token, slot) order.
 * counts[E], offsets[E+1] (exclusive scan), perm[P] = pair id t*k+s at its grouped
 * position, inv[P] = grouped position of pair t*k+s. */
void or_permute(const int32_t *idx, int T, int k, int E, int32_t *counts, int32_t *offsets,
                int32_t *perm, int32_t *inv) {
    int64_t P = (int64_t)T * k;
    for (int e = 0; e < E; e++) counts[e] = 0;
    for (int64_t p = 0; p < P; p++) counts[idx[p]]++;
    offsets[0] = 0;
    for (int e = 0; e < E; e++) offsets[e + 1] = offsets[e] + counts[e];
    int32_t *cursor = (int32_t *)malloc(sizeof(int32_t) * (size_t)E);
    for (int e = 0; e < E; e++) cursor[e] = offsets[e];
    for (int64_t p = 0; p < P; p++) {
        int e = idx[p];
        int32_t pos = cursor[e]++;
        perm[pos] = (int32_t)p;
        inv[p] = pos;
    }
    free(cursor);
}
