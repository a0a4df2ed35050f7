// Host side of the library: status strings, the IQ2-style grid, binary16 rounding, the
// two quantisers and host dequantisers. No CUDA here.
//
// The formats and quantisers are the library's own fixed layouts and rules (the pages --
// "DwarfStar" README, "模型权重" -- name IQ2_XXS for up/gate and Q2_K for down but print no
// layout). Every floating-point step follows the quantisers' written order with no fused
// multiply-add (this file is compiled with -ffp-contract=off), so the bytes are reproducible
// across machines.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

#include "../../include/ds4moe.h"
#include "internal.h"

namespace {

// ------------------------------------------------------------------ binary16

// binary16 bits -> double (exact).
double f16_value(uint16_t h) {
    const int e = (h >> 10) & 0x1f;
    const int frac = h & 0x3ff;
    double mag;
    if (e == 0x1f) {
        mag = frac ? std::nan("") : HUGE_VAL;
    } else if (e == 0) {
        mag = std::ldexp(static_cast<double>(frac), -24);
    } else {
        mag = std::ldexp(static_cast<double>(frac | 0x400), e - 25);
    }
    return (h & 0x8000) ? -mag : mag;
}

// double -> binary16, nearest with ties to even, working on the double's bit pattern.
uint16_t f16_round(double x) {
    uint64_t bits;
    std::memcpy(&bits, &x, sizeof bits);
    const uint16_t sign = static_cast<uint16_t>((bits >> 48) & 0x8000u);
    const uint64_t mag = bits & 0x7fffffffffffffffull;
    const int bexp = static_cast<int>(mag >> 52);
    if (bexp == 0x7ff) return (mag & 0xfffffffffffffull) ? 0x7e00 : static_cast<uint16_t>(sign | 0x7c00);
    if (bexp == 0) return sign;  // double subnormals are far below half's range
    const int e = bexp - 1023;
    if (e > 15) return static_cast<uint16_t>(sign | 0x7c00);
    const uint64_t sig = (mag & 0xfffffffffffffull) | (1ull << 52);  // 53-bit significand
    // keep 11 bits for normals (e >= -14); fewer for subnormals (quantum 2^-24)
    int drop = 42;
    if (e < -14) drop += (-14 - e);
    if (drop > 53) return sign;  // below half of the smallest subnormal
    uint64_t q = sig >> drop;
    const uint64_t rem = sig & ((1ull << drop) - 1);
    const uint64_t halfway = 1ull << (drop - 1);
    if (rem > halfway || (rem == halfway && (q & 1))) q++;
    uint32_t h;
    if (e >= -14) {
        h = static_cast<uint32_t>((e + 15) << 10) + static_cast<uint32_t>(q - 1024);  // carry bumps the exponent
    } else {
        h = static_cast<uint32_t>(q);  // q == 1024 is the smallest normal's bit pattern
    }
    if (h >= 0x7c00) return static_cast<uint16_t>(sign | 0x7c00);
    return static_cast<uint16_t>(sign | h);
}

bool f16_finite(uint16_t h) { return ((h >> 10) & 0x1f) != 0x1f; }

inline uint16_t rd16(const uint8_t *p) { return static_cast<uint16_t>(p[0] | (p[1] << 8)); }
inline void wr16(uint8_t *p, uint16_t v) {
    p[0] = static_cast<uint8_t>(v);
    p[1] = static_cast<uint8_t>(v >> 8);
}
inline uint32_t rd32(const uint8_t *p) {
    return static_cast<uint32_t>(p[0]) | (static_cast<uint32_t>(p[1]) << 8) |
           (static_cast<uint32_t>(p[2]) << 16) | (static_cast<uint32_t>(p[3]) << 24);
}
inline void wr32(uint8_t *p, uint32_t v) {
    for (int i = 0; i < 4; i++) p[i] = static_cast<uint8_t>(v >> (8 * i));
}

double rne(double v) { return std::nearbyint(v); }  // default rounding mode: to nearest, ties even
double clip(double v, double lo, double hi) { return std::min(std::max(v, lo), hi); }

// ------------------------------------------------------------------ the grid

struct Grid {
    uint8_t mag[256][8];
    double gt[8][256];  // transposed as doubles, for the search
    double norm2[256];
    Grid() {
        uint64_t state = 0x6473346D6F654951ull;  // the grid's fixed seed
        auto next = [&state]() {
            // splitmix64: Weyl step by the 64-bit golden ratio, then the variant-13 mix
            state += 0x9E3779B97F4A7C15ull;
            uint64_t z = state;
            z ^= z >> 30;
            z *= 0xBF58476D1CE4E5B9ull;
            z ^= z >> 27;
            z *= 0x94D049BB133111EBull;
            z ^= z >> 31;
            return z;
        };
        std::memset(mag, 1, sizeof mag[0]);
        int have = 1;
        while (have < 256) {
            const uint64_t r = next();
            uint8_t v[8];
            for (int i = 0; i < 8; i++) v[i] = static_cast<uint8_t>(1 + 2 * ((r >> (2 * i)) & 3u));
            bool fresh = true;
            for (int e = 0; e < have && fresh; e++) fresh = std::memcmp(mag[e], v, 8) != 0;
            if (fresh) std::memcpy(mag[have++], v, 8);
        }
        for (int e = 0; e < 256; e++) {
            double n = 0.0;
            for (int i = 0; i < 8; i++) {
                gt[i][e] = mag[e][i];
                n += gt[i][e] * gt[i][e];
            }
            norm2[e] = n;
        }
    }
};

const Grid &grid() {
    static const Grid g;
    return g;
}

// ------------------------------------------------------------------ Q2_K-style

bool q2k_block(const float *w, uint8_t *blk) {
    double step[16], off[16];
    double top_step = 0.0, top_off = 0.0;
    for (int j = 0; j < 16; j++) {
        double lo = w[16 * j], hi = w[16 * j];
        for (int i = 0; i < 16; i++) {
            const double v = w[16 * j + i];
            if (!std::isfinite(v)) return false;
            lo = v < lo ? v : lo;
            hi = v > hi ? v : hi;
        }
        lo = lo < 0.0 ? lo : 0.0;
        hi = hi > lo ? hi : lo;
        step[j] = (hi - lo) / 3.0;
        off[j] = 0.0 - lo;
        top_step = step[j] > top_step ? step[j] : top_step;
        top_off = off[j] > top_off ? off[j] : top_off;
    }
    const uint16_t dbits = f16_round(top_step / 15.0);
    const uint16_t mbits = f16_round(top_off / 15.0);
    if (!f16_finite(dbits) || !f16_finite(mbits)) return false;
    const double d = f16_value(dbits), dmin = f16_value(mbits);
    std::memset(blk, 0, 84);
    for (int j = 0; j < 16; j++) {
        const int sc = d > 0.0 ? static_cast<int>(clip(rne(step[j] / d), 0.0, 15.0)) : 0;
        const int mn = dmin > 0.0 ? static_cast<int>(clip(rne(off[j] / dmin), 0.0, 15.0)) : 0;
        blk[j] = static_cast<uint8_t>(sc | (mn << 4));
        const double den = d * sc;
        const double shift = dmin * mn;
        for (int i = 0; i < 16; i++) {
            const int n = 16 * j + i;
            int q = 0;
            if (den > 0.0) q = static_cast<int>(clip(rne((static_cast<double>(w[n]) + shift) / den), 0.0, 3.0));
            blk[16 + n / 4] |= static_cast<uint8_t>(q << (2 * (n & 3)));
        }
    }
    wr16(blk + 80, dbits);
    wr16(blk + 82, mbits);
    return true;
}

void q2k_block_values(const uint8_t *blk, float *w) {
    const double d = f16_value(rd16(blk + 80)), dmin = f16_value(rd16(blk + 82));
    for (int n = 0; n < 256; n++) {
        const int sc = blk[n / 16] & 15, mn = blk[n / 16] >> 4;
        const int q = (blk[16 + n / 4] >> (2 * (n & 3))) & 3;
        const double a = d * sc * q;  // exact
        const double b = dmin * mn;   // exact
        w[n] = static_cast<float>(a - b);
    }
}

// ------------------------------------------------------------------ Q4_K-style (the 4-bit variant)

// Sub-block j's 6-bit scale and min: low nibbles at byte 4 + j, the two high bits of each at
// byte 12 + j/2, nibble j % 2 (scale bits 0-1, min bits 2-3).
inline void q4k_sm(const uint8_t *blk, int j, int *sc, int *mn) {
    const int low = blk[4 + j], high = (blk[12 + j / 2] >> (4 * (j & 1))) & 15;
    *sc = (low & 15) | ((high & 3) << 4);
    *mn = (low >> 4) | ((high >> 2) << 4);
}

bool q4k_block(const float *w, uint8_t *blk) {
    double step[8], off[8];
    double top_step = 0.0, top_off = 0.0;
    for (int j = 0; j < 8; j++) {
        double lo = w[32 * j], hi = w[32 * j];
        for (int i = 0; i < 32; i++) {
            const double v = w[32 * j + i];
            if (!std::isfinite(v)) return false;
            lo = v < lo ? v : lo;
            hi = v > hi ? v : hi;
        }
        lo = lo < 0.0 ? lo : 0.0;
        hi = hi > lo ? hi : lo;
        step[j] = (hi - lo) / 15.0;
        off[j] = 0.0 - lo;
        top_step = step[j] > top_step ? step[j] : top_step;
        top_off = off[j] > top_off ? off[j] : top_off;
    }
    const uint16_t dbits = f16_round(top_step / 63.0);
    const uint16_t mbits = f16_round(top_off / 63.0);
    if (!f16_finite(dbits) || !f16_finite(mbits)) return false;
    const double d = f16_value(dbits), dmin = f16_value(mbits);
    std::memset(blk, 0, 144);
    wr16(blk, dbits);
    wr16(blk + 2, mbits);
    for (int j = 0; j < 8; j++) {
        const int sc = d > 0.0 ? static_cast<int>(clip(rne(step[j] / d), 0.0, 63.0)) : 0;
        const int mn = dmin > 0.0 ? static_cast<int>(clip(rne(off[j] / dmin), 0.0, 63.0)) : 0;
        blk[4 + j] = static_cast<uint8_t>((sc & 15) | ((mn & 15) << 4));
        blk[12 + j / 2] |= static_cast<uint8_t>(((sc >> 4) | ((mn >> 4) << 2)) << (4 * (j & 1)));
        const double den = d * sc;
        const double shift = dmin * mn;
        for (int i = 0; i < 32; i++) {
            const int n = 32 * j + i;
            int q = 0;
            if (den > 0.0) q = static_cast<int>(clip(rne((static_cast<double>(w[n]) + shift) / den), 0.0, 15.0));
            blk[16 + n / 2] |= static_cast<uint8_t>(q << (4 * (n & 1)));
        }
    }
    return true;
}

void q4k_block_values(const uint8_t *blk, float *w) {
    const double d = f16_value(rd16(blk)), dmin = f16_value(rd16(blk + 2));
    for (int n = 0; n < 256; n++) {
        int sc = 0, mn = 0;
        q4k_sm(blk, n / 32, &sc, &mn);
        const int q = (blk[16 + n / 2] >> (4 * (n & 1))) & 15;
        w[n] = static_cast<float>(d * sc * q - dmin * mn);  // both products exact, one rounding
    }
}

// ------------------------------------------------------------------ IQ2-style

bool iq2_block(const float *w, uint8_t *blk) {
    const Grid &G = grid();
    double amax = 0.0;
    for (int i = 0; i < 256; i++) {
        if (!std::isfinite(w[i])) return false;
        amax = std::max(amax, std::fabs(static_cast<double>(w[i])));
    }
    const uint16_t dbits = f16_round(amax / 7.0);
    if (!f16_finite(dbits)) return false;
    std::memset(blk, 0, 66);
    wr16(blk, dbits);
    const double d = f16_value(dbits);
    if (d == 0.0) return true;

    alignas(64) double p[4][256];
    for (int sb = 0; sb < 8; sb++) {
        uint32_t word = 0;
        for (int g = 0; g < 4; g++) {
            const float *wg = w + 32 * sb + 8 * g;
            bool neg[8];
            int count = 0;
            for (int i = 0; i < 8; i++) count += (neg[i] = wg[i] < 0.0f);
            if (count & 1) {  // odd: flip the smallest magnitude (first on ties)
                int at = 0;
                for (int i = 1; i < 8; i++)
                    if (std::fabs(static_cast<double>(wg[i])) < std::fabs(static_cast<double>(wg[at]))) at = i;
                neg[at] = !neg[at];
            }
            double a[8];
            for (int i = 0; i < 8; i++) a[i] = neg[i] ? -static_cast<double>(wg[i]) : static_cast<double>(wg[i]);
            for (int i = 0; i < 7; i++) word |= static_cast<uint32_t>(neg[i]) << (7 * g + i);
            for (int e = 0; e < 256; e++) p[g][e] = a[0] * G.gt[0][e];
            for (int i = 1; i < 8; i++)
                for (int e = 0; e < 256; e++) p[g][e] = p[g][e] + a[i] * G.gt[i][e];
        }
        double best_cost = HUGE_VAL;
        int best_s = 0;
        int best_idx[4] = {0, 0, 0, 0};
        for (int s = 0; s < 16; s++) {
            const double c = d * (s + 1) / 16.0;
            double cost = 0.0;
            int pick[4];
            for (int g = 0; g < 4; g++) {
                double emin = HUGE_VAL;
                int at = 0;
                for (int e = 0; e < 256; e++) {
                    const double err = c * G.norm2[e] - 2.0 * p[g][e];
                    if (err < emin) {
                        emin = err;
                        at = e;
                    }
                }
                pick[g] = at;
                cost += c * emin;
            }
            if (cost < best_cost) {
                best_cost = cost;
                best_s = s;
                std::copy(pick, pick + 4, best_idx);
            }
        }
        uint8_t *q = blk + 2 + 8 * sb;
        for (int g = 0; g < 4; g++) q[g] = static_cast<uint8_t>(best_idx[g]);
        wr32(q + 4, word | (static_cast<uint32_t>(best_s) << 28));
    }
    return true;
}

void iq2_block_values(const uint8_t *blk, float *w) {
    const Grid &G = grid();
    const double d = f16_value(rd16(blk));
    for (int sb = 0; sb < 8; sb++) {
        const uint8_t *q = blk + 2 + 8 * sb;
        const uint32_t word = rd32(q + 4);
        const double scale = d * ((word >> 28) + 1) / 16.0;
        for (int g = 0; g < 4; g++) {
            const uint32_t s7 = (word >> (7 * g)) & 0x7f;
            uint32_t signs = s7 | ((static_cast<uint32_t>(__builtin_popcount(s7)) & 1u) << 7);
            for (int i = 0; i < 8; i++) {
                const double v = scale * G.mag[q[g]][i];
                w[32 * sb + 8 * g + i] = static_cast<float>(((signs >> i) & 1) ? -v : v);
            }
        }
    }
}

// Runs body(row) over rows on all host cores; returns false if any call did.
template <class F>
bool for_rows(int64_t rows, F body) {
    const unsigned hw = std::max(1u, std::thread::hardware_concurrency());
    const int64_t nthreads = std::min<int64_t>(hw, std::max<int64_t>(1, rows));
    std::vector<char> ok(static_cast<size_t>(nthreads), 1);
    auto run = [&](int64_t t) {
        for (int64_t r = t; r < rows; r += nthreads)
            if (!body(r)) {
                ok[static_cast<size_t>(t)] = 0;
                return;
            }
    };
    if (nthreads == 1) {
        run(0);
    } else {
        std::vector<std::thread> pool;
        pool.reserve(static_cast<size_t>(nthreads));
        for (int64_t t = 0; t < nthreads; t++) pool.emplace_back(run, t);
        for (auto &th : pool) th.join();
    }
    return std::all_of(ok.begin(), ok.end(), [](char c) { return c != 0; });
}

bool shape_ok(int64_t rows, int64_t cols) { return rows >= 0 && cols > 0 && cols % 256 == 0; }

}  // namespace

// ------------------------------------------------------------------ internal API

namespace ds4moe {

void host_grid(uint8_t out[2048]) { std::memcpy(out, grid().mag, 2048); }
bool host_f16_finite(uint16_t h) { return f16_finite(h); }
double host_f16_value(uint16_t h) { return f16_value(h); }

}  // namespace ds4moe

// ------------------------------------------------------------------ C ABI

extern "C" {

const char *ds4moe_strerror(int status) {
    switch (status) {
        case DS4MOE_OK: return "ok";
        case DS4MOE_EINVAL: return "invalid argument";
        case DS4MOE_ENOMEM: return "out of memory";
        case DS4MOE_ECUDA: return "CUDA runtime error";
        case DS4MOE_EBADDATA: return "input data rejected (non-finite value or scale)";
        case DS4MOE_ETIMEOUT: return "device-side wait timed out";
        case DS4MOE_EUNSUPPORTED: return "unsupported shape or device";
        case DS4MOE_ERANGE: return "value outside the fp16 range of the tensor-core path";
        case DS4MOE_ECAPACITY: return "a call touched more experts than the handle's slots";
        default: return "unknown status";
    }
}

size_t ds4moe_q2k_bytes(int64_t rows, int64_t cols) {
    return shape_ok(rows, cols) ? static_cast<size_t>(rows) * static_cast<size_t>(cols / 256) * 84u : 0u;
}

size_t ds4moe_q4k_bytes(int64_t rows, int64_t cols) {
    return shape_ok(rows, cols) ? static_cast<size_t>(rows) * static_cast<size_t>(cols / 256) * 144u : 0u;
}

int ds4moe_quantize_q4k(const float *w, int64_t rows, int64_t cols, void *dst, size_t dst_bytes) {
    if (!w || !dst || !shape_ok(rows, cols) || dst_bytes < ds4moe_q4k_bytes(rows, cols)) return DS4MOE_EINVAL;
    const int64_t nb = cols / 256;
    uint8_t *out = static_cast<uint8_t *>(dst);
    const bool ok = for_rows(rows, [&](int64_t r) {
        for (int64_t b = 0; b < nb; b++)
            if (!q4k_block(w + r * cols + 256 * b, out + (r * nb + b) * 144)) return false;
        return true;
    });
    return ok ? DS4MOE_OK : DS4MOE_EBADDATA;
}

int ds4moe_dequantize_q4k(const void *src, int64_t rows, int64_t cols, float *dst) {
    if (!src || !dst || !shape_ok(rows, cols)) return DS4MOE_EINVAL;
    const int64_t nb = cols / 256;
    const uint8_t *in = static_cast<const uint8_t *>(src);
    for_rows(rows, [&](int64_t r) {
        for (int64_t b = 0; b < nb; b++) q4k_block_values(in + (r * nb + b) * 144, dst + r * cols + 256 * b);
        return true;
    });
    return DS4MOE_OK;
}

size_t ds4moe_iq2_bytes(int64_t rows, int64_t cols) {
    return shape_ok(rows, cols) ? static_cast<size_t>(rows) * static_cast<size_t>(cols / 256) * 66u : 0u;
}

int ds4moe_iq2_grid(uint8_t *out) {
    if (!out) return DS4MOE_EINVAL;
    ds4moe::host_grid(out);
    return DS4MOE_OK;
}

int ds4moe_quantize_q2k(const float *w, int64_t rows, int64_t cols, void *dst, size_t dst_bytes) {
    if (!w || !dst || !shape_ok(rows, cols) || dst_bytes < ds4moe_q2k_bytes(rows, cols)) return DS4MOE_EINVAL;
    const int64_t nb = cols / 256;
    uint8_t *out = static_cast<uint8_t *>(dst);
    const bool ok = for_rows(rows, [&](int64_t r) {
        for (int64_t b = 0; b < nb; b++)
            if (!q2k_block(w + r * cols + 256 * b, out + (r * nb + b) * 84)) return false;
        return true;
    });
    return ok ? DS4MOE_OK : DS4MOE_EBADDATA;
}

int ds4moe_quantize_iq2(const float *w, int64_t rows, int64_t cols, void *dst, size_t dst_bytes) {
    if (!w || !dst || !shape_ok(rows, cols) || dst_bytes < ds4moe_iq2_bytes(rows, cols)) return DS4MOE_EINVAL;
    const int64_t nb = cols / 256;
    uint8_t *out = static_cast<uint8_t *>(dst);
    grid();  // build once before the threads start
    const bool ok = for_rows(rows, [&](int64_t r) {
        for (int64_t b = 0; b < nb; b++)
            if (!iq2_block(w + r * cols + 256 * b, out + (r * nb + b) * 66)) return false;
        return true;
    });
    return ok ? DS4MOE_OK : DS4MOE_EBADDATA;
}

int ds4moe_dequantize_q2k(const void *src, int64_t rows, int64_t cols, float *dst) {
    if (!src || !dst || !shape_ok(rows, cols)) return DS4MOE_EINVAL;
    const int64_t nb = cols / 256;
    const uint8_t *in = static_cast<const uint8_t *>(src);
    for_rows(rows, [&](int64_t r) {
        for (int64_t b = 0; b < nb; b++) q2k_block_values(in + (r * nb + b) * 84, dst + r * cols + 256 * b);
        return true;
    });
    return DS4MOE_OK;
}

int ds4moe_dequantize_iq2(const void *src, int64_t rows, int64_t cols, float *dst) {
    if (!src || !dst || !shape_ok(rows, cols)) return DS4MOE_EINVAL;
    const int64_t nb = cols / 256;
    const uint8_t *in = static_cast<const uint8_t *>(src);
    grid();
    for_rows(rows, [&](int64_t r) {
        for (int64_t b = 0; b < nb; b++) iq2_block_values(in + (r * nb + b) * 66, dst + r * cols + 256 * b);
        return true;
    });
    return DS4MOE_OK;
}

}  // extern "C"
