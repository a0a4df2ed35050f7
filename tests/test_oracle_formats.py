"""Pins for the oracle's number formats, grid and quantisers (CPU only).

Each test checks the oracle against something other than itself: numpy's float16
rounding, the published splitmix64 reference outputs, hand-built blocks with values worked
out by hand, blocks whose values lie exactly on the code grid (quantise -> dequantise is then
a fixed point), and brute-force searches written with numpy.
"""
import hashlib
import os
import re

import numpy as np
import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


# ---------------------------------------------------------------- binary16

def test_half_to_double_all_patterns_match_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_double_to_half_matches_numpy_rounding():
    rng = np.random.default_rng(7)
    xs = list(rng.standard_normal(3000) * np.exp(rng.uniform(-22, 12, 3000)))
    # exact ties between neighbouring binary16 values (normal and subnormal), both parities
    for m in [0, 1, 2, 3, 1022, 1023]:
        for e in [-24, -20, -14, -3, 0, 5, 14]:
            xs.append((1024 + m + 0.5) * 2.0 ** (e - 10))
    for m in [0, 1, 2, 3, 511, 1022]:
        xs.append((m + 0.5) * 2.0 ** -24)
    xs += [0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e6, -1e6, 2.0 ** -25, 2.0 ** -25 * 1.0001, 6e-8]
    for x in xs:
        with np.errstate(over="ignore"):
            ref = int(np.array([x], np.float64).astype(np.float16).view(np.uint16)[0])
        assert oracle.double_to_half(x) == ref, x


# ---------------------------------------------------------------- splitmix64 and the grid

def test_splitmix64_published_reference_outputs():
    # Reference outputs of splitmix64 for seed 1234567 (Vigna's reference implementation).
    assert oracle.splitmix64(1234567, 5) == [
        6457827717110365317, 3203168211198807973, 9817491932198370423,
        4593380528125082431, 16408922859458223821]


def test_grid_properties_and_golden():
    g = oracle.iq2_grid()
    assert g.shape == (256, 8)
    assert np.all(g[0] == 1)
    assert set(np.unique(g)) <= {1, 3, 5, 7}
    assert len({bytes(r) for r in g}) == 256
    sha = hashlib.sha256(g.tobytes()).hexdigest()
    fmt = open(os.path.join(ROOT, "FORMAT.md")).read()
    assert re.search(r"GRID_SHA256 = ([0-9a-f]{64})", fmt).group(1) == sha
    rows = [l.split() for l in open(os.path.join(HERE, "golden", "iq2_grid.txt")) if not l.startswith("#")]
    assert np.array_equal(np.array(rows, dtype=np.uint8), g)


def test_grid_entries_are_the_splitmix64_draws():
    # entry n>0 is the n-th distinct proposal m_i = 2*((r >> 2i) & 3) + 1 of the seeded stream
    draws = oracle.splitmix64(0x6473346D6F654951, 400)
    seen = [bytes([1] * 8)]
    for r in draws:
        v = bytes(2 * ((r >> (2 * i)) & 3) + 1 for i in range(8))
        if v not in seen:
            seen.append(v)
        if len(seen) == 256:
            break
    assert np.array_equal(np.frombuffer(b"".join(seen), np.uint8).reshape(256, 8), oracle.iq2_grid())


# ---------------------------------------------------------------- Q2_K-style blocks

def _half_bits(v):
    return int(np.array([v], np.float16).view(np.uint16)[0])


def test_q2k_dequant_hand_built_block():
    blk = np.zeros(84, np.uint8)
    blk[80:82] = np.array([_half_bits(1.0)], np.uint16).view(np.uint8)   # d = 1
    blk[82:84] = np.array([_half_bits(2.0)], np.uint16).view(np.uint8)   # dmin = 2
    blk[0] = 0x31           # sub-block 0: sc = 1, m = 3
    blk[1] = 0x0F           # sub-block 1: sc = 15, m = 0
    blk[16] = 0b11100100    # weights 0..3 have q = 0, 1, 2, 3
    blk[20] = 0b00000011    # weight 16 has q = 3, weights 17..19 q = 0
    w = oracle.dequant_q2k(blk, 1, 256)[0]
    assert list(w[:5]) == [-6.0, -5.0, -4.0, -3.0, -6.0]   # 1*1*q - 2*3
    assert list(w[16:18]) == [45.0, 0.0]                   # 1*15*3 - 0
    assert np.all(w[32:] == 0.0)                           # sc = m = 0 elsewhere


def _exact_q2k_block(rng):
    """A block whose fp32 values are exact and which the quantiser must reproduce."""
    while True:
        blk = np.zeros(84, np.uint8)
        d = np.float16(rng.uniform(2 ** -8, 2 ** -6))
        dmin = np.float16(rng.uniform(2 ** -8, 2 ** -6))
        sc = rng.integers(1, 16, 16)
        m = rng.integers(0, 16, 16)
        sc[rng.integers(16)] = 15
        m[rng.integers(16)] = 15
        q = rng.integers(0, 4, 256)
        for j in range(16):
            a, b = rng.choice(16, 2, replace=False)
            q[16 * j + a], q[16 * j + b] = 0, 3
        blk[:16] = sc | (m << 4)
        for k in range(256):
            blk[16 + k // 4] |= q[k] << (2 * (k % 4))
        blk[80:82] = np.array([d]).view(np.uint8)
        blk[82:84] = np.array([dmin]).view(np.uint8)
        exact = [float(d) * sc[k // 16] * q[k] - float(dmin) * m[k // 16] for k in range(256)]
        if all(float(np.float32(v)) == v for v in exact):
            return blk, np.array(exact)


def test_q2k_round_trip_fixed_point():
    rng = np.random.default_rng(11)
    for _ in range(40):
        blk, exact = _exact_q2k_block(rng)
        w = oracle.dequant_q2k(blk, 1, 256)[0]
        assert np.array_equal(w.astype(np.float64), exact)
        assert np.array_equal(oracle.quantize_q2k(w[None, :]), blk)


def test_q2k_zero_and_constant_blocks():
    z = oracle.quantize_q2k(np.zeros((1, 256), np.float32))
    assert np.all(z == 0)
    # constants on the code grid: 45 * 2^-10 = d*sc*q with d = 2^-10, sc = 15, q = 3;
    # -15 * 2^-10 = -dmin*m with dmin = 2^-10, m = 15 (and d = 0)
    for v in (45 / 1024, -15 / 1024):
        c = np.full((1, 256), v, np.float32)
        w = oracle.dequant_q2k(oracle.quantize_q2k(c), 1, 256)
        assert np.array_equal(w, c)
    c = np.full((1, 256), 0.25, np.float32)   # off the grid: within half a step of d*sc*q
    w = oracle.dequant_q2k(oracle.quantize_q2k(c), 1, 256)
    assert np.max(np.abs(w - c)) <= 0.25 / 45 * 1.5


def test_q2k_error_bound_on_gaussian_blocks():
    rng = np.random.default_rng(3)
    w = (rng.standard_normal((64, 256)) * 0.02).astype(np.float32)
    blob = oracle.quantize_q2k(w).reshape(64, 84)
    wh = oracle.dequant_q2k(blob, 64, 256)
    for r in range(64):
        d = float(blob[r, 80:82].view(np.float16)[0])
        dmin = float(blob[r, 82:84].view(np.float16)[0])
        for j in range(16):
            sc = blob[r, j] & 15
            # rounding the affine grid (step a_j = d*sc +- d/2, offset b_j +- dmin/2)
            bound = 0.5 * d * sc + 1.5 * d + 0.5 * dmin + 1e-6
            assert np.max(np.abs(w[r, 16 * j:16 * j + 16] - wh[r, 16 * j:16 * j + 16])) <= bound


def test_q2k_rejects_non_finite():
    w = np.zeros((1, 256), np.float32)
    w[0, 5] = np.nan
    with pytest.raises(ValueError):
        oracle.quantize_q2k(w)


# ---------------------------------------------------------------- Q4_K-style blocks

def test_q4k_dequant_hand_built_block():
    blk = np.zeros(144, np.uint8)
    blk[0:2] = np.array([_half_bits(0.5)], np.uint16).view(np.uint8)    # d = 0.5
    blk[2:4] = np.array([_half_bits(0.25)], np.uint16).view(np.uint8)   # dmin = 0.25
    # sub-block 0: sc = 5 (0b000101), m = 18 (0b010010): low nibbles 5 and 2, high bits 0 and 1
    blk[4] = 0x25
    blk[12] = 0b0100          # j = 0 in bits 0-3: sc high bits 00, m high bits 01
    # sub-block 3: sc = 63 (0b111111), m = 0: low nibble 15, high bits 11 in byte 12 + 1, bits 4-7
    blk[7] = 0x0F
    blk[13] = 0b0011 << 4
    blk[16] = 0x21            # weights 0, 1: q = 1, 2
    blk[17] = 0xF0            # weights 2, 3: q = 0, 15
    blk[16 + 48] = 0x07       # weight 96 (sub-block 3): q = 7, weight 97: q = 0
    w = oracle.dequant_q4k(blk, 1, 256)[0]
    # w = d*sc*q - dmin*m: sub-block 0: 2.5 q - 4.5; sub-block 3: 31.5 q
    assert list(w[:5]) == [-2.0, 0.5, -4.5, 33.0, -4.5]
    assert list(w[96:98]) == [220.5, 0.0]
    assert np.all(w[32:96] == 0.0) and np.all(w[128:] == 0.0)


def _exact_q4k_block(rng):
    """A block whose fp32 values are exact and which the quantiser must reproduce."""
    while True:
        d = np.float16(rng.uniform(2 ** -9, 2 ** -7))
        dmin = np.float16(rng.uniform(2 ** -9, 2 ** -7))
        sc = rng.integers(1, 64, 8)
        m = rng.integers(0, 64, 8)
        sc[rng.integers(8)] = 63
        m[rng.integers(8)] = 63
        q = rng.integers(0, 16, 256)
        for j in range(8):
            a, b = rng.choice(32, 2, replace=False)
            q[32 * j + a], q[32 * j + b] = 0, 15
        blk = np.zeros(144, np.uint8)
        blk[0:2] = np.array([d], np.float16).view(np.uint8)
        blk[2:4] = np.array([dmin], np.float16).view(np.uint8)
        for j in range(8):
            blk[4 + j] = (sc[j] & 15) | ((m[j] & 15) << 4)
            blk[12 + j // 2] |= ((sc[j] >> 4) | ((m[j] >> 4) << 2)) << (4 * (j % 2))
        for k in range(256):
            blk[16 + k // 2] |= q[k] << (4 * (k % 2))
        exact = np.array([float(d) * sc[k // 32] * q[k] - float(dmin) * m[k // 32] for k in range(256)])
        if np.all(np.abs(exact) < 60000) and np.array_equal(exact.astype(np.float32).astype(np.float64), exact):
            return blk, exact


def test_q4k_round_trip_fixed_point():
    rng = np.random.default_rng(13)
    for _ in range(40):
        blk, exact = _exact_q4k_block(rng)
        w = oracle.dequant_q4k(blk, 1, 256)[0]
        assert np.array_equal(w.astype(np.float64), exact)
        assert np.array_equal(oracle.quantize_q4k(w[None, :]), blk)


def test_q4k_zero_and_constant_blocks():
    assert np.all(oracle.quantize_q4k(np.zeros((1, 256), np.float32)) == 0)
    # constants on the code grid: 945 * 2^-12 = d*sc*q with d = 2^-12, sc = 63, q = 15;
    # -63 * 2^-12 = -dmin*m with dmin = 2^-12, m = 63 (and d = 0)
    for v in (945 / 4096, -63 / 4096):
        c = np.full((1, 256), v, np.float32)
        assert np.array_equal(oracle.dequant_q4k(oracle.quantize_q4k(c), 1, 256), c)


def test_q4k_error_bound_on_gaussian_blocks():
    rng = np.random.default_rng(5)
    w = (rng.standard_normal((64, 256)) * 0.02).astype(np.float32)
    blob = oracle.quantize_q4k(w).reshape(64, 144)
    wh = oracle.dequant_q4k(blob, 64, 256)
    for r in range(64):
        d = float(blob[r, 0:2].view(np.float16)[0])
        dmin = float(blob[r, 2:4].view(np.float16)[0])
        for j in range(8):
            sc = (blob[r, 4 + j] & 15) | (((blob[r, 12 + j // 2] >> (4 * (j % 2))) & 3) << 4)
            # rounding the affine grid (step a_j = d*sc +- d/2 over 15 steps, offset +- dmin/2)
            bound = 0.5 * d * sc + 7.5 * d + 0.5 * dmin + 1e-6
            assert np.max(np.abs(w[r, 32 * j:32 * j + 32] - wh[r, 32 * j:32 * j + 32])) <= bound
    # and the 4-bit codes are finer than the 2-bit ones on the same weights
    e2 = np.abs(oracle.dequant_q2k(oracle.quantize_q2k(w), 64, 256) - w).mean()
    assert np.abs(wh - w).mean() < 0.3 * e2


def test_q4k_rejects_non_finite():
    w = np.zeros((1, 256), np.float32)
    w[0, 7] = np.inf
    with pytest.raises(ValueError):
        oracle.quantize_q4k(w)


# ---------------------------------------------------------------- IQ2-style blocks

def test_iq2_dequant_hand_built_block():
    g = oracle.iq2_grid()
    blk = np.zeros(66, np.uint8)
    blk[0:2] = np.array([_half_bits(0.5)], np.uint16).view(np.uint8)     # d = 0.5
    blk[2:6] = [1, 0, 0, 0]                       # sub-block 0: group 0 uses entry 1
    u = (0b0000011) | (3 << 28)                   # group 0: elements 0,1 negative; s = 3
    blk[6:10] = np.array([u], np.uint32).view(np.uint8)
    w = oracle.dequant_iq2(blk, 1, 256)[0]
    scale = 0.5 * 4 / 16                          # d*(s+1)/16
    exp0 = [scale * v for v in g[1]]
    exp0[0], exp0[1] = -exp0[0], -exp0[1]        # two stored negatives -> parity 0, element 7 +
    assert list(w[:8]) == exp0
    assert list(w[8:32]) == [scale] * 24          # groups 1..3: entry 0 (ones), no signs
    assert np.all(w[32:] == 0.5 / 16)             # sub-blocks 1..7: s = 0, entry 0, d/16


def test_iq2_parity_sets_the_eighth_sign():
    blk = np.zeros(66, np.uint8)
    blk[0:2] = np.array([_half_bits(1.0)], np.uint16).view(np.uint8)
    u = 0b0000100 | (0b1100000 << 7)   # group 0: one stored negative (odd), group 1: two
    blk[6:10] = np.array([u], np.uint32).view(np.uint8)
    w = oracle.dequant_iq2(blk, 1, 256)[0]
    assert w[2] < 0 and w[7] < 0 and np.sum(w[:8] < 0) == 2
    assert w[8 + 5] < 0 and w[8 + 6] < 0 and w[8 + 7] > 0 and np.sum(w[8:16] < 0) == 2


def _exact_iq2_block(rng, all_s15=False):
    g = oracle.iq2_grid()
    blk = np.zeros(66, np.uint8)
    d = np.float16(rng.uniform(2 ** -9, 2 ** -5))
    blk[0:2] = np.array([d]).view(np.uint8)
    vals = np.zeros(256)
    jmax = rng.integers(8)
    for j in range(8):
        s = 15 if (all_s15 or j == jmax) else int(rng.integers(16))
        idx = rng.integers(0, 256, 4)
        if j == jmax:
            while 7 not in g[idx[0]]:
                idx[0] = rng.integers(256)
        u = s << 28
        for gi in range(4):
            s7 = int(rng.integers(128))
            u |= s7 << (7 * gi)
            par = bin(s7).count("1") & 1
            for i in range(8):
                neg = (s7 >> i) & 1 if i < 7 else par
                v = float(d) * (s + 1) / 16 * g[idx[gi], i]
                vals[32 * j + 8 * gi + i] = -v if neg else v
        blk[2 + 8 * j:6 + 8 * j] = idx
        blk[6 + 8 * j:10 + 8 * j] = np.array([u], np.uint32).view(np.uint8)
    return blk, vals


def test_iq2_round_trip_fixed_point():
    rng = np.random.default_rng(5)
    for _ in range(30):
        blk, vals = _exact_iq2_block(rng, all_s15=True)
        w = oracle.dequant_iq2(blk, 1, 256)[0]
        assert np.array_equal(w.astype(np.float64), vals)
        assert np.array_equal(oracle.quantize_iq2(w[None, :]), blk)   # no alias at s = 15
    for _ in range(30):
        blk, vals = _exact_iq2_block(rng)
        w = oracle.dequant_iq2(blk, 1, 256)[0]
        assert np.array_equal(w.astype(np.float64), vals)
        # other scales may alias (s+1)G = (s'+1)G'; the values must still be reproduced
        w2 = oracle.dequant_iq2(oracle.quantize_iq2(w[None, :]), 1, 256)[0]
        assert np.array_equal(w2, w)


def test_iq2_emitted_groups_have_even_negatives():
    rng = np.random.default_rng(9)
    w = (rng.standard_normal((16, 256)) * 0.02).astype(np.float32)
    wh = oracle.dequant_iq2(oracle.quantize_iq2(w), 16, 256)
    negs = (wh.reshape(-1, 8) < 0).sum(axis=1)
    assert np.all(negs % 2 == 0)


def _iq2_sse_bruteforce(wsub, d, grid):
    """Exhaustive (s, idx per group) SSE for a 32-weight sub-block, with the sign rule."""
    a = np.zeros((4, 8))
    for gi in range(4):
        wg = wsub[8 * gi:8 * gi + 8].astype(np.float64)
        neg = wg < 0
        if neg.sum() % 2:
            im = int(np.argmin(np.abs(wg)))
            neg[im] = ~neg[im]
        a[gi] = np.where(neg, -wg, wg)
    G = grid.astype(np.float64)
    best = np.inf
    per_s = []
    for s in range(16):
        c = d * (s + 1) / 16
        err = ((a[:, None, :] - c * G[None, :, :]) ** 2).sum(-1)   # [4, 256]
        tot = err.min(axis=1).sum()
        per_s.append(tot)
        best = min(best, tot)
    return best, a


def test_iq2_quantiser_choice_is_optimal_bruteforce():
    rng = np.random.default_rng(21)
    grid = oracle.iq2_grid()
    w = (rng.standard_normal((8, 256)) * 0.02).astype(np.float32)
    blob = oracle.quantize_iq2(w).reshape(8, 66)
    for r in range(8):
        d = float(blob[r, 0:2].view(np.float16)[0])
        assert d == float(np.float16(np.abs(w[r]).astype(np.float64).max() / 7))
        for j in range(8):
            best, a = _iq2_sse_bruteforce(w[r, 32 * j:32 * j + 32], d, grid)
            sb = blob[r, 2 + 8 * j:10 + 8 * j]
            s = int(sb[4:8].view(np.uint32)[0] >> 28)
            c = d * (s + 1) / 16
            chosen = sum(((a[gi] - c * grid[sb[gi]]) ** 2).sum() for gi in range(4))
            assert chosen <= best * (1 + 1e-12) + 1e-30


def test_iq2_zero_block():
    assert np.all(oracle.quantize_iq2(np.zeros((2, 256), np.float32)) == 0)
