"""Pins for the oracle's router logits (CPU only): closed forms that a dropped term, a wrong
index, a transposed operand or a wrong bias would break, a correctly rounded brute-force sum, and
the fp32 error bound that the device's logits are checked against (valid for an fp32 summation
of the stated depth, and not vacuous)."""
import math

import numpy as np

import synth
from oracle.router import bf16_to_f64, fp32_bound, router_logits


def _bits(a):
    return synth.f32_to_bf16_bits(np.asarray(a, np.float32))


def test_integer_inputs_give_the_exact_integer_matmul():
    # small integers are exact in bf16, and so is every partial sum
    rng = np.random.default_rng(0)
    T, D, E = 5, 512, 24
    x = rng.integers(-3, 4, size=(T, D)).astype(np.float32)
    w = rng.integers(-3, 4, size=(E, D)).astype(np.float32)
    b = rng.integers(-50, 51, size=E).astype(np.float32)
    got = router_logits(_bits(x), _bits(w), b)
    ref = x.astype(np.int64) @ w.astype(np.int64).T + b.astype(np.int64)
    assert got.shape == (T, E) and got.dtype == np.float64
    assert np.array_equal(got, ref.astype(np.float64))


def test_single_nonzero_per_router_row():
    # one column per expert: the logit is that product plus the bias (exact in fp64)
    rng = np.random.default_rng(1)
    T, D, E = 3, 256, 8
    x = rng.standard_normal((T, D)).astype(np.float32)
    xb = _bits(x)
    cols = rng.choice(D, size=E, replace=False)
    w = np.zeros((E, D), np.float32)
    w[np.arange(E), cols] = rng.standard_normal(E).astype(np.float32)
    wb = _bits(w)
    b = rng.standard_normal(E).astype(np.float32)
    xv, wv = bf16_to_f64(xb), bf16_to_f64(wb)
    prod = xv[:, cols] * wv[np.arange(E), cols][None, :]
    assert np.array_equal(router_logits(xb, wb, b), prod + b.astype(np.float64)[None, :])
    assert np.array_equal(router_logits(xb, wb), prod)


def test_against_a_correctly_rounded_sum():
    # math.fsum of the exact products and the bias is the exact sum rounded once
    rng = np.random.default_rng(3)
    T, D, E = 3, 512, 7
    xb = _bits(rng.standard_normal((T, D)))
    wb = _bits(0.02 * rng.standard_normal((E, D)))
    b = (0.1 * rng.standard_normal(E)).astype(np.float32)
    got = router_logits(xb, wb, b)
    xv, wv = bf16_to_f64(xb), bf16_to_f64(wb)
    for t in range(T):
        for e in range(E):
            ref = math.fsum([xv[t, d] * wv[e, d] for d in range(D)] + [float(b[e])])
            mag = math.fsum(abs(xv[t, d] * wv[e, d]) for d in range(D)) + abs(float(b[e]))
            assert abs(got[t, e] - ref) <= 1e-14 * mag


def test_fp32_bound_holds_for_fp32_sums_and_is_not_vacuous():
    rng = np.random.default_rng(2)
    T, D, E = 4, 4096, 16
    xb = _bits(rng.standard_normal((T, D)))
    wb = _bits(0.02 * rng.standard_normal((E, D)))
    b = (0.1 * rng.standard_normal(E)).astype(np.float32)
    exact = router_logits(xb, wb, b)
    bound = fp32_bound(xb, wb, b)
    xv = bf16_to_f64(xb).astype(np.float32)
    wv = bf16_to_f64(wb).astype(np.float32)
    # an fp32 summation of the stated depth: 32 lane sums of 8-column strips, halved, then the bias
    prod = (xv[:, None, :] * wv[None, :, :]).astype(np.float32).reshape(T, E, D // 256, 32, 8)
    lanes = np.zeros((T, E, 32), np.float32)
    for i in range(D // 256):
        for j in range(8):
            lanes = (lanes + prod[:, :, i, :, j]).astype(np.float32)
    while lanes.shape[-1] > 1:
        h = lanes.shape[-1] // 2
        lanes = (lanes[..., :h] + lanes[..., h:]).astype(np.float32)
    f32 = (lanes[..., 0] + b[None, :]).astype(np.float32).astype(np.float64)
    assert np.all(np.abs(f32 - exact) <= bound)
    assert np.max(np.abs(f32 - exact)) > 0          # the fp32 sums do round
    assert np.max(bound) < 0.01 * np.std(exact)     # and the bound is far below the logits' spread


def test_the_seeded_router_keeps_the_workloads_routing_mix():
    # the benchmark's router: logits of unit spread, and on a Zipf workload the same skew of the
    # group sizes as the drawn logits (the most loaded expert takes about as many pairs)
    import oracle
    wl = synth.WORKLOADS["prefill_t2048"].replace(T=256)
    L, x = synth.draw_inputs(wl)
    w, b = synth.router_weights(wl)
    assert w.shape == (wl.E, wl.D) and w.dtype == np.uint16 and b.shape == (wl.E,)
    R = router_logits(x, w, b)
    assert 0.8 < np.std(R - b[None, :]) < 1.2
    top_drawn = np.bincount(oracle.route(L, wl.k)[0].ravel(), minlength=wl.E).max()
    top_router = np.bincount(oracle.route(R.astype(np.float32), wl.k)[0].ravel(), minlength=wl.E).max()
    assert 0.5 * top_drawn < top_router < 2.0 * top_drawn


def _truncate_f32(v):
    """fp32 rounding toward zero of fp64 values (the addition a truncating unit performs)."""
    v = np.asarray(v, np.float64)
    r = v.astype(np.float32)
    up = np.abs(r.astype(np.float64)) > np.abs(v)
    r[up] = np.nextafter(r[up], np.float32(0))
    return r


def test_tensor_core_bound_holds_for_block_sums_and_is_not_vacuous():
    # the order the tensor-core router takes: 16-column blocks summed (here by halving, each
    # addition truncated), added in increasing order into one accumulator (truncated), then the bias
    from oracle.router import tensor_core_depth
    rng = np.random.default_rng(5)
    T, D, E = 3, 2048, 8
    xb = _bits(rng.standard_normal((T, D)))
    wb = _bits(0.02 * rng.standard_normal((E, D)))
    b = (0.1 * rng.standard_normal(E)).astype(np.float32)
    exact = router_logits(xb, wb, b)
    bound = fp32_bound(xb, wb, b, depth=tensor_core_depth(D))
    assert np.all(bound >= fp32_bound(xb, wb, b))  # the block order is the looser one
    xv = bf16_to_f64(xb)
    wv = bf16_to_f64(wb)
    prod = (xv[:, None, :] * wv[None, :, :]).reshape(T, E, D // 16, 16)  # exact products
    acc = np.zeros((T, E), np.float32)
    for blk in range(D // 16):
        p = prod[:, :, blk, :].astype(np.float32)
        while p.shape[-1] > 1:
            h = p.shape[-1] // 2
            p = _truncate_f32(p[..., :h].astype(np.float64) + p[..., h:].astype(np.float64))
        acc = _truncate_f32(acc.astype(np.float64) + p[..., 0].astype(np.float64))
    got = _truncate_f32(acc.astype(np.float64) + b.astype(np.float64)[None, :]).astype(np.float64)
    assert np.all(np.abs(got - exact) <= bound)
    assert np.max(np.abs(got - exact)) > 0
    assert np.max(bound) < 0.02 * np.std(exact)
