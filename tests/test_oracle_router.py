"""Pins for the oracle's router logits (CPU only): closed forms that a dropped term, a wrong
index, a transposed operand or a wrong bias would break, and the fp32 error bound of any order of
summation against the exact (fp64) sum."""
import numpy as np

import synth
from oracle.router import bf16_to_f32, router_logits


def _bits(a):
    return synth.f32_to_bf16_bits(np.asarray(a, np.float32))


def test_integer_inputs_give_the_exact_integer_matmul():
    # small integers are exact in bf16 and every partial sum stays exact in fp32
    rng = np.random.default_rng(0)
    T, D, E = 5, 512, 24
    x = rng.integers(-3, 4, size=(T, D)).astype(np.float32)
    w = rng.integers(-3, 4, size=(E, D)).astype(np.float32)
    b = rng.integers(-50, 51, size=E).astype(np.float32)
    got = router_logits(_bits(x), _bits(w), b)
    ref = x.astype(np.int64) @ w.astype(np.int64).T + b.astype(np.int64)
    assert np.array_equal(got, ref.astype(np.float32))
    assert got.shape == (T, E) and got.dtype == np.float32


def test_single_nonzero_per_router_row():
    # one column per expert: the logit is that product plus the bias, rounded once
    rng = np.random.default_rng(1)
    T, D, E = 3, 256, 8
    x = rng.standard_normal((T, D)).astype(np.float32)
    xb = _bits(x)
    cols = rng.choice(D, size=E, replace=False)
    w = np.zeros((E, D), np.float32)
    w[np.arange(E), cols] = rng.standard_normal(E).astype(np.float32)
    wb = _bits(w)
    b = rng.standard_normal(E).astype(np.float32)
    got = router_logits(xb, wb, b)
    xv, wv = bf16_to_f32(xb), bf16_to_f32(wb)
    ref = (xv[:, cols] * wv[np.arange(E), cols][None, :]).astype(np.float32) + b[None, :]
    assert np.array_equal(got, ref.astype(np.float32))
    assert np.array_equal(router_logits(xb, wb), (xv[:, cols] * wv[np.arange(E), cols][None, :]).astype(np.float32))


def test_within_the_fp32_summation_bound_of_the_exact_sum():
    rng = np.random.default_rng(2)
    T, D, E = 4, 4096, 16
    xb = _bits(rng.standard_normal((T, D)))
    wb = _bits(0.02 * rng.standard_normal((E, D)))
    b = (0.1 * rng.standard_normal(E)).astype(np.float32)
    got = router_logits(xb, wb, b).astype(np.float64)
    xv, wv = bf16_to_f32(xb).astype(np.float64), bf16_to_f32(wb).astype(np.float64)
    exact = xv @ wv.T + b.astype(np.float64)
    # each term passes through at most D/256*8 + 5 + 1 fp32 additions
    n = D // 256 * 8 + 6
    bound = n * 2.0 ** -24 * (np.abs(xv) @ np.abs(wv).T + np.abs(b))
    assert np.all(np.abs(got - exact) <= bound)
    assert np.max(np.abs(got - exact)) > 0          # the sums do round: the bound is not vacuous


def test_the_order_is_the_documented_one():
    # products that cancel only in the documented order: lane 0's columns 0 and 1 add 2^30 and
    # -2^30 before any other term, so the 1s of the other lanes survive; any order that adds a
    # 1 to 2^30 first would lose it
    D, E = 256, 8
    x = np.zeros((1, D), np.float32)
    w = np.zeros((E, D), np.float32)
    x[0, 0], x[0, 1] = 2.0 ** 15, 2.0 ** 15
    w[:, 0], w[:, 1] = 2.0 ** 15, -(2.0 ** 15)
    x[0, 8:D:8] = 1.0                   # columns 8, 16, ...: lanes 1..31, one term each
    w[:, 8:D:8] = 1.0
    got = router_logits(_bits(x), _bits(w))
    assert np.all(got == 31.0)


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
    top_router = np.bincount(oracle.route(R, wl.k)[0].ravel(), minlength=wl.E).max()
    assert 0.5 * top_drawn < top_router < 2.0 * top_drawn
