"""Pins for the oracle's routing, grouping and expert FFN (CPU only).

Routing is checked against numpy's lexicographic sort and scipy's softmax/expit; grouping
against numpy's stable argsort and its invariants; the FFN against a naive loop-by-loop
evaluation of the SwiGLU definition with math.exp, and against closed forms (x = 0, all
experts identical, a single shared expert)."""
import math

import numpy as np
import pytest
from scipy.special import expit, softmax

import oracle
import synth


def _bruteforce_topk(l, k):
    order = np.lexsort((np.arange(l.size), -l.astype(np.float64)))
    return order[:k]


@pytest.mark.parametrize("mode", [0, 1])
def test_route_matches_sort_and_library_gates(mode):
    rng = np.random.default_rng(1)
    L = rng.standard_normal((50, 32)).astype(np.float32)
    L[3, 7] = L[3, 9] = L[3].max() + 1        # exact top-1 tie: lower index first
    L[5, :] = 0.25                            # all tied: experts 0..k-1
    idx, g = oracle.route(L, 6, mode)
    for t in range(50):
        sel = _bruteforce_topk(L[t], 6)
        assert list(idx[t]) == list(sel)
        ls = L[t, sel].astype(np.float64)
        ref = softmax(ls) if mode == 0 else expit(ls) / expit(ls).sum()
        assert np.allclose(g[t], ref, rtol=0, atol=1e-15)
        assert abs(g[t].sum() - 1.0) <= 1e-12
    assert list(idx[3][:2]) == [7, 9]
    assert list(idx[5]) == [0, 1, 2, 3, 4, 5]


def test_route_special_cases():
    rng = np.random.default_rng(2)
    L = rng.standard_normal((10, 16)).astype(np.float32)
    idx, g = oracle.route(L, 1)
    assert np.all(g == 1.0)
    assert np.array_equal(idx[:, 0], np.argmax(L, axis=1))
    idx, g = oracle.route(L, 16)
    assert all(sorted(r) == list(range(16)) for r in idx)


def _keys(l):
    """The ranking keys of one token's logits: NaN counts as -inf."""
    k = l.astype(np.float64)
    k[np.isnan(k)] = -np.inf
    return k


@pytest.mark.parametrize("mode", [0, 1])
def test_route_nan_and_infinite_logits(mode):
    """NaN ranks as -inf (ties to the lower index), +inf and -inf rank where they belong; the
    selection is numpy's lexsort over the keys. Gate weights: closed forms of the stated rule."""
    nan, inf = np.float32(np.nan), np.float32(np.inf)
    rows = [
        [1.0, nan, 7.0, 2.0, 0.5, -3.0, 4.0, 0.0],     # one NaN: never chosen over a finite logit
        [nan, 9.0, nan, 8.0, 1.0, 2.0, 3.0, 4.0],      # NaNs among the top logits
        [0.5, inf, 3.0, -1.0, inf, 2.0, 1.0, 0.0],     # two +inf: they share the weight
        [-inf, 2.0, -inf, 1.0, 0.0, -1.0, -2.0, -3.0],  # -inf at the bottom
        [nan] * 8,                                     # all NaN: experts 0..k-1, equal weights
        [-inf] * 8,                                    # all -inf: the same
        [nan, -inf, nan, -inf, 5.0, nan, -inf, nan],   # one finite logit; NaN and -inf tie
    ]
    L = np.array(rows, np.float32)
    k = 4
    idx, g = oracle.route(L, k, mode)
    for t in range(len(rows)):
        keys = _keys(L[t])
        sel = np.lexsort((np.arange(8), -keys))[:k]
        assert list(idx[t]) == list(sel), t
        assert abs(g[t].sum() - 1.0) <= 1e-12, t
    assert list(idx[0]) == [2, 6, 3, 0]
    assert list(idx[1]) == [1, 3, 7, 6]
    assert list(idx[4]) == [0, 1, 2, 3] and np.all(g[4] == 0.25)
    assert list(idx[5]) == [0, 1, 2, 3] and np.all(g[5] == 0.25)
    assert list(idx[6]) == [4, 0, 1, 2]       # the finite logit, then NaN and -inf tie, by index
    if mode == 0:
        assert list(g[2]) == [0.5, 0.5, 0.0, 0.0]
        assert list(g[6]) == [1.0, 0.0, 0.0, 0.0]
        ls = np.array([2.0, 1.0, 0.0, -1.0])
        assert np.allclose(g[3], softmax(ls), rtol=0, atol=1e-15)
    else:
        s = expit(np.array([inf, inf, 3.0, 2.0], np.float64))
        assert np.allclose(g[2], s / s.sum(), rtol=0, atol=1e-15)
        assert list(g[6]) == [1.0, 0.0, 0.0, 0.0]
        s = expit(np.array([2.0, 1.0, 0.0, -1.0]))
        assert np.allclose(g[3], s / s.sum(), rtol=0, atol=1e-15)


def test_route_sigmoid_gates_far_below_zero():
    """The sigmoid weights keep their ratio where sigmoid itself underflows double precision: for
    v far below 0, sigmoid(v) = exp(v) (1 + O(exp(v))), so the weights are the softmax of v."""
    L = np.array([[-800.0, -801.0, -803.0, -900.0, -5000.0]], np.float32)
    idx, g = oracle.route(L, 3, 1)
    assert list(idx[0]) == [0, 1, 2]
    ref = softmax(np.array([-800.0, -801.0, -803.0]))
    assert np.allclose(g[0], ref, rtol=0, atol=1e-15)


def test_route_boundary_ties_of_the_tie_workload():
    wl = synth.WORKLOADS["prefill_t8192_d7168"].replace(T=400, D=256)
    L, _ = synth.draw_inputs(wl)
    idx, _ = oracle.route(L, wl.k)
    n_tied = 0
    for t in range(wl.T):
        o = np.argsort(-L[t], kind="stable")
        if L[t, o[0]] == L[t, o[1]]:
            n_tied += 1
            assert idx[t, 0] == min(o[0], o[1]) and idx[t, 1] == max(o[0], o[1])
        assert list(idx[t]) == list(_bruteforce_topk(L[t], wl.k))
    assert n_tied >= 20


def test_permute_invariants_and_stability():
    rng = np.random.default_rng(4)
    T, k, E = 97, 4, 13
    L = rng.standard_normal((T, E)).astype(np.float32)
    idx, _ = oracle.route(L, k)
    counts, offsets, perm, inv = oracle.permute(idx, E)
    P = T * k
    assert counts.sum() == P and offsets[0] == 0 and offsets[E] == P
    assert np.all(np.diff(offsets) == counts)
    assert sorted(perm) == list(range(P))
    assert np.array_equal(perm[inv], np.arange(P))
    assert np.array_equal(perm, np.argsort(idx.reshape(-1), kind="stable"))
    for e in range(E):
        assert np.all(idx.reshape(-1)[perm[offsets[e]:offsets[e + 1]]] == e)
    tok = perm // k
    assert np.all(np.bincount(tok, minlength=T) == k)


def test_permute_empty_experts():
    idx = np.array([[3, 1], [3, 1]], np.int32)
    counts, offsets, perm, inv = oracle.permute(idx, 6)
    assert list(counts) == [0, 2, 0, 2, 0, 0]
    assert list(offsets) == [0, 0, 2, 2, 4, 4, 4]
    assert list(perm) == [1, 3, 0, 2]


# ---------------------------------------------------------------- FFN

def _tiny_layer(T=3, D=256, F=256, E=4, k=2, seed=0, shared=True):
    wl = synth.Workload("t", T=T, D=D, F=F, E=E, k=k, seed=seed, shared=shared)
    L, x = synth.draw_inputs(wl)
    gate = [oracle.quantize_iq2(synth.expert_weight(seed, e, synth.GATE, F, D)) for e in range(E)]
    up = [oracle.quantize_iq2(synth.expert_weight(seed, e, synth.UP, F, D)) for e in range(E)]
    down = [oracle.quantize_q2k(synth.expert_weight(seed, e, synth.DOWN, D, F)) for e in range(E)]
    sh = synth.shared_weights(seed, D, F) if shared else None
    return wl, L, x, gate, up, down, sh


def _naive_expert(xv, wg, wu, wd):
    D = len(xv)
    F = len(wg)
    h = []
    for r in range(F):
        u = sum(float(wu[r][c]) * xv[c] for c in range(D))
        v = sum(float(wg[r][c]) * xv[c] for c in range(D))
        h.append(v / (1.0 + math.exp(-v)) * u)
    return [sum(float(wd[r][c]) * h[c] for c in range(F)) for r in range(D)]


def test_ffn_matches_naive_loops():
    # non-square (d_ff != d_model), so that a transposed or swapped matrix cannot pass
    wl, L, x, gate, up, down, sh = _tiny_layer(T=2, k=2, F=512)
    delta, idx, g = oracle.moe_ffn(x, L, wl.k, gate, up, down, wl.D, wl.F, shared=sh)
    xf = oracle.bf16_to_f64(x)
    sg, su, sd = (oracle.bf16_to_f64(s).reshape(-1, wl.D if i < 2 else wl.F).tolist() for i, s in enumerate(sh))
    for t in range(wl.T):
        xv = xf[t].tolist()
        ref = _naive_expert(xv, sg, su, sd)
        for s in range(wl.k):
            e = int(idx[t, s])
            wg = oracle.dequant_iq2(gate[e], wl.F, wl.D).tolist()
            wu = oracle.dequant_iq2(up[e], wl.F, wl.D).tolist()
            wd = oracle.dequant_q2k(down[e], wl.D, wl.F).tolist()
            y = _naive_expert(xv, wg, wu, wd)
            ref = [a + g[t, s] * b for a, b in zip(ref, y)]
        assert np.max(np.abs(np.array(ref) - delta[t])) <= 1e-12 * max(1.0, np.max(np.abs(ref)))


def test_ffn_q4_matches_naive_loops():
    # the 4-bit variant's branch: Q4_K-style gate, up and down, on a non-square layer (d_ff != d_model)
    # so that a transposed or swapped matrix cannot pass
    T, D, F, E, k, seed = 2, 256, 512, 4, 2, 3
    wl = synth.Workload("t4", T=T, D=D, F=F, E=E, k=k, seed=seed, shared=True)
    L, x = synth.draw_inputs(wl)
    gate = [oracle.quantize_q4k(synth.expert_weight(seed, e, synth.GATE, F, D)) for e in range(E)]
    up = [oracle.quantize_q4k(synth.expert_weight(seed, e, synth.UP, F, D)) for e in range(E)]
    down = [oracle.quantize_q4k(synth.expert_weight(seed, e, synth.DOWN, D, F)) for e in range(E)]
    sh = synth.shared_weights(seed, D, F)
    delta, idx, g = oracle.moe_ffn(x, L, k, gate, up, down, D, F, shared=sh, fmt="q4")
    xf = oracle.bf16_to_f64(x)
    sg, su, sd = (oracle.bf16_to_f64(s).reshape(-1, D if i < 2 else F).tolist() for i, s in enumerate(sh))
    for t in range(T):
        xv = xf[t].tolist()
        ref = _naive_expert(xv, sg, su, sd)
        for s_ in range(k):
            e = int(idx[t, s_])
            y = _naive_expert(xv, oracle.dequant_q4k(gate[e], F, D).tolist(), oracle.dequant_q4k(up[e], F, D).tolist(),
                              oracle.dequant_q4k(down[e], D, F).tolist())
            ref = [a + g[t, s_] * b for a, b in zip(ref, y)]
        assert np.max(np.abs(np.array(ref) - delta[t])) <= 1e-12 * max(1.0, np.max(np.abs(ref)))


def test_ffn_zero_input_gives_zero():
    wl, L, x, gate, up, down, sh = _tiny_layer()
    delta, _, _ = oracle.moe_ffn(np.zeros_like(x), L, wl.k, gate, up, down, wl.D, wl.F, shared=sh)
    assert np.all(delta == 0.0)


def test_ffn_identical_experts_reduce_to_one_expert():
    wl, L, x, gate, up, down, _ = _tiny_layer(T=5, E=6, k=3, shared=False)
    same = lambda b: [b[0]] * wl.E  # noqa: E731
    delta, _, _ = oracle.moe_ffn(x, L, wl.k, same(gate), same(up), same(down), wl.D, wl.F)
    xf = oracle.bf16_to_f64(x)
    y = oracle.expert_ffn_dense(xf, oracle.dequant_iq2(gate[0], wl.F, wl.D).astype(np.float64),
                                oracle.dequant_iq2(up[0], wl.F, wl.D).astype(np.float64),
                                oracle.dequant_q2k(down[0], wl.D, wl.F).astype(np.float64))
    assert np.allclose(delta, y, rtol=1e-12, atol=1e-14)   # gate weights sum to 1


def test_ffn_token_subset_equals_full():
    wl, L, x, gate, up, down, sh = _tiny_layer(T=6, E=5, k=2)
    full, _, _ = oracle.moe_ffn(x, L, wl.k, gate, up, down, wl.D, wl.F, shared=sh)
    sub, _, _ = oracle.moe_ffn(x, L, wl.k, gate, up, down, wl.D, wl.F, shared=sh, tokens=[4, 1])
    assert np.allclose(sub, full[[4, 1]], rtol=1e-13, atol=1e-16)   # BLAS blocking may differ


def test_silu_closed_forms():
    from oracle.moe import silu
    assert silu(np.array([0.0]))[0] == 0.0
    assert abs(silu(np.array([1.0]))[0] - 1.0 / (1.0 + math.exp(-1.0))) < 1e-16
    assert silu(np.array([-1000.0]))[0] == 0.0
