"""The seeded workloads against the recipe they follow: the five layer configurations (tokens,
d_model, d_ff, experts, top-k, seed, the logit bias and the tie fraction), and what the drawn
inputs must show -- exact ties at the large prefill chunk, the Zipf-skewed expert popularity that
makes a few groups large and many small, the mildly uneven decode micro-batch, and activations
drawn from N(0, 1) and rounded to bf16. Routing here is the oracle's (CPU only)."""
import numpy as np
import pytest

import oracle
import synth

# name: (T, d_model, d_ff, experts, top-k, seed, bias, tie fraction, shared expert)
CONFIGS = {
    "tiny_t4": (4, 256, 256, 8, 2, 0, (), 0.0, False),
    "decode_t1": (1, 4096, 2048, 256, 8, 1, (), 0.0, True),
    "decode_t32": (32, 4096, 2048, 256, 8, 2, ("normal", 0.5), 0.0, True),
    "prefill_t2048": (2048, 4096, 2048, 256, 8, 3, ("zipf", 1.0), 0.0, True),
    "prefill_t8192_d7168": (8192, 7168, 2048, 256, 8, 4, ("zipf", 1.2), 0.05, True),
}


@pytest.mark.parametrize("name", sorted(CONFIGS))
def test_workload_shapes(name):
    wl = synth.WORKLOADS[name]
    got = (wl.T, wl.D, wl.F, wl.E, wl.k, wl.seed, wl.bias, wl.tie_frac, wl.shared)
    assert got == CONFIGS[name]
    assert wl.fmt == "q2" and wl.slots == 0


def _logits(name):
    # the logits are drawn before the activations, so a narrow d_model leaves them unchanged
    wl = synth.WORKLOADS[name]
    L, _ = synth.draw_inputs(wl.replace(D=16))
    return wl, L


def test_narrow_activations_leave_the_logits_unchanged():
    wl = synth.WORKLOADS["decode_t32"]
    assert np.array_equal(synth.draw_inputs(wl)[0], synth.draw_inputs(wl.replace(D=16))[0])


def test_large_prefill_has_five_percent_exact_ties_at_the_top_and_at_the_k_boundary():
    wl, L = _logits("prefill_t8192_d7168")
    o = np.argsort(-L, axis=1, kind="stable")
    r = np.arange(wl.T)
    top = L[r, o[:, 0]] == L[r, o[:, 1]]
    edge = L[r, o[:, wl.k - 1]] == L[r, o[:, wl.k]]
    n = int(round(0.05 * wl.T))
    assert top.sum() == n and edge.sum() == n and (top & edge).sum() == n


@pytest.mark.parametrize("name", ["tiny_t4", "decode_t1", "decode_t32", "prefill_t2048"])
def test_other_workloads_have_no_forced_ties(name):
    wl, L = _logits(name)
    o = np.argsort(-L, axis=1, kind="stable")
    r = np.arange(wl.T)
    assert not np.any(L[r, o[:, 0]] == L[r, o[:, 1]])


@pytest.mark.parametrize("name", ["prefill_t2048", "prefill_t8192_d7168"])
def test_zipf_bias_makes_a_few_groups_large_and_most_small(name):
    wl, L = _logits(name)
    idx, _ = oracle.route(L, wl.k)
    counts = np.bincount(idx.ravel(), minlength=wl.E)
    mean = wl.T * wl.k / wl.E
    assert counts.sum() == wl.T * wl.k
    assert np.sort(counts)[-5:].min() >= 10 * mean     # the five most popular experts: hundreds or thousands
    assert np.median(counts) <= 0.05 * mean            # most experts: a few tokens or none
    # the bias is what orders popularity: the most popular experts have the largest bias
    rng = np.random.default_rng(wl.seed)
    rng.standard_normal((wl.T, wl.E))
    rank = rng.permutation(wl.E) + 1                   # the recipe's ranks, drawn right after the logits
    assert set(np.argsort(-counts, kind="stable")[:3]) <= set(np.argsort(rank)[:6])


def test_decode_micro_batch_is_mildly_uneven():
    wl, L = _logits("decode_t32")
    idx, _ = oracle.route(L, wl.k)
    counts = np.bincount(idx.ravel(), minlength=wl.E)
    # 256 pairs over 256 experts: uniform draws would touch about 162 experts; the N(0, 0.5)
    # bias concentrates them somewhat, but no expert takes a large share
    assert 100 <= np.count_nonzero(counts) <= 160
    assert counts.max() <= 16


def test_activations_are_standard_normal_in_bf16():
    wl = synth.WORKLOADS["prefill_t2048"]
    _, x = synth.draw_inputs(wl)
    assert x.dtype == np.uint16 and x.shape == (wl.T, wl.D)
    xf = (x.astype(np.uint32) << 16).view(np.float32)
    assert abs(xf.mean()) < 0.01 and abs(xf.std() - 1.0) < 0.01
    # bf16 rounding of the fp32 draw: the same values from an independent re-draw, truncated
    # bits compared within one bf16 step
    rng = np.random.default_rng(wl.seed)
    rng.standard_normal((wl.T, wl.E))
    rng.permutation(wl.E)
    ref = rng.standard_normal((wl.T, wl.D)).astype(np.float32)
    assert np.all(np.abs(xf - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-30)
