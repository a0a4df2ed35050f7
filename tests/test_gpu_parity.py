"""GPU parity through the C ABI against the oracle: routing, grouping and dequantised
weights bit-exact; the expert FFN within the normalised max error 2e-3 (the bound stated
for bf16/fp32-accumulate against fp64); determinism; edge cases."""
import numpy as np
import pytest

import oracle
import synth
from helpers import FFN_TOL, Layer, norm_max_err, sample_tokens

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ds4():
    import torch
    import bit_quantized_routed_gb300 as m
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    m.build()
    return m


# ---------------------------------------------------------------- routing and grouping

@pytest.mark.parametrize("T,E,k,mode", [(1, 256, 8, 0), (333, 256, 8, 0), (50, 8, 2, 1), (17, 32, 32, 0),
                                        (9, 1000, 32, 1), (5, 33, 1, 0)])
def test_route_bitexact(ds4, T, E, k, mode):
    import torch
    rng = np.random.default_rng(T * 7 + E)
    L = rng.standard_normal((T, E)).astype(np.float32)
    L[0, E // 3] = L[0, E // 2] = np.float32(9.0)          # exact top tie
    if T > 2:
        L[2, :] = np.float32(0.5)                          # everything tied
    idx_ref, g_ref = oracle.route(L, k, mode)
    idx, w = ds4.ds4moe_route(torch.from_numpy(L).cuda(), k, mode)
    assert np.array_equal(idx.cpu().numpy(), idx_ref)
    assert np.max(np.abs(w.cpu().numpy() - g_ref)) <= 1e-6


_NAN, _INF = np.float32(np.nan), np.float32(np.inf)
# rows of 8 logits: a NaN ranks as -inf (ties to the lower index), +inf and -inf where they belong
_SPECIAL_ROWS = [
    [1.0, _NAN, 7.0, 2.0, 0.5, -3.0, 4.0, 0.0],
    [_NAN, 9.0, _NAN, 8.0, 1.0, 2.0, 3.0, 4.0],
    [0.5, _INF, 3.0, -1.0, _INF, 2.0, 1.0, 0.0],
    [-_INF, 2.0, -_INF, 1.0, 0.0, -1.0, -2.0, -3.0],
    [_NAN] * 8,
    [-_INF] * 8,
    [_NAN, -_INF, _NAN, -_INF, 5.0, _NAN, -_INF, _NAN],
]


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("E", [8, 256, 1000])
def test_route_nan_and_infinite_logits(ds4, mode, E):
    import torch
    rng = np.random.default_rng(E + mode)
    L = rng.standard_normal((len(_SPECIAL_ROWS) + 1, E)).astype(np.float32)
    for t, row in enumerate(_SPECIAL_ROWS):
        L[t] = -np.inf if E > 8 else 0.0     # wider rows: the special values, then -inf
        L[t, :8] = row
    L[-1, E // 2] = np.nan                   # a NaN among ordinary logits
    for k in (1, 4, 8):
        idx_ref, g_ref = oracle.route(L, k, mode)
        idx, w = ds4.ds4moe_route(torch.from_numpy(L).cuda(), k, mode)
        w = w.cpu().numpy()
        assert np.array_equal(idx.cpu().numpy(), idx_ref)
        assert np.all(np.isfinite(w))
        assert np.max(np.abs(w - g_ref)) <= 1e-6


def test_route_zero_tokens(ds4):
    import torch
    idx, w = ds4.ds4moe_route(torch.zeros((0, 16), device="cuda"), 4)
    assert idx.shape == (0, 4)


@pytest.mark.parametrize("name", ["tiny_t4", "decode_t1", "decode_t32", "prefill_t2048", "prefill_t8192_d7168"])
def test_group_bitexact_on_workloads(ds4, name):
    import torch
    wl = synth.WORKLOADS[name]
    L, _ = synth.draw_inputs(wl)
    idx_ref, _ = oracle.route(L, wl.k)
    ref = oracle.permute(idx_ref, wl.E)
    idx, _ = ds4.ds4moe_route(torch.from_numpy(L).cuda(), wl.k)
    assert np.array_equal(idx.cpu().numpy(), idx_ref)
    got = ds4.ds4moe_group(idx, wl.E)
    for a, b in zip(got, ref):
        assert np.array_equal(a.cpu().numpy(), b)


def test_group_one_expert_takes_all(ds4):
    import torch
    idx = np.full((3000, 4), 5, np.int32)
    idx[:, 1:] = np.arange(1, 4)[None, :] + 10
    ref = oracle.permute(idx, 64)
    got = ds4.ds4moe_group(torch.from_numpy(idx).cuda(), 64)
    for a, b in zip(got, ref):
        assert np.array_equal(a.cpu().numpy(), b)


@pytest.mark.parametrize("T,k,E", [(777, 3, 40), (1, 1, 8), (4097, 8, 256), (33, 5, 7)])
def test_group_bitexact_ragged_pair_counts(ds4, T, k, E):
    # pair counts that leave every warp's share, and its last batch of loads, partly empty
    import torch
    rng = np.random.default_rng(T * k + E)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    ref = oracle.permute(idx, E)
    got = ds4.ds4moe_group(torch.from_numpy(idx).cuda(), E)
    for a, b in zip(got, ref):
        assert np.array_equal(a.cpu().numpy(), b)


# ---------------------------------------------------------------- device dequantisation

@pytest.mark.parametrize("D,F", [(512, 768), (768, 512)])   # even and odd blocks per row (chunk permutation)
def test_device_dequant_bitexact(ds4, D, F):
    import torch
    wl = synth.Workload("dq", T=1, D=D, F=F, E=3, k=1, seed=11)
    lay = Layer(wl, quantized=False, experts=range(3))
    lay.gate[1] = oracle.quantize_iq2(synth.expert_weight(5, 1, synth.GATE, wl.F, wl.D))
    lay.down[1] = oracle.quantize_q2k(synth.expert_weight(5, 1, synth.DOWN, wl.D, wl.F))
    W = lay.upload(ds4)
    for e in range(3):
        for m, (blob, rows, cols, deq) in enumerate([(lay.gate[e], wl.F, wl.D, oracle.dequant_iq2),
                                                     (lay.up[e], wl.F, wl.D, oracle.dequant_iq2),
                                                     (lay.down[e], wl.D, wl.F, oracle.dequant_q2k)]):
            ref = deq(blob, rows, cols)
            d32 = torch.empty((rows, cols), dtype=torch.float32, device="cuda")
            d16 = torch.empty((rows, cols), dtype=torch.float16, device="cuda")
            ds4.ds4moe_weights_dequantize(W, e, m, d32, d16)
            assert np.array_equal(d32.cpu().numpy().view(np.uint32), ref.view(np.uint32))
            assert np.array_equal(d16.cpu().numpy().view(np.uint16), ref.astype(np.float16).view(np.uint16))
    W.close()


# ---------------------------------------------------------------- the expert FFN

def _ffn_case(ds4, wl, quantized=True, tokens=None, gemm_min=None, mode=0, out_init=None):
    lay = Layer(wl, quantized=quantized)
    W = lay.upload(ds4)
    if gemm_min is not None:
        ds4.ds4moe_set_option(W, ds4.DS4MOE_OPT_GEMM_MIN_TOKENS, gemm_min)
        ds4.ds4moe_set_option(W, ds4.DS4MOE_OPT_SHARED_GEMM_MIN_TOKENS, gemm_min)
    got = lay.run(ds4, W, out_init=out_init, mode=mode)
    W.close()
    ref, _, _ = lay.oracle_delta(tokens=tokens, mode=mode)
    if out_init is not None:
        got = got - out_init
    if tokens is not None:
        got = got[tokens]
    return norm_max_err(got, ref)


def test_ffn_tiny_workload(ds4):
    err = _ffn_case(ds4, synth.WORKLOADS["tiny_t4"])
    assert err <= FFN_TOL, err


@pytest.mark.parametrize("T,D,F,E,k,mode", [(37, 512, 768, 8, 3, 0), (5, 256, 512, 6, 6, 1), (64, 768, 256, 4, 1, 0)])
def test_ffn_several_tiles_ragged(ds4, T, D, F, E, k, mode):
    wl = synth.Workload("mid", T=T, D=D, F=F, E=E, k=k, seed=T + D, bias=("zipf", 1.0))
    err = _ffn_case(ds4, wl, mode=mode)
    assert err <= FFN_TOL, err


def test_ffn_accumulates_into_residual(ds4):
    wl = synth.Workload("res", T=7, D=256, F=256, E=5, k=2, seed=3)
    rng = np.random.default_rng(0)
    out0 = rng.standard_normal((wl.T, wl.D)).astype(np.float32)
    err = _ffn_case(ds4, wl, out_init=out0)
    assert err <= FFN_TOL, err


def test_ffn_deterministic(ds4):
    wl = synth.Workload("det", T=40, D=512, F=512, E=16, k=4, seed=9, bias=("zipf", 1.0))
    lay = Layer(wl, quantized=False)
    W = lay.upload(ds4)
    a = lay.run(ds4, W)
    b = lay.run(ds4, W)
    W.close()
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("name", ["decode_t1", "decode_t32", "prefill_t2048", "prefill_t8192_d7168"])
def test_ffn_full_size_sampled(ds4, name):
    """Every workload at its full size, in the call the benchmark times: all tokens of the decode
    workloads; for the prefill chunks, tokens at 64 column positions of the largest group's
    256-token tiles and at both ends of its ragged last tile, tokens of one-token, small and mid
    groups, and tied tokens (helpers.sample_tokens)."""
    wl = synth.WORKLOADS[name]
    lay = Layer(wl, quantized=False)
    tokens = None if wl.T <= 32 else sample_tokens(lay.L, wl.k)
    W = lay.upload(ds4)
    got = lay.run(ds4, W)
    W.close()
    ref, _, _ = lay.oracle_delta(tokens=tokens)
    err = norm_max_err(got if tokens is None else got[tokens], ref)
    assert err <= FFN_TOL, err


# ---------------------------------------------------------------- the tensor-core path

@pytest.mark.parametrize("T,D,F,E,k,shared", [(4, 256, 256, 8, 2, True), (37, 512, 768, 8, 3, True),
                                              (600, 256, 512, 4, 2, False), (300, 768, 256, 6, 4, True)])
def test_ffn_tensor_core_path_forced(ds4, T, D, F, E, k, shared):
    """Every group (and the shared expert) on tcgen05: several M tiles, N tiles and a ragged tail."""
    wl = synth.Workload("tc", T=T, D=D, F=F, E=E, k=k, seed=T + F, bias=("zipf", 1.0), shared=shared)
    err = _ffn_case(ds4, wl, gemm_min=1)
    assert err <= FFN_TOL, err


@pytest.mark.parametrize("T,D,F,E,k,shared,fmt", [(300, 1024, 512, 6, 4, True, "q2"), (37, 512, 768, 8, 3, True, "q2"),
                                                  (600, 512, 512, 4, 2, False, "q2"), (70, 768, 512, 6, 4, True, "q2"),
                                                  (130, 1024, 512, 8, 4, True, "q4")])
def test_ffn_tensor_core_cta_pairs(ds4, T, D, F, E, k, shared, fmt):
    """The tensor-core kernels on CTA pairs (cta_group::2: one MMA over two CTAs' shared memory,
    256 weight rows, each CTA holding half of the token tile) against the oracle, and equal to
    the single-CTA kernels bit for bit (every output element is accumulated in the same order).
    d_model 768 takes pairs for the first GEMM only (the down GEMM needs a multiple of 512)."""
    import torch
    wl = synth.Workload("pair", T=T, D=D, F=F, E=E, k=k, seed=T + D, bias=("zipf", 1.0), shared=shared)
    L, x = synth.draw_inputs(wl)
    if fmt == "q4":
        gate, up, down = synth.random_q4_expert_blobs(wl)
    else:
        gate, up, down = synth.random_expert_blobs(wl)
    sh = synth.shared_weights(wl.seed, D, F) if shared else None
    W = ds4.ds4moe_weights_create(gate, up, down, D, F, shared=sh, max_tokens=T, max_k=k, fmt=fmt)
    ds4.ds4moe_set_option(W, ds4.DS4MOE_OPT_GEMM_MIN_TOKENS, 1)
    ds4.ds4moe_set_option(W, ds4.DS4MOE_OPT_SHARED_GEMM_MIN_TOKENS, 1)
    xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    Ld = torch.from_numpy(L).cuda()
    outs = []
    for pairs in (0, 1, 1):
        ds4.ds4moe_set_option(W, ds4.DS4MOE_OPT_GEMM_PAIRS, pairs)
        out = torch.zeros((T, D), dtype=torch.float32, device="cuda")
        ds4.ds4moe_expert_ffn(xd, W, Ld, k, out)
        assert ds4.ds4moe_last_status(W) == 0
        outs.append(out.cpu().numpy())
    W.close()
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))
    assert np.array_equal(outs[1].view(np.uint32), outs[2].view(np.uint32))
    ref, _, _ = oracle.moe_ffn(x, L, k, gate, up, down, D, F, shared=sh, fmt=fmt)
    assert norm_max_err(outs[1], ref) <= FFN_TOL


def test_ffn_mixed_gemv_and_tensor_core_groups(ds4):
    wl = synth.Workload("mix", T=300, D=512, F=512, E=16, k=4, seed=17, bias=("zipf", 1.2))
    L, _ = synth.draw_inputs(wl)
    counts = np.bincount(oracle.route(L, wl.k)[0].reshape(-1), minlength=wl.E)
    assert (counts >= 33).any() and ((counts > 0) & (counts < 33)).any()
    err = _ffn_case(ds4, wl)   # default thresholds: both paths in one call
    assert err <= FFN_TOL, err


@pytest.mark.parametrize("case", ["x", "h", "h_shared", "h_pairs", "h_shared_small"])
def test_ffn_tensor_core_fp16_overflow_is_recomputed(ds4, case):
    """Values beyond fp16's range on the tensor-core path (a bf16 token of 1e5, or tokens whose
    SwiGLU h exceeds 65504) flag their group (or the shared expert); the call recomputes it in
    fp32 on the GEMV kernels and the result matches the oracle, with a clean status."""
    import torch
    shared = case in ("h_shared", "h_pairs", "h_shared_small")
    wl = synth.Workload("ovf", T=40, D=512, F=256, E=4, k=2, seed=5, shared=shared)
    lay = Layer(wl, quantized=False)
    xf = (lay.x.astype(np.uint32) << 16).view(np.float32).copy()
    if case == "x":
        xf[3, 7] = 1e5                      # beyond fp16
    else:
        xf[5, :16] = 30000.0                # fits fp16, but h = silu(v) u is far beyond it
    lay.x = synth.f32_to_bf16_bits(xf)
    W = lay.upload(ds4)
    if case != "h_shared_small":  # (default thresholds: routed groups on the small-group kernels and
        # the shared expert's gate/up on its warp-MMA kernel, its down on the tensor cores)
        ds4.ds4moe_set_option(W, ds4.DS4MOE_OPT_GEMM_MIN_TOKENS, 1)
        ds4.ds4moe_set_option(W, ds4.DS4MOE_OPT_SHARED_GEMM_MIN_TOKENS, 1)
    if case == "h_pairs":
        ds4.ds4moe_set_option(W, ds4.DS4MOE_OPT_GEMM_PAIRS, 1)
    got = lay.run(ds4, W)                   # asserts a clean status
    again = lay.run(ds4, W)
    W.close()
    assert np.array_equal(got.view(np.uint32), again.view(np.uint32))
    ref, _, _ = lay.oracle_delta()
    assert norm_max_err(got, ref) <= FFN_TOL, norm_max_err(got, ref)
    if case != "x":
        assert np.max(np.abs(ref)) > 65504.0   # the overflow was real


# ---------------------------------------------------------------- the small-group kernels

# (T, D, F, E, k, shared, small_groups, tokens): groups of up to ~30 tokens (chunks of 6), odd
# block counts (D = 2304: 9 blocks per row, F = 1280: 80 gate/up tiles), the bf16 shared expert on
# tcgen05 beside them, and the same layer on the fused GEMV kernels for comparison.
@pytest.mark.parametrize("T,D,F,E,k,shared,sg,tokens", [
    (4, 256, 256, 8, 2, False, 1, None),
    (9, 512, 256, 4, 2, True, 1, None),
    (45, 1024, 512, 6, 4, True, 1, None),
    (45, 1024, 512, 6, 4, True, 0, None),
    (13, 2304, 1280, 16, 5, False, 1, None),
    (48, 4096, 2048, 24, 6, True, 1, [0, 17, 47]),
])
def test_small_group_kernels_match_oracle(ds4, T, D, F, E, k, shared, sg, tokens):
    wl = synth.Workload("sg", T=T, D=D, F=F, E=E, k=k, seed=T + D + F, bias=("normal", 0.5), shared=shared)
    lay = Layer(wl, quantized=D * F <= 1024 * 512)
    W = lay.upload(ds4)
    ds4.ds4moe_set_option(W, ds4.DS4MOE_OPT_SMALL_GROUPS, sg)
    got = lay.run(ds4, W)
    again = lay.run(ds4, W)
    W.close()
    assert np.array_equal(got.view(np.uint32), again.view(np.uint32))   # deterministic
    ref, _, _ = lay.oracle_delta(tokens=tokens)
    err = norm_max_err(got if tokens is None else got[tokens], ref)
    assert err <= FFN_TOL, err


def test_small_groups_beside_tensor_core_groups(ds4):
    # more than 64 tokens: groups of at least 7 tokens on tcgen05, the rest on the small-group kernels
    wl = synth.Workload("sgmix", T=200, D=1024, F=512, E=32, k=4, seed=23, bias=("zipf", 1.0))
    L, _ = synth.draw_inputs(wl)
    counts = np.bincount(oracle.route(L, wl.k)[0].reshape(-1), minlength=wl.E)
    assert (counts >= 7).any() and ((counts > 0) & (counts < 7)).any()
    err = _ffn_case(ds4, wl, quantized=False)
    assert err <= FFN_TOL, err


def test_small_groups_at_one_token_without_the_fused_kernel(ds4):
    # T = 1 on the separate kernels: the routed experts on the small-group kernels, the shared
    # expert on the single-token decode kernels
    wl = synth.Workload("sg1", T=1, D=2048, F=2048, E=64, k=6, seed=31, shared=True)
    lay = Layer(wl, quantized=False)
    W = lay.upload(ds4)
    ds4.ds4moe_set_option(W, ds4.DS4MOE_OPT_SINGLE_STEP, 0)
    got = lay.run(ds4, W)
    W.close()
    ref, _, _ = lay.oracle_delta()
    assert norm_max_err(got, ref) <= FFN_TOL


# ---------------------------------------------------------------- the single-token kernel

# (D, E, k, shared, mode, fused): the fused kernel covers F == 2048, D <= 4096; D = 7168 takes
# the separate single-token kernels. D = 3072 leaves half of the second x half empty.
@pytest.mark.parametrize("D,E,k,shared,mode,fused", [
    (4096, 256, 8, True, 0, True), (4096, 256, 8, True, 1, True), (2048, 64, 6, True, 1, True),
    (1024, 16, 8, False, 0, True), (3072, 32, 4, True, 1, True), (4096, 300, 1, False, 1, True),
    (4096, 8, 8, True, 0, True), (2048, 8, 8, False, 1, True), (7168, 64, 6, True, 1, False)])
def test_single_token_kernel_matches_oracle(ds4, D, E, k, shared, mode, fused):
    wl = synth.Workload("one", T=1, D=D, F=2048, E=E, k=k, seed=D + E, shared=shared)
    lay = Layer(wl, quantized=False)
    W = lay.upload(ds4)
    before = ds4.ds4moe_get_stats(W)
    got = lay.run(ds4, W, mode=mode)
    after = ds4.ds4moe_get_stats(W)
    W.close()
    assert (after["launches"] - before["launches"] == 1) == fused
    ref, _, _ = lay.oracle_delta(mode=mode)
    err = norm_max_err(got, ref)
    assert err <= FFN_TOL, err


@pytest.mark.parametrize("mode", [0, 1])
def test_single_token_kernel_breaks_ties_like_the_oracle(ds4, mode):
    # many equal logits (and -0 next to +0): the selection must take the lower expert index
    wl = synth.Workload("ties", T=1, D=1024, F=2048, E=64, k=8, seed=77, shared=False)
    lay = Layer(wl, quantized=False)
    vals = np.array([-1.0, 0.0, -0.0, 0.5, 2.0], np.float32)
    lay.L = vals[np.random.default_rng(5).integers(0, len(vals), size=(1, wl.E))]
    W = lay.upload(ds4)
    before = ds4.ds4moe_get_stats(W)["launches"]
    got = lay.run(ds4, W, mode=mode)
    assert ds4.ds4moe_get_stats(W)["launches"] - before == 1  # the fused kernel ran
    W.close()
    ref, _, _ = lay.oracle_delta(mode=mode)
    assert norm_max_err(got, ref) <= FFN_TOL


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("E", [64, 300])   # the fused kernel's two top-k routines (E <= 256, above)
def test_single_token_kernel_nan_and_infinite_logits(ds4, mode, E):
    """The fused kernel's own top-k and gate weights on NaN, +inf and -inf logits, through the
    whole layer: a different selection or a NaN weight would change the output far beyond the
    tolerance (every expert's blocks differ)."""
    wl = synth.Workload("nan1", T=1, D=1024, F=2048, E=E, k=8, seed=91 + E, shared=True)
    lay = Layer(wl, quantized=False, experts=range(E))
    W = lay.upload(ds4)
    rng = np.random.default_rng(E)
    for row in _SPECIAL_ROWS:
        L = np.full((1, E), -np.inf, np.float32)
        L[0, :8] = row
        perm = rng.permutation(E)                # the special values at scattered experts
        lay.L = L[:, np.argsort(perm)]
        before = ds4.ds4moe_get_stats(W)["launches"]
        got = lay.run(ds4, W, mode=mode)
        assert ds4.ds4moe_get_stats(W)["launches"] - before == 1   # the fused kernel ran
        ref, idx, g = lay.oracle_delta(mode=mode)
        assert np.all(np.isfinite(g)) and np.all(np.isfinite(got))
        assert norm_max_err(got, ref) <= FFN_TOL, (row, norm_max_err(got, ref))
    W.close()


@pytest.mark.parametrize("T", [1, 3, 32])
@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("E", [64, 300])   # the route kernel's register layouts of 2 and 10 logits per lane
def test_separate_kernels_route_nan_and_infinite_logits_like_the_oracle(ds4, T, mode, E):
    """Without the fused kernel (the route, grouping and expert kernels): top-k and gate weights on
    NaN, +inf and -inf logits, through the whole layer, each token a different special row among
    -inf logits."""
    wl = synth.Workload("nang", T=T, D=1024, F=2048, E=E, k=8, seed=93 + T, shared=True)
    lay = Layer(wl, quantized=False, experts=range(E))
    W = lay.upload(ds4)
    ds4.ds4moe_set_option(W, ds4.DS4MOE_OPT_SINGLE_STEP, 0)
    rng = np.random.default_rng(T + E)
    L = np.full((T, E), -np.inf, np.float32)
    for t in range(T):
        L[t, :8] = _SPECIAL_ROWS[t % len(_SPECIAL_ROWS)]
        L[t] = L[t, np.argsort(rng.permutation(E))]   # the special values at scattered experts
    lay.L = L
    got = lay.run(ds4, W, mode=mode)
    W.close()
    ref, idx, g = lay.oracle_delta(mode=mode)
    assert np.all(np.isfinite(g)) and np.all(np.isfinite(got))
    assert norm_max_err(got, ref) <= FFN_TOL


def test_single_token_kernel_equals_separate_kernels_and_is_deterministic(ds4):
    import torch
    wl = synth.WORKLOADS["decode_t1"]
    lay = Layer(wl, quantized=False)
    W = lay.upload(ds4)
    a = lay.run(ds4, W)
    b = lay.run(ds4, W)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    ds4.ds4moe_set_option(W, ds4.DS4MOE_OPT_SINGLE_STEP, 0)
    c = lay.run(ds4, W)
    W.close()
    assert norm_max_err(a, c) <= FFN_TOL   # two valid paths, each within tolerance of the oracle


# ---------------------------------------------------------------- router logits in front of routing

def _valid_selection(sel, ref, bound):
    """Whether the expert set sel can be the top-k of some logits within bound of ref: every
    selected expert's upper end reaches every unselected expert's lower end."""
    mask = np.zeros(ref.size, bool)
    mask[sel] = True
    if mask.all():
        return True
    return np.min(ref[mask] + bound[mask]) >= np.max(ref[~mask] - bound[~mask])


def _router_on_tensor_cores(T, E):
    return T >= 64 and E % 128 == 0


@pytest.mark.parametrize("T,D,E,bias", [(1, 4096, 256, True), (37, 512, 64, False), (4, 256, 8, True),
                                        (130, 1024, 128, True), (3, 7168, 256, False), (64, 256, 128, False),
                                        (200, 4096, 256, False), (321, 7168, 256, True), (63, 2048, 256, True)])
def test_router_logits_within_the_fp32_bound_and_the_selection_from_them(ds4, T, D, E, bias):
    """The device's fp32 logits against the exact (fp64) sum: within the fp32 summation bound of
    the order the call takes (CUDA cores below 64 tokens, the tensor cores' 16-column blocks from 64
    tokens on). The selection is then exact wherever the k-th and (k+1)-th exact logits are further
    apart than their bounds allow to swap, and a valid top-k within the bounds elsewhere; the
    selection from the device's own logits is the oracle's selection from the same fp32 values,
    bit for bit."""
    import torch
    from oracle.router import fp32_bound, router_logits, tensor_core_depth
    rng = np.random.default_rng(T + D + E)
    x = synth.f32_to_bf16_bits(rng.standard_normal((T, D)).astype(np.float32))
    w = synth.f32_to_bf16_bits((0.02 * rng.standard_normal((E, D))).astype(np.float32))
    b = (0.1 * rng.standard_normal(E)).astype(np.float32) if bias else None
    ref = router_logits(x, w, b)
    bound = fp32_bound(x, w, b, depth=tensor_core_depth(D) if _router_on_tensor_cores(T, E) else None)
    xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    wd = torch.from_numpy(w.view(np.int16)).cuda().view(torch.bfloat16)
    bd = torch.from_numpy(b).cuda() if bias else None
    got = ds4.ds4moe_router_logits(xd, wd, bd)
    assert ds4.ds4moe_router_last_status() == 0
    g = got.cpu().numpy()
    assert np.all(np.abs(g.astype(np.float64) - ref) <= bound)
    again = ds4.ds4moe_router_logits(xd, wd, bd).cpu().numpy()
    assert np.array_equal(again.view(np.uint32), g.view(np.uint32))  # the same bits on every run
    k = min(8, E)
    idx, _ = ds4.ds4moe_route(got, k)
    idx = idx.cpu().numpy()
    assert np.array_equal(idx, oracle.route(g, k)[0])
    n_exact = 0
    for t in range(T):
        o = np.lexsort((np.arange(E), -ref[t]))
        if k < E and ref[t, o[k - 1]] - ref[t, o[k]] > bound[t, o[k - 1]] + bound[t, o[k]]:
            assert set(idx[t]) == set(o[:k]), t
            n_exact += 1
        assert _valid_selection(idx[t], ref[t], bound[t]), t
    assert n_exact >= (T + 1) // 2 or k == E


def test_router_logits_follow_the_documented_order(ds4):
    """The library's documented summation order is a property of its kernel: lane 0's columns 0
    and 1 add 2^30 and -2^30 before any other term, so the 1s that the other 31 lanes carry survive
    (the logit is exactly 31, the exact sum); an order that adds a 1 to 2^30 first loses it."""
    import torch
    D, E = 256, 8
    x = np.zeros((1, D), np.float32)
    w = np.zeros((E, D), np.float32)
    x[0, 0], x[0, 1] = 2.0 ** 15, 2.0 ** 15
    w[:, 0], w[:, 1] = 2.0 ** 15, -(2.0 ** 15)
    x[0, 8:D:8] = 1.0
    w[:, 8:D:8] = 1.0
    xd = torch.from_numpy(synth.f32_to_bf16_bits(x).view(np.int16)).cuda().view(torch.bfloat16)
    wd = torch.from_numpy(synth.f32_to_bf16_bits(w).view(np.int16)).cuda().view(torch.bfloat16)
    got = ds4.ds4moe_router_logits(xd, wd).cpu().numpy()
    assert np.all(got == 31.0)


def test_router_logits_tensor_core_order(ds4):
    """From 64 tokens on, 16-column blocks are added in increasing order into one fp32 accumulator:
    2^30 (column 0), then 1 (column 16, lost: the fp32 spacing at 2^30 is 128), then -2^30 (column
    32) leaves exactly 0; an order that cancels the large terms first keeps the 1 (the CUDA-core
    order of fewer tokens gives 1)."""
    import torch
    D, E = 256, 128
    w = np.zeros((E, D), np.float32)
    w[:, 0], w[:, 16], w[:, 32] = 2.0 ** 15, 1.0, -(2.0 ** 15)
    wd = torch.from_numpy(synth.f32_to_bf16_bits(w).view(np.int16)).cuda().view(torch.bfloat16)
    for T, want in ((64, 0.0), (200, 0.0), (63, 1.0)):
        x = np.zeros((T, D), np.float32)
        x[:, 0], x[:, 16], x[:, 32] = 2.0 ** 15, 1.0, 2.0 ** 15
        xd = torch.from_numpy(synth.f32_to_bf16_bits(x).view(np.int16)).cuda().view(torch.bfloat16)
        got = ds4.ds4moe_router_logits(xd, wd).cpu().numpy()
        assert np.all(got == want), (T, np.unique(got))


def test_layer_from_hidden_states(ds4):
    # router in front: the logits come from the router on the device, the oracle takes its own
    import torch
    from oracle.router import fp32_bound, router_logits
    wl = synth.Workload("hid", T=1, D=4096, F=2048, E=256, k=8, seed=41, shared=True)
    rng = np.random.default_rng(41)
    lay = Layer(wl, quantized=False)
    w = synth.f32_to_bf16_bits((0.02 * rng.standard_normal((wl.E, wl.D))).astype(np.float32))
    b = (0.1 * rng.standard_normal(wl.E)).astype(np.float32)
    exact = router_logits(lay.x, w, b)
    lay.L = exact.astype(np.float32)
    # the selection is unambiguous: the 8th and 9th exact logits lie further apart than the fp32 bound
    o = np.sort(exact[0])[::-1]
    assert o[wl.k - 1] - o[wl.k] > 2 * np.max(fp32_bound(lay.x, w, b))
    # the layer's random blobs were made for the experts of the drawn logits: cover these too
    lay.gate, lay.up, lay.down = synth.random_expert_blobs(wl, np.unique(oracle.route(lay.L, wl.k)[0]))
    W = lay.upload(ds4)
    x = torch.from_numpy(lay.x.view(np.int16)).cuda().view(torch.bfloat16)
    logits = ds4.ds4moe_router_logits(x, torch.from_numpy(w.view(np.int16)).cuda().view(torch.bfloat16),
                                      torch.from_numpy(b).cuda())
    out = torch.zeros((wl.T, wl.D), dtype=torch.float32, device="cuda")
    ds4.ds4moe_expert_ffn(x, W, logits, wl.k, out)
    assert ds4.ds4moe_last_status(W) == 0
    W.close()
    ref, _, _ = lay.oracle_delta()
    assert norm_max_err(out.cpu().numpy(), ref) <= FFN_TOL


def test_single_token_kernel_bounded_wait_runs_out_and_the_handle_recovers(ds4):
    # the grid barrier waits for an arrival nothing sends: the wait gives up (about 2 s), every
    # CTA leaves through its abort path, the status word says so, and the next call is normal
    import torch
    wl = synth.Workload("wait_test", T=1, D=512, F=2048, E=16, k=4, seed=61, shared=True)
    lay = Layer(wl, quantized=False)
    W = lay.upload(ds4)
    ds4.ds4moe_set_option(W, ds4.DS4MOE_OPT_WAIT_TEST, 1)
    x = torch.from_numpy(lay.x.view(np.int16)).cuda().view(torch.bfloat16)
    out = torch.zeros((1, wl.D), dtype=torch.float32, device="cuda")
    before = ds4.ds4moe_get_stats(W)["launches"]
    ds4.ds4moe_expert_ffn(x, W, torch.from_numpy(lay.L).cuda(), wl.k, out)
    assert ds4.ds4moe_get_stats(W)["launches"] - before == 1   # the fused kernel took the call
    assert ds4.ds4moe_last_status(W) == ds4.DS4MOE_ETIMEOUT
    ds4.ds4moe_set_option(W, ds4.DS4MOE_OPT_WAIT_TEST, 0)
    got = lay.run(ds4, W)                                       # asserts a clean status
    W.close()
    ref, _, _ = lay.oracle_delta()
    assert norm_max_err(got, ref) <= FFN_TOL
