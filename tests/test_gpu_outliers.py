"""Activations with outlier columns, on every path that quantises them, against the oracle.

Hidden states of large language models carry a few channels hundreds of times larger than the
rest. The kernels that take x as int16 (the fused single-token kernel: one power-of-two scale per
1024-column quarter; the small-group kernels and the 4-bit variant's GEMV: one per token row) lose
the small channels' low bits to such a column, and the tensor-core path holds x in fp16. Each path
gets x ~ N(0, 1) with four columns at 300-1000 times that, an all-zero token beside a token scaled
by 16, and is checked against the oracle's fp64 FFN at the normalised max error 2e-3."""
import numpy as np
import pytest

import oracle
import synth
from helpers import FFN_TOL, Layer, norm_max_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ds4():
    import torch
    import bit_quantized_routed_gb300 as m
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    m.build()
    return m


def outlier_x(x_bits, seed):
    """x with four outlier columns (300-1000 times the rest, either sign); with two or more tokens,
    token 0 all zeros and token 1's ordinary columns scaled by 16 (a large token beside a zero one;
    its outlier columns as the others')."""
    rng = np.random.default_rng(seed)
    x = (x_bits.astype(np.uint32) << 16).view(np.float32).copy()
    T, D = x.shape
    if T >= 2:
        x[1] *= 16.0
    cols = rng.choice(D, 4, replace=False)
    x[:, cols] = (rng.uniform(300.0, 1000.0, (T, 4)) * rng.choice([-1.0, 1.0], (T, 4))).astype(np.float32)
    if T >= 2:
        x[0] = 0.0
    return synth.f32_to_bf16_bits(x)


def _check(ds4, lay, W, mode=0, tokens=None, expect_launches=None):
    before = ds4.ds4moe_get_stats(W)["launches"]
    got = lay.run(ds4, W, mode=mode)
    if expect_launches is not None:
        assert ds4.ds4moe_get_stats(W)["launches"] - before == expect_launches
    ref, _, _ = lay.oracle_delta(tokens=tokens, mode=mode)
    err = norm_max_err(got if tokens is None else got[tokens], ref)
    assert err <= FFN_TOL, err
    return got


@pytest.mark.parametrize("mode", [0, 1])
def test_fused_single_token_kernel(ds4, mode):
    wl = synth.Workload("out1", T=1, D=4096, F=2048, E=64, k=8, seed=71, shared=True)
    lay = Layer(wl, quantized=False)
    lay.x = outlier_x(lay.x, 1)
    W = lay.upload(ds4)
    _check(ds4, lay, W, mode=mode, expect_launches=1)
    # an all-zero token: the expert FFN of 0 is exactly 0
    lay.x = np.zeros_like(lay.x)
    got = lay.run(ds4, W, mode=mode)
    W.close()
    assert np.all(got == 0.0)


def test_small_group_kernels(ds4):
    wl = synth.Workload("out_sg", T=48, D=2048, F=1024, E=24, k=6, seed=72, bias=("normal", 0.5), shared=True)
    lay = Layer(wl, quantized=False)
    lay.x = outlier_x(lay.x, 2)
    W = lay.upload(ds4)
    got = _check(ds4, lay, W)
    W.close()
    assert np.all(got[0] == 0.0)       # the zero token


def test_tensor_core_path(ds4):
    wl = synth.Workload("out_tc", T=300, D=768, F=512, E=6, k=4, seed=73, bias=("zipf", 1.0), shared=True)
    lay = Layer(wl, quantized=False)
    lay.x = outlier_x(lay.x, 3)
    W = lay.upload(ds4)
    ds4.ds4moe_set_option(W, ds4.DS4MOE_OPT_GEMM_MIN_TOKENS, 1)
    ds4.ds4moe_set_option(W, ds4.DS4MOE_OPT_SHARED_GEMM_MIN_TOKENS, 1)
    got = _check(ds4, lay, W)
    W.close()
    assert np.all(got[0] == 0.0)


def test_mixed_prefill_call(ds4):
    # the default dispatch above 64 tokens: small groups, tensor-core groups and the shared expert
    wl = synth.Workload("out_mix", T=200, D=1024, F=512, E=32, k=4, seed=74, bias=("zipf", 1.0), shared=True)
    lay = Layer(wl, quantized=False)
    lay.x = outlier_x(lay.x, 4)
    W = lay.upload(ds4)
    _check(ds4, lay, W)
    W.close()


@pytest.mark.parametrize("T", [1, 40])
def test_q4_gemv(ds4, T):
    import torch
    wl = synth.Workload("out_q4", T=T, D=4096 if T == 1 else 1024, F=2048 if T == 1 else 512, E=32, k=8,
                        seed=75 + T, shared=True)
    L, x = synth.draw_inputs(wl)
    x = outlier_x(x, 5 + T)
    gate, up, down = synth.random_q4_expert_blobs(wl)
    sh = synth.shared_weights(wl.seed, wl.D, wl.F)
    W = ds4.ds4moe_weights_create(gate, up, down, wl.D, wl.F, shared=sh, max_tokens=T, max_k=wl.k, fmt="q4")
    xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    out = torch.zeros((T, wl.D), dtype=torch.float32, device="cuda")
    ds4.ds4moe_expert_ffn(xd, W, torch.from_numpy(L).cuda(), wl.k, out)
    assert ds4.ds4moe_last_status(W) == 0
    W.close()
    ref, _, _ = oracle.moe_ffn(x, L, wl.k, gate, up, down, wl.D, wl.F, shared=sh, fmt="q4")
    got = out.cpu().numpy()
    assert norm_max_err(got, ref) <= FFN_TOL
    if T >= 2:
        assert np.all(got[0] == 0.0)
