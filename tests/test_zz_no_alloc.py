"""The allocation-free entry point, ds4moe_expert_ffn_static, through the C ABI.

It serves callers that cannot allocate device memory while they run (a plug-in whose host
framework owns every device allocation, a serving loop that must not call cudaMalloc): its
intermediates live in the library's static device region. Its output must match the regular
entry point, ds4moe_expert_ffn, and the oracle, on the same inputs, on two calls in a row (the
region keeps the previous call's contents, which must not leak into the next result); calls
beyond the region's size are refused. This file is named to be collected last."""
import numpy as np
import pytest

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


def _inputs(lay):
    import torch
    x = torch.from_numpy(lay.x.view(np.int16)).cuda().view(torch.bfloat16)
    logits = torch.from_numpy(lay.L).cuda()
    return x, logits


@pytest.mark.parametrize("wl", [
    synth.Workload("small", T=5, D=512, F=768, E=16, k=4, seed=21, bias=("zipf", 1.0)),
    synth.WORKLOADS["decode_t1"],
    synth.WORKLOADS["decode_t32"].replace(T=8),
])
def test_static_entry_matches_expert_ffn(ds4, wl):
    import torch
    lay = Layer(wl, quantized=False)
    W = lay.upload(ds4)
    x, logits = _inputs(lay)
    ref = torch.zeros((wl.T, wl.D), dtype=torch.float32, device="cuda")
    ds4.ds4moe_expert_ffn(x, W, logits, wl.k, ref)
    ref = ref.cpu().numpy()
    exact, _, _ = lay.oracle_delta()
    for _ in range(2):
        out = torch.zeros((wl.T, wl.D), dtype=torch.float32, device="cuda")
        ds4.ds4moe_expert_ffn_static(x, W, logits, wl.k, out)
        assert ds4.ds4moe_last_status(W) == 0
        got = out.cpu().numpy()
        assert norm_max_err(got, ref) <= FFN_TOL, norm_max_err(got, ref)      # the regular entry point
        assert norm_max_err(got, exact) <= FFN_TOL, norm_max_err(got, exact)  # and the oracle itself
    W.close()


def test_static_entry_size_limit_at_d_model_7168(ds4):
    """At top-8 with d_model 7168 and d_ff 2048 the region holds 9 tokens (9 x 9 rows of
    (7168 + 2048) fp32 values, 2.99 MB) and not 10 (3.32 MB): 9 runs and matches the oracle, 10 is
    refused with EINVAL before anything is launched."""
    import torch
    wl = synth.Workload("lim", T=10, D=7168, F=2048, E=16, k=8, seed=29, shared=False)
    lay = Layer(wl, quantized=False)
    W = lay.upload(ds4)
    x, logits = _inputs(lay)
    out = torch.zeros((9, wl.D), dtype=torch.float32, device="cuda")
    ds4.ds4moe_expert_ffn_static(x[:9], W, logits[:9], wl.k, out)
    assert ds4.ds4moe_last_status(W) == 0
    ref, _, _ = lay.oracle_delta(tokens=list(range(9)))
    assert norm_max_err(out.cpu().numpy(), ref) <= FFN_TOL
    out10 = torch.zeros((10, wl.D), dtype=torch.float32, device="cuda")
    with pytest.raises(ds4.Ds4moeError) as ei:
        ds4.ds4moe_expert_ffn_static(x, W, logits, wl.k, out10)
    assert ei.value.status == ds4.DS4MOE_EINVAL
    torch.cuda.synchronize()
    assert float(out10.abs().max()) == 0.0
    W.close()


def test_static_entry_rejects_calls_beyond_its_region(ds4):
    import torch
    wl = synth.WORKLOADS["decode_t32"]   # 32 tokens x 9 rows x (4096 + 2048) x 4 B > 3 MiB
    lay = Layer(wl.replace(T=1), quantized=False)
    W = lay.upload(ds4, max_tokens=wl.T)
    x = torch.zeros((wl.T, wl.D), dtype=torch.bfloat16, device="cuda")
    logits = torch.zeros((wl.T, wl.E), dtype=torch.float32, device="cuda")
    out = torch.zeros((wl.T, wl.D), dtype=torch.float32, device="cuda")
    with pytest.raises(ds4.Ds4moeError) as ei:
        ds4.ds4moe_expert_ffn_static(x, W, logits, wl.k, out)
    assert ei.value.status == ds4.DS4MOE_EINVAL
    assert float(out.abs().max()) == 0.0   # nothing was launched
    W.close()
