"""The 4-bit variant on the GPU through the C ABI: device dequantisation bit-exact against the
oracle's Q4_K-style dequantiser, and the expert FFN of q4 handles within the normalised max
error 2e-3 of the oracle's fp64 FFN, at one token, decode micro-batches and a batch whose
shared expert runs on the tensor cores."""
import numpy as np
import pytest

import oracle
import synth
from helpers import FFN_TOL, norm_max_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ds4():
    import torch
    import bit_quantized_routed_gb300 as m
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    m.build()
    return m


def test_q4_device_dequant_bitexact(ds4):
    import torch
    wl = synth.Workload("q4_dq", T=1, D=768, F=512, E=3, k=2, seed=31, shared=False)
    gate, up, down = synth.random_q4_expert_blobs(wl)
    W = ds4.ds4moe_weights_create(gate, up, down, wl.D, wl.F, max_tokens=1, max_k=2, fmt="q4")
    for e in range(wl.E):
        for m, blob, (rows, cols) in ((ds4.DS4MOE_GATE, gate[e], (wl.F, wl.D)), (ds4.DS4MOE_UP, up[e], (wl.F, wl.D)),
                                      (ds4.DS4MOE_DOWN, down[e], (wl.D, wl.F))):
            dst = torch.empty((rows, cols), dtype=torch.float32, device="cuda")
            ds4.ds4moe_weights_dequantize(W, e, m, dst_f32=dst)
            torch.cuda.synchronize()
            ref = oracle.dequant_q4k(blob, rows, cols)
            assert np.array_equal(dst.cpu().numpy().view(np.uint32), ref.view(np.uint32)), (e, m)
    h16 = torch.empty((wl.F, wl.D), dtype=torch.float16, device="cuda")
    with pytest.raises(ds4.Ds4moeError) as ei:
        ds4.ds4moe_weights_dequantize(W, 0, ds4.DS4MOE_GATE, dst_f16=h16)
    assert ei.value.status == ds4.DS4MOE_EUNSUPPORTED
    W.close()


@pytest.mark.parametrize("T,D,F,E,k,shared,mode,quantized", [
    (1, 1024, 512, 16, 4, True, 0, False),
    (1, 4096, 2048, 32, 8, True, 0, True),     # the decode shape, host-quantised N(0, 0.02) experts
    (1, 7168, 512, 16, 4, True, 1, False),     # d_model 7168: two ring stages, four warps per shared row
    (1, 256, 256, 8, 2, False, 0, False),      # the smallest shape, no shared expert
    (5, 512, 768, 16, 4, True, 1, False),
    (40, 512, 512, 24, 4, False, 0, False),
    (100, 512, 512, 24, 4, True, 0, False),    # shared expert on the tensor cores, routed on the GEMV
])
def test_q4_ffn_matches_oracle(ds4, T, D, F, E, k, shared, mode, quantized):
    import torch
    wl = synth.Workload("q4_ffn", T=T, D=D, F=F, E=E, k=k, seed=40 + T, shared=shared)
    L, x = synth.draw_inputs(wl)
    if quantized:
        idx, _ = oracle.route(L, k, mode)
        used = set(int(e) for e in np.unique(idx))
        z = np.zeros(F * D // 256 * 144, np.uint8)
        gate, up, down = [z] * E, [z] * E, [z] * E
        for e in used:
            gate[e] = ds4.ds4moe_quantize_q4k(synth.expert_weight(wl.seed, e, synth.GATE, F, D))
            up[e] = ds4.ds4moe_quantize_q4k(synth.expert_weight(wl.seed, e, synth.UP, F, D))
            down[e] = ds4.ds4moe_quantize_q4k(synth.expert_weight(wl.seed, e, synth.DOWN, D, F))
    else:
        gate, up, down = synth.random_q4_expert_blobs(wl)
    sh = synth.shared_weights(wl.seed, D, F) if shared else None
    W = ds4.ds4moe_weights_create(gate, up, down, D, F, shared=sh, max_tokens=T, max_k=k, fmt="q4")
    xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    out = torch.zeros((T, D), dtype=torch.float32, device="cuda")
    ds4.ds4moe_expert_ffn(xd, W, torch.from_numpy(L).cuda(), k, out, gate_mode=mode)
    assert ds4.ds4moe_last_status(W) == 0
    W.close()
    tok = None if T <= 40 else np.arange(0, T, 7)
    ref, _, _ = oracle.moe_ffn(x, L, k, gate, up, down, D, F, shared=sh, mode=mode, tokens=tok, fmt="q4")
    got = out.cpu().numpy() if tok is None else out.cpu().numpy()[tok]
    assert norm_max_err(got, ref) <= FFN_TOL


def test_q4_handle_is_refused_by_the_allocation_free_entry(ds4):
    import torch
    wl = synth.Workload("q4_static", T=2, D=256, F=256, E=4, k=2, seed=3, shared=False)
    gate, up, down = synth.random_q4_expert_blobs(wl)
    W = ds4.ds4moe_weights_create(gate, up, down, wl.D, wl.F, max_tokens=2, max_k=2, fmt="q4")
    L, x = synth.draw_inputs(wl)
    xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    out = torch.zeros((2, wl.D), dtype=torch.float32, device="cuda")
    with pytest.raises(ds4.Ds4moeError) as ei:
        ds4.ds4moe_expert_ffn_static(xd, W, torch.from_numpy(L).cuda(), 2, out)
    assert ei.value.status == ds4.DS4MOE_EUNSUPPORTED
    W.close()
