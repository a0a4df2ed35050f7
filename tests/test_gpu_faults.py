"""Failure handling on the GPU, made on the host (no kernel is made to fault or hang): a forced
device-allocation failure during handle creation, and device pointers that break the alignment
the kernels need. Each is refused with its status, leaves nothing behind, and the next call is
normal."""
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


@pytest.mark.parametrize("nth", [1, 5, 20])
def test_allocation_failure_during_creation_frees_everything(ds4, nth):
    import torch
    wl = synth.Workload("enomem", T=8, D=512, F=512, E=8, k=2, seed=3, shared=True)
    lay = Layer(wl, quantized=False)
    W = lay.upload(ds4)            # the first creation loads the module and sets up the context
    W.close()
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    ds4.ds4moe_test_fail_allocation(nth)
    with pytest.raises(ds4.Ds4moeError) as ei:
        lay.upload(ds4)
    assert ei.value.status == ds4.DS4MOE_ENOMEM
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert abs(free1 - free0) <= 2 * 2 ** 20, (free0, free1)    # nothing kept
    W = lay.upload(ds4)            # the hook fired once: the next creation is normal
    got = lay.run(ds4, W)
    W.close()
    ref, _, _ = lay.oracle_delta()
    assert norm_max_err(got, ref) <= FFN_TOL


def test_misaligned_activations_or_output_are_refused(ds4):
    import torch
    wl = synth.Workload("align", T=4, D=256, F=256, E=8, k=2, seed=4, shared=False)
    lay = Layer(wl, quantized=False)
    W = lay.upload(ds4)
    L = ds4.lib()
    xbuf = torch.from_numpy(np.concatenate([lay.x.reshape(-1), np.zeros(8, np.uint16)]).view(np.int16)).cuda()
    logits = torch.from_numpy(lay.L).cuda()
    obuf = torch.zeros(wl.T * wl.D + 4, dtype=torch.float32, device="cuda")
    s = ds4._stream()
    for xo, oo in ((1, 0), (0, 1), (4, 2)):   # x 2, 0, 8 bytes off; out 0, 4, 8 bytes off
        rc = L.ds4moe_expert_ffn(xbuf.data_ptr() + 2 * xo, W.handle, logits.data_ptr(), wl.T, wl.k, 0,
                                 obuf.data_ptr() + 4 * oo, s)
        assert rc == ds4.DS4MOE_EINVAL, (xo, oo)
    torch.cuda.synchronize()
    assert float(obuf.abs().max()) == 0.0      # nothing was launched
    assert ds4.ds4moe_last_status(W) == 0
    got = lay.run(ds4, W)                      # aligned buffers: a normal call
    W.close()
    ref, _, _ = lay.oracle_delta()
    assert norm_max_err(got, ref) <= FFN_TOL
