"""The C-ABI library on the host (no GPU needed): it loads, exports every symbol the header
declares, and its host quantisers, dequantisers and grid agree byte for byte with the
oracle's independent implementation. Device entry points are only called with arguments
that the host-side checks reject before any CUDA call."""
import os
import re

import numpy as np
import pytest

import oracle
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ds4():
    import bit_quantized_routed_gb300 as m
    m.build()
    return m


def _declared():
    hdr = open(os.path.join(ROOT, "include", "ds4moe.h")).read()
    hdr = re.sub(r"/\*.*?\*/", "", hdr, flags=re.S)
    return sorted(set(re.findall(r"\b(ds4moe_[a-z0-9_]+)\s*\(", hdr)))


def test_library_exports_every_declared_symbol(ds4):
    import ctypes
    declared = _declared()
    assert len(declared) >= 16
    L = ctypes.CDLL(ds4.LIB_PATH)
    for name in declared:
        assert hasattr(L, name), name
    assert sorted(ds4.EXPORTED) == declared


def test_sizes_and_strerror(ds4):
    assert ds4.ds4moe_q2k_bytes(4096, 2048) == 4096 * 8 * 84
    assert ds4.ds4moe_iq2_bytes(2048, 4096) == 2048 * 16 * 66
    assert ds4.ds4moe_iq2_bytes(1, 255) == 0 and ds4.ds4moe_q2k_bytes(-1, 256) == 0
    assert ds4.ds4moe_strerror(0) == "ok"
    assert "invalid" in ds4.ds4moe_strerror(1)


def test_grid_matches_oracle(ds4):
    assert np.array_equal(ds4.ds4moe_iq2_grid(), oracle.iq2_grid())


def _weights(rows, cols, seed):
    rng = np.random.default_rng(seed)
    w = (rng.standard_normal((rows, cols)) * 0.02).astype(np.float32)
    w[0, :7] = [0.0, -0.0, 1e-9, -1e-9, 0.05, -0.05, 0.0]     # zeros, tiny values
    w[1, :256] = 0.0                                           # an all-zero block
    w[2, :256] = np.float32(0.01)                              # a constant block
    w[3, 256:512] = -np.abs(w[3, 256:512])                     # all-negative block
    return w


@pytest.mark.parametrize("shape,seed", [((6, 512), 1), ((5, 768), 2)])
def test_quantizers_byte_identical_to_oracle(ds4, shape, seed):
    w = _weights(*shape, seed)
    assert np.array_equal(ds4.ds4moe_quantize_q2k(w), oracle.quantize_q2k(w))
    assert np.array_equal(ds4.ds4moe_quantize_iq2(w), oracle.quantize_iq2(w))
    assert np.array_equal(ds4.ds4moe_quantize_q4k(w), oracle.quantize_q4k(w))


def test_quantizers_byte_identical_on_expert_weights(ds4):
    w = synth.expert_weight(7, 3, synth.GATE, 16, 1024)
    assert np.array_equal(ds4.ds4moe_quantize_iq2(w), oracle.quantize_iq2(w))
    w = synth.expert_weight(7, 3, synth.DOWN, 16, 1024)
    assert np.array_equal(ds4.ds4moe_quantize_q2k(w), oracle.quantize_q2k(w))
    assert np.array_equal(ds4.ds4moe_quantize_q4k(w), oracle.quantize_q4k(w))


def test_host_dequantizers_match_oracle_bitwise(ds4):
    rows, cols = 8, 512
    b = synth.random_iq2_blob(3, 0, 0, rows, cols)
    assert np.array_equal(ds4.ds4moe_dequantize_iq2(b, rows, cols).view(np.uint32),
                          oracle.dequant_iq2(b, rows, cols).view(np.uint32))
    b = synth.random_q2k_blob(3, 0, 2, rows, cols)
    assert np.array_equal(ds4.ds4moe_dequantize_q2k(b, rows, cols).view(np.uint32),
                          oracle.dequant_q2k(b, rows, cols).view(np.uint32))
    b = synth.random_q4k_blob(3, 0, 1, rows, cols)
    assert np.array_equal(ds4.ds4moe_dequantize_q4k(b, rows, cols).view(np.uint32),
                          oracle.dequant_q4k(b, rows, cols).view(np.uint32))


def test_quantizer_rejects_non_finite(ds4):
    w = np.zeros((2, 256), np.float32)
    w[1, 3] = np.inf
    with pytest.raises(ds4.Ds4moeError) as ei:
        ds4.ds4moe_quantize_iq2(w)
    assert ei.value.status == ds4.DS4MOE_EBADDATA
    with pytest.raises(ValueError):
        ds4.ds4moe_quantize_q2k(np.zeros((2, 100), np.float32))


def test_device_entry_points_reject_bad_arguments_on_host(ds4):
    L = ds4.lib()
    # k > E, E too large, bad gate mode: rejected before any CUDA call
    assert L.ds4moe_route(None, 4, 8, 9, 0, None, None, None) == ds4.DS4MOE_EINVAL
    assert L.ds4moe_route(None, 4, 2000, 2, 0, None, None, None) == ds4.DS4MOE_EINVAL
    assert L.ds4moe_route(None, 4, 8, 2, 7, None, None, None) == ds4.DS4MOE_EINVAL
    assert L.ds4moe_route(None, 4, 8, 2, 0, None, None, None) == ds4.DS4MOE_EINVAL  # null pointers
    assert L.ds4moe_route(None, 0, 8, 2, 0, None, None, None) == ds4.DS4MOE_OK      # T = 0: no-op
    # router logits: D a multiple of 256 (<= 8192), E a multiple of 8 in [8, 1024], pointers checked before any launch
    assert L.ds4moe_router_logits(None, None, None, 1, 300, 8, None, None) == ds4.DS4MOE_EINVAL
    assert L.ds4moe_router_logits(None, None, None, 1, 256, 12, None, None) == ds4.DS4MOE_EINVAL
    assert L.ds4moe_router_logits(None, None, None, 1, 256, 2048, None, None) == ds4.DS4MOE_EINVAL
    assert L.ds4moe_router_logits(None, None, None, 1, 8448, 8, None, None) == ds4.DS4MOE_EINVAL  # D > 8192
    assert L.ds4moe_router_logits(None, None, None, -1, 256, 8, None, None) == ds4.DS4MOE_EINVAL
    assert L.ds4moe_router_logits(None, None, None, 1, 256, 8, None, None) == ds4.DS4MOE_EINVAL  # null pointers
    assert L.ds4moe_router_logits(None, None, None, 0, 256, 8, None, None) == ds4.DS4MOE_OK      # T = 0: no-op
    assert L.ds4moe_group(None, 4, 2, 8, None, None, None, None, None) == ds4.DS4MOE_EINVAL
    assert L.ds4moe_expert_ffn(None, None, None, 1, 1, 0, None, None) == ds4.DS4MOE_EINVAL
    assert L.ds4moe_set_option(None, 0, 1) == ds4.DS4MOE_EINVAL
    assert L.ds4moe_weights_dequantize(None, 0, 0, None, None, None) == ds4.DS4MOE_EINVAL
    assert L.ds4moe_weights_create(None, None) == ds4.DS4MOE_EINVAL
    # pooled handles: at least one slot, a descriptor; pool state only of a pooled handle
    assert L.ds4moe_weights_create_pooled(None, 4, None) == ds4.DS4MOE_EINVAL
    assert L.ds4moe_weights_create_pooled(None, 0, None) == ds4.DS4MOE_EINVAL
    assert L.ds4moe_pool_info(None, None, None, None, None) == ds4.DS4MOE_EINVAL


def _blobs(wl, fmt="q2"):
    if fmt == "q4":
        return [list(b) for b in synth.random_q4_expert_blobs(wl)]
    return [list(b) for b in synth.random_expert_blobs(wl)]


@pytest.mark.parametrize("fmt,mat,byte", [("q2", 0, 0), ("q2", 1, 0), ("q2", 2, 80), ("q2", 2, 82),
                                          ("q4", 0, 0), ("q4", 2, 2)])
@pytest.mark.parametrize("bad", [0x7E00, 0x7C00, 0xFC00])   # NaN, +inf, -inf as fp16
def test_weights_create_rejects_a_non_finite_block_scale_before_any_device_call(ds4, fmt, mat, byte, bad):
    """A corrupted blob (one block's fp16 d or dmin not finite) is refused with EBADDATA. The check
    comes before the handle touches the device, so it runs here, without a GPU."""
    wl = synth.Workload("bad", T=1, D=256, F=512, E=3, k=2, seed=5, shared=False)
    gate, up, down = _blobs(wl, fmt)
    mats = [gate, up, down]
    blk = 144 if fmt == "q4" else (84 if mat == 2 else 66)
    b = mats[mat][1].copy()
    at = 5 * blk + byte                       # block 5 of expert 1
    b[at], b[at + 1] = bad & 0xFF, bad >> 8
    mats[mat][1] = b
    with pytest.raises(ds4.Ds4moeError) as ei:
        ds4.ds4moe_weights_create(gate, up, down, wl.D, wl.F, max_tokens=1, max_k=2, fmt=fmt)
    assert ei.value.status == ds4.DS4MOE_EBADDATA


def test_misaligned_device_pointers_are_refused_on_host(ds4):
    L = ds4.lib()
    # router logits: x and the router must be 16-byte aligned, logits and bias 4-byte aligned;
    # the pointers are never dereferenced when the check fails
    assert L.ds4moe_router_logits(0x1002, 0x2000, None, 1, 256, 8, 0x3000, None) == ds4.DS4MOE_EINVAL
    assert L.ds4moe_router_logits(0x1000, 0x2008, None, 1, 256, 8, 0x3000, None) == ds4.DS4MOE_EINVAL
    assert L.ds4moe_router_logits(0x1000, 0x2000, 0x4002, 1, 256, 8, 0x3000, None) == ds4.DS4MOE_EINVAL
    assert L.ds4moe_router_logits(0x1000, 0x2000, None, 1, 256, 8, 0x3001, None) == ds4.DS4MOE_EINVAL


def test_allocation_failure_hook_arguments(ds4):
    L = ds4.lib()
    assert L.ds4moe_test_fail_allocation(-1) == ds4.DS4MOE_EINVAL
    assert L.ds4moe_test_fail_allocation(0) == ds4.DS4MOE_OK
