"""The oracle -- TEST INFRASTRUCTURE ONLY.

A plain, slow CPU restatement (fp64) of what the routed-MoE expert FFN over 2-bit experts
computes: block formats (quantise / dequantise), top-k routing, grouping of (token, slot)
pairs by expert, and the SwiGLU expert FFN with its gate-weighted combine. Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import this
package. It shares no code with the product library and never imports it.

Sources (page titles and sections):
  * "DwarfStar" (the ds4 README), "模型权重": only routed experts are quantised, up/gate to
    IQ2_XXS and down to Q2_K; shared expert, projections and router stay unquantised.
  * "DwarfStar 深度解析", §2.1 (routed MoE: the experts a token uses are chosen per token)
    and §3.4.3 (the quantisation split; the router stays at full precision).
  * The byte layouts, the grid and the quantisers are the library's fixed readings, including
    the Q4_K-style block of the 4-bit variant ("DwarfStar" README, "模型权重": the q4 build).

Parity pins: every function here is checked in ``tests/test_oracle_*.py`` against something
other than itself (numpy's float16 rounding, a published splitmix64 output, hand-built
blocks with known values, brute-force searches, dense fp64 matrix products, invariants).
"""
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")

_lib = None


def build(force=False):
    """Compile oracle.c with gcc (-O2, no fused multiply-add) into oracle/_build."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + ".%d.tmp" % os.getpid()
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                           "-shared", "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        u8p = ctypes.POINTER(ctypes.c_uint8)
        f32p = ctypes.POINTER(ctypes.c_float)
        f64p = ctypes.POINTER(ctypes.c_double)
        i32p = ctypes.POINTER(ctypes.c_int32)
        i64 = ctypes.c_int64
        L.or_half_to_double.argtypes = [ctypes.c_uint16]
        L.or_half_to_double.restype = ctypes.c_double
        L.or_double_to_half.argtypes = [ctypes.c_double]
        L.or_double_to_half.restype = ctypes.c_uint16
        L.or_splitmix64_next.argtypes = [ctypes.POINTER(ctypes.c_uint64)]
        L.or_splitmix64_next.restype = ctypes.c_uint64
        L.or_iq2_grid.argtypes = [u8p]
        L.or_q2k_quantize.argtypes = [f32p, i64, i64, u8p]
        L.or_q2k_quantize.restype = ctypes.c_int
        L.or_iq2_quantize.argtypes = [f32p, i64, i64, u8p, u8p]
        L.or_iq2_quantize.restype = ctypes.c_int
        L.or_q2k_dequant.argtypes = [u8p, i64, i64, f32p]
        L.or_q4k_quantize.argtypes = [f32p, i64, i64, u8p]
        L.or_q4k_quantize.restype = ctypes.c_int
        L.or_q4k_dequant.argtypes = [u8p, i64, i64, f32p]
        L.or_iq2_dequant.argtypes = [u8p, i64, i64, u8p, f32p]
        L.or_route.argtypes = [f32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, i32p, f64p]
        L.or_permute.argtypes = [i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, i32p, i32p, i32p, i32p]
        _lib = L
    return _lib


def _p(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


Q2K_BLOCK_BYTES = 84
Q4K_BLOCK_BYTES = 144
IQ2_BLOCK_BYTES = 66


def half_to_double(h):
    return lib().or_half_to_double(int(h))


def double_to_half(x):
    return lib().or_double_to_half(float(x))


def splitmix64(seed, n):
    st = ctypes.c_uint64(seed)
    return [lib().or_splitmix64_next(ctypes.byref(st)) for _ in range(n)]


_grid = None


def iq2_grid():
    """The 256 x 8 grid of magnitudes (uint8), built by splitmix64 from the grid's fixed seed."""
    global _grid
    if _grid is None:
        g = np.zeros(2048, np.uint8)
        lib().or_iq2_grid(_p(g, ctypes.c_uint8))
        _grid = g.reshape(256, 8)
    return _grid


def quantize_q2k(w):
    w = np.ascontiguousarray(w, np.float32)
    rows, cols = w.shape
    assert cols % 256 == 0
    out = np.zeros(rows * cols // 256 * Q2K_BLOCK_BYTES, np.uint8)
    if lib().or_q2k_quantize(_p(w, ctypes.c_float), rows, cols, _p(out, ctypes.c_uint8)) != 0:
        raise ValueError("q2k quantisation rejected the input (non-finite or fp16 overflow)")
    return out


def quantize_q4k(w):
    """The Q4_K-style quantiser (the 4-bit variant) of fp32 [rows, cols]."""
    w = np.ascontiguousarray(w, np.float32)
    rows, cols = w.shape
    assert cols % 256 == 0
    out = np.zeros(rows * cols // 256 * Q4K_BLOCK_BYTES, np.uint8)
    if lib().or_q4k_quantize(_p(w, ctypes.c_float), rows, cols, _p(out, ctypes.c_uint8)) != 0:
        raise ValueError("q4k quantisation rejected the input (non-finite or fp16 overflow)")
    return out


def dequant_q4k(blob, rows, cols):
    blob = np.ascontiguousarray(blob, np.uint8)
    assert blob.size == rows * cols // 256 * Q4K_BLOCK_BYTES
    out = np.empty((rows, cols), np.float32)
    lib().or_q4k_dequant(_p(blob, ctypes.c_uint8), rows, cols, _p(out, ctypes.c_float))
    return out


def quantize_iq2(w):
    w = np.ascontiguousarray(w, np.float32)
    rows, cols = w.shape
    assert cols % 256 == 0
    g = np.ascontiguousarray(iq2_grid().reshape(-1))
    out = np.zeros(rows * cols // 256 * IQ2_BLOCK_BYTES, np.uint8)
    if lib().or_iq2_quantize(_p(w, ctypes.c_float), rows, cols, _p(g, ctypes.c_uint8),
                             _p(out, ctypes.c_uint8)) != 0:
        raise ValueError("iq2 quantisation rejected the input (non-finite or fp16 overflow)")
    return out


def dequant_q2k(blob, rows, cols):
    blob = np.ascontiguousarray(blob, np.uint8)
    assert blob.size == rows * cols // 256 * Q2K_BLOCK_BYTES
    out = np.empty((rows, cols), np.float32)
    lib().or_q2k_dequant(_p(blob, ctypes.c_uint8), rows, cols, _p(out, ctypes.c_float))
    return out


def dequant_iq2(blob, rows, cols):
    blob = np.ascontiguousarray(blob, np.uint8)
    assert blob.size == rows * cols // 256 * IQ2_BLOCK_BYTES
    g = np.ascontiguousarray(iq2_grid().reshape(-1))
    out = np.empty((rows, cols), np.float32)
    lib().or_iq2_dequant(_p(blob, ctypes.c_uint8), rows, cols, _p(g, ctypes.c_uint8),
                         _p(out, ctypes.c_float))
    return out


GATE_SOFTMAX = 0
GATE_SIGMOID = 1


def route(logits, k, mode=GATE_SOFTMAX):
    """Top-k experts per token (logit descending, ties to the lower index, a NaN logit ranked as
    -inf) and gate weights (fp64): softmax over the selected logits, or normalised sigmoids, with
    equal selected logits (equal infinities included) weighted equally. Returns idx int32 [T,k],
    g float64 [T,k]."""
    logits = np.ascontiguousarray(logits, np.float32)
    T, E = logits.shape
    idx = np.zeros((T, k), np.int32)
    g = np.zeros((T, k), np.float64)
    lib().or_route(_p(logits, ctypes.c_float), T, E, k, mode, _p(idx, ctypes.c_int32),
                   _p(g, ctypes.c_double))
    return idx, g


def permute(idx, E):
    """Stable counting sort of pairs (t, s) by expert. Returns counts[E], offsets[E+1],
    perm[P] (pair id t*k+s at each grouped position) and inv[P] (the inverse)."""
    idx = np.ascontiguousarray(idx, np.int32)
    T, k = idx.shape
    P = T * k
    counts = np.zeros(E, np.int32)
    offsets = np.zeros(E + 1, np.int32)
    perm = np.zeros(P, np.int32)
    inv = np.zeros(P, np.int32)
    lib().or_permute(_p(idx, ctypes.c_int32), T, k, E, _p(counts, ctypes.c_int32),
                     _p(offsets, ctypes.c_int32), _p(perm, ctypes.c_int32), _p(inv, ctypes.c_int32))
    return counts, offsets, perm, inv


from .moe import bf16_to_f64, expert_ffn_dense, moe_ffn  # noqa: E402,F401
