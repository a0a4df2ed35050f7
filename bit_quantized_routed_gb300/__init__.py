"""Python binding of the ds4moe C ABI (include/ds4moe.h): argument marshalling only.

Every step of the hot path runs in the library's CUDA kernels; PyTorch supplies device
memory and the current stream. The functions keep the C names. If the shared library is
missing the import of any function raises -- there is no fallback path.
"""
import ctypes
import os

import numpy as np

from ._build import LIB_PATH, build  # noqa: F401

DS4MOE_OK = 0
DS4MOE_EINVAL = 1
DS4MOE_ENOMEM = 2
DS4MOE_ECUDA = 3
DS4MOE_EBADDATA = 4
DS4MOE_ETIMEOUT = 5
DS4MOE_EUNSUPPORTED = 6
DS4MOE_ERANGE = 7
DS4MOE_ECAPACITY = 8

DS4MOE_GATE_SOFTMAX = 0
DS4MOE_GATE_SIGMOID = 1
DS4MOE_GATE, DS4MOE_UP, DS4MOE_DOWN = 0, 1, 2
DS4MOE_OPT_GEMM_MIN_TOKENS = 0
DS4MOE_OPT_SHARED_GEMM_MIN_TOKENS = 1
DS4MOE_OPT_PROFILE = 2
DS4MOE_OPT_SINGLE_STEP = 3
DS4MOE_OPT_TRACE = 4
DS4MOE_OPT_SMALL_GROUPS = 5
DS4MOE_OPT_WAIT_TEST = 6
DS4MOE_OPT_GEMM_PAIRS = 7
STAGES = ["route", "group", "gather", "up_gemv", "up_gemm", "down_gemv", "down_gemm", "combine", "step", "pool",
          "repair"]

EXPORTED = [
    "ds4moe_strerror", "ds4moe_q2k_bytes", "ds4moe_iq2_bytes", "ds4moe_q4k_bytes", "ds4moe_iq2_grid",
    "ds4moe_quantize_q2k", "ds4moe_quantize_iq2", "ds4moe_quantize_q4k", "ds4moe_dequantize_q2k",
    "ds4moe_dequantize_iq2", "ds4moe_dequantize_q4k",
    "ds4moe_weights_create", "ds4moe_weights_create_q4", "ds4moe_weights_create_pooled", "ds4moe_pool_info", "ds4moe_weights_destroy", "ds4moe_set_option", "ds4moe_weights_dequantize",
    "ds4moe_router_logits", "ds4moe_router_last_status", "ds4moe_route", "ds4moe_group", "ds4moe_expert_ffn", "ds4moe_get_stats", "ds4moe_last_status",
    "ds4moe_expert_ffn_static", "ds4moe_step_trace", "ds4moe_test_fail_allocation",
]


class Ds4moeError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__("%s: %s (status %d)" % (where, ds4moe_strerror(status), status))


class _Desc(ctypes.Structure):
    _fields_ = [
        ("d_model", ctypes.c_int), ("d_ff", ctypes.c_int), ("n_experts", ctypes.c_int),
        ("gate_iq2", ctypes.POINTER(ctypes.c_void_p)), ("up_iq2", ctypes.POINTER(ctypes.c_void_p)),
        ("down_q2k", ctypes.POINTER(ctypes.c_void_p)),
        ("shared_gate_bf16", ctypes.c_void_p), ("shared_up_bf16", ctypes.c_void_p),
        ("shared_down_bf16", ctypes.c_void_p),
        ("max_tokens", ctypes.c_int), ("max_k", ctypes.c_int),
    ]


class _Stats(ctypes.Structure):
    _fields_ = [("calls", ctypes.c_uint64), ("launches", ctypes.c_uint64), ("stage_ms", ctypes.c_float * len(STAGES))]


_lib = None


def lib():
    """The loaded libds4moe.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libds4moe.so is not built (%s); run bit_quantized_routed_gb300.build()" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        vp, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
        sig = {
            "ds4moe_strerror": ([i32], ctypes.c_char_p),
            "ds4moe_q2k_bytes": ([i64, i64], sz),
            "ds4moe_iq2_bytes": ([i64, i64], sz),
            "ds4moe_q4k_bytes": ([i64, i64], sz),
            "ds4moe_quantize_q4k": ([vp, i64, i64, vp, sz], i32),
            "ds4moe_dequantize_q4k": ([vp, i64, i64, vp], i32),
            "ds4moe_weights_create_q4": ([ctypes.POINTER(_Desc), ctypes.POINTER(vp)], i32),
            "ds4moe_iq2_grid": ([vp], i32),
            "ds4moe_quantize_q2k": ([vp, i64, i64, vp, sz], i32),
            "ds4moe_quantize_iq2": ([vp, i64, i64, vp, sz], i32),
            "ds4moe_dequantize_q2k": ([vp, i64, i64, vp], i32),
            "ds4moe_dequantize_iq2": ([vp, i64, i64, vp], i32),
            "ds4moe_weights_create": ([ctypes.POINTER(_Desc), ctypes.POINTER(vp)], i32),
            "ds4moe_weights_create_pooled": ([ctypes.POINTER(_Desc), i32, ctypes.POINTER(vp)], i32),
            "ds4moe_pool_info": ([vp, ctypes.POINTER(i32), ctypes.POINTER(ctypes.c_uint64),
                                  ctypes.POINTER(ctypes.c_uint64), vp], i32),
            "ds4moe_weights_destroy": ([vp], None),
            "ds4moe_set_option": ([vp, i32, i32], i32),
            "ds4moe_weights_dequantize": ([vp, i32, i32, vp, vp, vp], i32),
            "ds4moe_router_logits": ([vp, vp, vp, i32, i32, i32, vp, vp], i32),
            "ds4moe_router_last_status": ([vp], i32),
            "ds4moe_route": ([vp, i32, i32, i32, i32, vp, vp, vp], i32),
            "ds4moe_group": ([vp, i32, i32, i32, vp, vp, vp, vp, vp], i32),
            "ds4moe_expert_ffn": ([vp, vp, vp, i32, i32, i32, vp, vp], i32),
            "ds4moe_get_stats": ([vp, ctypes.POINTER(_Stats)], i32),
            "ds4moe_last_status": ([vp, vp], i32),
            "ds4moe_expert_ffn_static": ([vp, vp, vp, i32, i32, i32, vp, vp], i32),
            "ds4moe_step_trace": ([vp, vp, i32, ctypes.POINTER(i32)], i32),
            "ds4moe_test_fail_allocation": ([i32], i32),
        }
        for name, (args, res) in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def _check(rc, where):
    if rc != DS4MOE_OK:
        raise Ds4moeError(rc, where)


def ds4moe_test_fail_allocation(n):
    """Test hook: the n-th device allocation of any later handle creation fails (0: off)."""
    _check(lib().ds4moe_test_fail_allocation(int(n)), "ds4moe_test_fail_allocation")


def ds4moe_strerror(status):
    return lib().ds4moe_strerror(int(status)).decode()


def ds4moe_q2k_bytes(rows, cols):
    return lib().ds4moe_q2k_bytes(rows, cols)


def ds4moe_iq2_bytes(rows, cols):
    return lib().ds4moe_iq2_bytes(rows, cols)


def ds4moe_q4k_bytes(rows, cols):
    return lib().ds4moe_q4k_bytes(rows, cols)


def ds4moe_iq2_grid():
    g = np.zeros(2048, np.uint8)
    _check(lib().ds4moe_iq2_grid(g.ctypes.data), "ds4moe_iq2_grid")
    return g.reshape(256, 8)


def _quantize(fn, nbytes, w):
    w = np.ascontiguousarray(w, np.float32)
    rows, cols = w.shape
    n = nbytes(rows, cols)
    if n == 0:
        raise ValueError("cols must be a positive multiple of 256")
    out = np.empty(n, np.uint8)
    _check(fn(w.ctypes.data, rows, cols, out.ctypes.data, n), fn.__name__)
    return out


def ds4moe_quantize_q2k(w):
    """Host quantisation of fp32 [rows, cols] to Q2_K-style blocks (uint8 array)."""
    return _quantize(lib().ds4moe_quantize_q2k, ds4moe_q2k_bytes, w)


def ds4moe_quantize_iq2(w):
    """Host quantisation of fp32 [rows, cols] to IQ2-style blocks (uint8 array)."""
    return _quantize(lib().ds4moe_quantize_iq2, ds4moe_iq2_bytes, w)


def _dequantize(fn, nbytes, blob, rows, cols):
    blob = np.ascontiguousarray(blob, np.uint8)
    if blob.size != nbytes(rows, cols):
        raise ValueError("blob size does not match the shape")
    out = np.empty((rows, cols), np.float32)
    _check(fn(blob.ctypes.data, rows, cols, out.ctypes.data), fn.__name__)
    return out


def ds4moe_dequantize_q2k(blob, rows, cols):
    return _dequantize(lib().ds4moe_dequantize_q2k, ds4moe_q2k_bytes, blob, rows, cols)


def ds4moe_quantize_q4k(w):
    """Host quantisation of fp32 [rows, cols] to the 4-bit variant's Q4_K-style blocks."""
    return _quantize(lib().ds4moe_quantize_q4k, ds4moe_q4k_bytes, w)


def ds4moe_dequantize_q4k(blob, rows, cols):
    return _dequantize(lib().ds4moe_dequantize_q4k, ds4moe_q4k_bytes, blob, rows, cols)


def ds4moe_dequantize_iq2(blob, rows, cols):
    return _dequantize(lib().ds4moe_dequantize_iq2, ds4moe_iq2_bytes, blob, rows, cols)


# ------------------------------------------------------------------ device side

def _stream(stream=None):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t, dtype=None, what="tensor"):
    import torch
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda or not t.is_contiguous():
        raise ValueError("%s must be a contiguous CUDA tensor" % what)
    if dtype is not None and t.dtype != dtype:
        raise ValueError("%s must have dtype %s" % (what, dtype))
    return ctypes.c_void_p(t.data_ptr())


class Weights:
    """A resident weights handle (ds4moe_weights_create / ds4moe_weights_destroy)."""

    def __init__(self, handle, d_model, d_ff, n_experts, max_tokens, max_k, has_shared):
        self.handle = handle
        self.d_model, self.d_ff, self.n_experts = d_model, d_ff, n_experts
        self.max_tokens, self.max_k, self.has_shared = max_tokens, max_k, has_shared

    def close(self):
        if self.handle:
            lib().ds4moe_weights_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def ds4moe_weights_create(gate_iq2, up_iq2, down_q2k, d_model, d_ff, shared=None, max_tokens=1, max_k=8,
                          n_slots=None, fmt="q2"):
    """Upload per-expert packed blobs (lists of uint8 arrays) and an optional bf16 shared
    expert (gate, up, down as uint16 arrays of bf16 bits) to the current CUDA device. With
    n_slots, a pooled handle (ds4moe_weights_create_pooled): the experts stay in pinned host
    memory and stream into n_slots device slots as calls touch them. fmt="q4": the 4-bit variant,
    all three per-expert blobs Q4_K-style (ds4moe_weights_create_q4)."""
    E = len(gate_iq2)
    keep = []

    def ptrs(blobs, nbytes):
        arr = (ctypes.c_void_p * E)()
        for e, b in enumerate(blobs):
            b = np.ascontiguousarray(b, np.uint8)
            if b.size != nbytes:
                raise ValueError("expert %d blob has %d bytes, expected %d" % (e, b.size, nbytes))
            keep.append(b)
            arr[e] = b.ctypes.data
        return arr

    if fmt == "q4":
        gi = ptrs(gate_iq2, ds4moe_q4k_bytes(d_ff, d_model))
        ui = ptrs(up_iq2, ds4moe_q4k_bytes(d_ff, d_model))
        dq = ptrs(down_q2k, ds4moe_q4k_bytes(d_model, d_ff))
    else:
        gi = ptrs(gate_iq2, ds4moe_iq2_bytes(d_ff, d_model))
        ui = ptrs(up_iq2, ds4moe_iq2_bytes(d_ff, d_model))
        dq = ptrs(down_q2k, ds4moe_q2k_bytes(d_model, d_ff))
    desc = _Desc(d_model, d_ff, E, gi, ui, dq, None, None, None, max_tokens, max_k)
    if shared is not None:
        sh = [np.ascontiguousarray(s, np.uint16).reshape(-1) for s in shared]
        if any(s.size != d_model * d_ff for s in sh):
            raise ValueError("shared expert matrices must have d_model * d_ff elements")
        keep.extend(sh)
        desc.shared_gate_bf16, desc.shared_up_bf16, desc.shared_down_bf16 = (s.ctypes.data for s in sh)
    h = ctypes.c_void_p()
    if fmt == "q4":
        if n_slots is not None:
            raise ValueError("the 4-bit variant has no pooled handle")
        _check(lib().ds4moe_weights_create_q4(ctypes.byref(desc), ctypes.byref(h)), "ds4moe_weights_create_q4")
    elif n_slots is None:
        _check(lib().ds4moe_weights_create(ctypes.byref(desc), ctypes.byref(h)), "ds4moe_weights_create")
    else:
        _check(lib().ds4moe_weights_create_pooled(ctypes.byref(desc), int(n_slots), ctypes.byref(h)),
               "ds4moe_weights_create_pooled")
    return Weights(h, d_model, d_ff, E, max_tokens, max_k, shared is not None)


def ds4moe_pool_info(weights):
    """(n_slots, hits, misses, slot_expert int32 [n_slots]) of a pooled handle."""
    n = ctypes.c_int(0)
    _check(lib().ds4moe_pool_info(weights.handle, ctypes.byref(n), None, None, None), "ds4moe_pool_info")
    hits, misses = ctypes.c_uint64(0), ctypes.c_uint64(0)
    slots = np.zeros(n.value, np.int32)
    _check(lib().ds4moe_pool_info(weights.handle, None, ctypes.byref(hits), ctypes.byref(misses), slots.ctypes.data),
           "ds4moe_pool_info")
    return n.value, hits.value, misses.value, slots


def ds4moe_weights_destroy(weights):
    weights.close()


def ds4moe_set_option(weights, option, value):
    _check(lib().ds4moe_set_option(weights.handle, option, value), "ds4moe_set_option")


def ds4moe_weights_dequantize(weights, expert, matrix, dst_f32=None, dst_f16=None, stream=None):
    import torch
    _check(lib().ds4moe_weights_dequantize(weights.handle, expert, matrix,
                                           _ptr(dst_f32, torch.float32, "dst_f32"),
                                           _ptr(dst_f16, torch.float16, "dst_f16"), _stream(stream)),
           "ds4moe_weights_dequantize")


def ds4moe_router_logits(x, w_router, bias=None, logits=None, stream=None):
    """Router logits on the device in the library's fixed fp32 order. x: bf16 CUDA [T, D];
    w_router: bf16 CUDA [E, D]; bias: fp32 CUDA [E] or None. Returns fp32 [T, E]."""
    import torch
    T, D = x.shape
    E = w_router.shape[0]
    if w_router.shape[1] != D:
        raise ValueError("w_router must be [E, D]")
    if logits is None:
        logits = torch.empty((T, E), dtype=torch.float32, device=x.device)
    _check(lib().ds4moe_router_logits(_ptr(x, torch.bfloat16, "x"), _ptr(w_router, torch.bfloat16, "w_router"),
                                      _ptr(bias, torch.float32, "bias") if bias is not None else None, T, D, E,
                                      _ptr(logits, torch.float32, "logits"), _stream(stream)),
           "ds4moe_router_logits")
    return logits


def ds4moe_route(logits, k, gate_mode=DS4MOE_GATE_SOFTMAX, topk_idx=None, topk_w=None, stream=None):
    """Top-k routing on the device. logits: fp32 CUDA [T, E]. Returns (idx int32 [T,k], w fp32 [T,k])."""
    import torch
    T, E = logits.shape
    if topk_idx is None:
        topk_idx = torch.empty((T, k), dtype=torch.int32, device=logits.device)
    if topk_w is None:
        topk_w = torch.empty((T, k), dtype=torch.float32, device=logits.device)
    _check(lib().ds4moe_route(_ptr(logits, torch.float32, "logits"), T, E, k, gate_mode,
                              _ptr(topk_idx, torch.int32, "topk_idx"), _ptr(topk_w, torch.float32, "topk_w"),
                              _stream(stream)), "ds4moe_route")
    return topk_idx, topk_w


def ds4moe_group(topk_idx, n_experts, stream=None):
    """Stable grouping of pairs by expert. Returns (counts, offsets, perm, inv) int32 CUDA tensors."""
    import torch
    T, k = topk_idx.shape
    dev = topk_idx.device
    counts = torch.empty(n_experts, dtype=torch.int32, device=dev)
    offsets = torch.empty(n_experts + 1, dtype=torch.int32, device=dev)
    perm = torch.empty(max(1, T * k), dtype=torch.int32, device=dev)
    inv = torch.empty(max(1, T * k), dtype=torch.int32, device=dev)
    _check(lib().ds4moe_group(_ptr(topk_idx, torch.int32, "topk_idx"), T, k, n_experts, _ptr(counts),
                              _ptr(offsets), _ptr(perm), _ptr(inv), _stream(stream)), "ds4moe_group")
    return counts, offsets, perm[:T * k], inv[:T * k]


def ds4moe_expert_ffn(x, weights, logits, k, out, gate_mode=DS4MOE_GATE_SOFTMAX, stream=None):
    """out += expert FFN of x, in place. x: bf16 CUDA [T, D]; logits: fp32 CUDA [T, E];
    out: fp32 CUDA [T, D]."""
    import torch
    T = x.shape[0]
    if x.shape != (T, weights.d_model) or out.shape != (T, weights.d_model) or logits.shape != (T, weights.n_experts):
        raise ValueError("shape mismatch")
    _check(lib().ds4moe_expert_ffn(_ptr(x, torch.bfloat16, "x"), weights.handle,
                                   _ptr(logits, torch.float32, "logits"), T, k, gate_mode,
                                   _ptr(out, torch.float32, "out"), _stream(stream)), "ds4moe_expert_ffn")


def ds4moe_get_stats(weights):
    """Returns {"calls", "launches", "stage_ms": {stage name: ms of the last profiled call}}."""
    st = _Stats()
    _check(lib().ds4moe_get_stats(weights.handle, ctypes.byref(st)), "ds4moe_get_stats")
    return {"calls": st.calls, "launches": st.launches,
            "stage_ms": {n: float(st.stage_ms[i]) for i, n in enumerate(STAGES)}}


def ds4moe_step_trace(weights, max_ctas=1024):
    """Per-CTA timestamps (ns) of the last single-token call: array [CTAs, 6]."""
    out = np.zeros(max_ctas * 6, np.uint64)
    n = ctypes.c_int(0)
    _check(lib().ds4moe_step_trace(weights.handle, out.ctypes.data, out.size, ctypes.byref(n)), "ds4moe_step_trace")
    return out[:n.value].reshape(-1, 6)


def ds4moe_router_last_status(stream=None):
    """DS4MOE_ETIMEOUT if a tensor-core router call since the last query gave up a bounded wait."""
    return lib().ds4moe_router_last_status(_stream(stream))


def ds4moe_last_status(weights, stream=None):
    return lib().ds4moe_last_status(weights.handle, _stream(stream))


def ds4moe_expert_ffn_static(x, weights, logits, k, out, gate_mode=DS4MOE_GATE_SOFTMAX, stream=None):
    """out += expert FFN of x, like ds4moe_expert_ffn, but with the per-call intermediates in
    the library's static device region: the call allocates no device memory. For callers
    that may not allocate while they serve (see include/ds4moe.h)."""
    import torch
    T = x.shape[0]
    if x.shape != (T, weights.d_model) or out.shape != (T, weights.d_model) or logits.shape != (T, weights.n_experts):
        raise ValueError("shape mismatch")
    _check(lib().ds4moe_expert_ffn_static(_ptr(x, torch.bfloat16, "x"), weights.handle,
                                          _ptr(logits, torch.float32, "logits"), T, k, gate_mode,
                                          _ptr(out, torch.float32, "out"), _stream(stream)),
           "ds4moe_expert_ffn_static")
