"""Oracle router logits -- TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

The step in front of routing: logits[t][e] = sum_d x[t][d] * W[e][d] + bias[e] over the token's
bf16 activations and the unquantised router ("DwarfStar" README, "模型权重": projections and
router stay unquantised; "DwarfStar 深度解析" §3.4.3: the router is kept at full precision),
read here as bf16 weights and an fp32 bias. The oracle is that definition in fp64: every bf16
value is exact in fp64 and so is every product (8 + 8 significant bits), and the sum of D such
products differs from the exact sum by far less than the fp32 rounding any device order incurs.

A device computes the same sum in fp32 in some order of its own. Whatever the order, a term
that passes through at most n fp32 additions leaves the sum within
    n * 2^-24 * (sum_d |x[t][d] W[e][d]| + |bias[e]|)
of the exact value (the standard bound of recursive summation, to first order); fp32_bound
returns it for the depth n = 8 D / 256 + 6 by default, which covers every order that adds within
lanes, then across at most 32 lanes by halving, then across segments, then the bias (the library
documents its order for small calls as one of these). tensor_core_depth(D) is the depth for an
order that sums each block of 16 consecutive columns (in any order: at most 15 additions for a
term), adds the blocks into one accumulator in increasing order (D / 16 additions) and then the
bias, counting every addition twice so that it may truncate instead of rounding to nearest (an
error of at most 2^-23 of its result instead of 2^-24); the library documents its order for large
calls as one of these.
"""
import numpy as np


def bf16_to_f64(bits):
    """bf16 bit patterns (uint16) to their exact fp64 values."""
    bits = np.asarray(bits, np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def router_logits(x_bf16, w_bf16, bias=None):
    """x_bf16 uint16 [T][D], w_bf16 uint16 [E][D] (bf16 bits), bias fp32 [E] or None.
    Returns the logits in fp64 [T][E]."""
    x = bf16_to_f64(x_bf16)
    w = bf16_to_f64(w_bf16)
    assert x.ndim == 2 and w.ndim == 2 and w.shape[1] == x.shape[1]
    out = x @ w.T
    if bias is not None:
        out = out + np.asarray(bias, np.float32).astype(np.float64)[None, :]
    return out


def tensor_core_depth(D):
    """The summation depth of a 16-column-block accumulation with possibly truncating additions
    (see the module docstring)."""
    return 2 * (D // 16 + 16)


def fp32_bound(x_bf16, w_bf16, bias=None, depth=None):
    """Bound [T][E] on |fp32 logit - exact logit| for any fp32 summation of depth at most
    `depth` (default 8 D / 256 + 6; see the module docstring)."""
    x = np.abs(bf16_to_f64(x_bf16))
    w = np.abs(bf16_to_f64(w_bf16))
    D = x.shape[1]
    mag = x @ w.T
    if bias is not None:
        mag = mag + np.abs(np.asarray(bias, np.float32).astype(np.float64))[None, :]
    n = 8 * D // 256 + 6 if depth is None else depth
    return n * 2.0 ** -24 * mag
