"""Oracle router logits -- TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

The step in front of routing: logits[t][e] = sum_d x[t][d] * W[e][d] + bias[e] over the token's
bf16 activations and the unquantised router ("DwarfStar" README, "模型权重": projections and
router stay unquantised; "DwarfStar 深度解析" §3.4.3: the router is kept at full precision),
read here as bf16 weights and an fp32 bias. The top-k that follows selects experts by these
values, so the oracle takes them in the same precision and the same order as the library's
router kernel (a reading: the pages give no order), which makes the selection comparable bit
for bit:

  * every product of two bf16 values is exact in fp32 (8 + 8 significant bits), for products in
    fp32's normal range;
  * the columns are cut into segments of 1024 (the last one shorter when D is not a multiple);
  * within a segment, 32 partial sums p_l (l = 0..31), each starting at 0 and adding in fp32, in
    increasing d, the products of the segment's columns d with (d // 8) % 32 == l; then, for
    o = 16, 8, 4, 2, 1: p_l <- p_l + p_(l xor o) in fp32 (every l ends with the same value, the
    segment sum);
  * the segment sums added in fp32 in increasing segment order, then bias[e] in fp32.
"""
import numpy as np


def bf16_to_f32(bits):
    """bf16 bit patterns (uint16) to their exact fp32 values."""
    bits = np.asarray(bits, np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32)


def router_logits(x_bf16, w_bf16, bias=None):
    """x_bf16 uint16 [T][D], w_bf16 uint16 [E][D] (bf16 bits), bias fp32 [E] or None.
    Returns fp32 [T][E] in the order above. D must be a multiple of 256."""
    x = bf16_to_f32(x_bf16)
    w = bf16_to_f32(w_bf16)
    T, D = x.shape
    E = w.shape[0]
    assert w.shape[1] == D and D % 256 == 0
    b = None if bias is None else np.asarray(bias, np.float32)
    lanes = np.arange(32)
    out = np.empty((T, E), np.float32)
    for t in range(T):
        prod = (w * x[t][None, :]).astype(np.float32)       # exact products
        prod = prod.reshape(E, D // 256, 32, 8)              # column = 256 i + 8 l + j
        s = None
        for g0 in range(0, D // 256, 4):                     # a segment: 1024 columns = 4 blocks of 256
            p = np.zeros((E, 32), np.float32)
            for i in range(g0, min(g0 + 4, D // 256)):
                for j in range(8):
                    p = (p + prod[:, i, :, j]).astype(np.float32)
            for o in (16, 8, 4, 2, 1):
                p = (p + p[:, lanes ^ o]).astype(np.float32)
            s = p[:, 0] if s is None else (s + p[:, 0]).astype(np.float32)
        if b is not None:
            s = (s + b).astype(np.float32)
        out[t] = s
    return out
