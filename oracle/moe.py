"""Oracle expert FFN -- TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

What one routed-MoE layer's expert FFN computes, in fp64, with the weights taken as their
exact dequantised values and the activations as the bf16 values given:

  * per token, route to k experts (top-k of the router logits, gate weights g);
  * per selected expert e:  u = W_up x,  v = W_gate x,  h = silu(v) * u,  y = W_down h;
  * an always-on shared expert (weight 1, bf16 weights) computes y_sh the same way;
  * delta[t] = y_sh[t] + sum over slots s (in slot order) of g[t,s] * y[t,s];
    the layer output is the residual plus delta.

Sources: "DwarfStar" (ds4 README), "模型权重" (routed experts quantised, shared expert
unquantised); "DwarfStar 深度解析" §2.1 (per-token dynamic expert choice) and §3.4.3
(the expert tree: up/gate/down per routed expert, shared experts kept at full precision).
SwiGLU (silu(gate) * up) is the plain reading of the gate/up pair the pages list; the
pages do not spell the activation out.
"""
from concurrent.futures import ThreadPoolExecutor
import os

import numpy as np

from . import dequant_iq2, dequant_q2k, dequant_q4k, permute, route


def bf16_to_f64(bits):
    """bf16 bit patterns (uint16) to their exact fp64 values."""
    bits = np.asarray(bits, np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def silu(v):
    with np.errstate(over="ignore"):
        return v / (1.0 + np.exp(-v))


def expert_ffn_dense(x, w_gate, w_up, w_down):
    """One SwiGLU expert on rows x [n, D] (fp64) with dense fp64 weights
    w_gate, w_up [F, D] and w_down [D, F]. Returns y [n, D]."""
    u = x @ w_up.T
    v = x @ w_gate.T
    h = silu(v) * u
    return h @ w_down.T


def moe_ffn(x_bf16, logits, k, gate_blobs, up_blobs, down_blobs, d_model, d_ff,
            shared=None, mode=0, tokens=None, fmt="q2", threads=None):
    """Delta added to the residual by one routed-MoE expert FFN.

    x_bf16      uint16 [T, D] (bf16 bits);  logits float32 [T, E]
    gate_blobs, up_blobs: per expert, IQ2-style blobs of [d_ff, d_model]
    down_blobs: per expert, Q2_K-style blob of [d_model, d_ff]
    fmt:        "q2" (the above) or "q4": all three per-expert blobs Q4_K-style
    shared:     None, or (gate, up, down) bf16 bits of shapes [F, D], [F, D], [D, F]
    tokens:     None for all tokens, or the token ids to evaluate (others are not computed)
    threads:    experts evaluated at a time (default: the host's cores, at most 16)

    Returns (delta float64 [n_tokens, D], idx int32 [T, k], g float64 [T, k]).
    """
    T, E = logits.shape
    D, F = d_model, d_ff
    threads = threads or min(16, os.cpu_count() or 1)
    idx, g = route(logits, k, mode)
    counts, offsets, perm, _ = permute(idx, E)
    tok = np.arange(T) if tokens is None else np.asarray(tokens, np.int64)
    pos_of = {int(t): i for i, t in enumerate(tok)}
    x = bf16_to_f64(x_bf16)

    y = np.zeros((len(tok), k, D), np.float64)

    def one_expert(e):
        """The SwiGLU outputs of expert e for its evaluated pairs (rows, slots, y)."""
        pairs = perm[offsets[e]:offsets[e + 1]]
        pairs = [int(p) for p in pairs if int(p) // k in pos_of]
        if not pairs:
            return None
        if fmt == "q4":
            wg = dequant_q4k(gate_blobs[e], F, D).astype(np.float64)
            wu = dequant_q4k(up_blobs[e], F, D).astype(np.float64)
            wd = dequant_q4k(down_blobs[e], D, F).astype(np.float64)
        else:
            wg = dequant_iq2(gate_blobs[e], F, D).astype(np.float64)
            wu = dequant_iq2(up_blobs[e], F, D).astype(np.float64)
            wd = dequant_q2k(down_blobs[e], D, F).astype(np.float64)
        rows = np.array([pos_of[p // k] for p in pairs])
        slots = np.array([p % k for p in pairs])
        return rows, slots, expert_ffn_dense(x[tok[rows]], wg, wu, wd)

    # experts are independent: several at a time (threads; the C dequantisers and numpy's
    # matrix products release the interpreter lock), each written to its own (row, slot) cells
    with ThreadPoolExecutor(max(1, min(threads, E))) as ex:
        for res in ex.map(one_expert, range(E)):
            if res is not None:
                rows, slots, ye = res
                y[rows, slots] = ye

    delta = np.zeros((len(tok), D), np.float64)
    if shared is not None:
        sg, su, sd = (bf16_to_f64(s) for s in shared)
        delta += expert_ffn_dense(x[tok], sg.reshape(F, D), su.reshape(F, D), sd.reshape(D, F))
    gt = g[tok]
    for s in range(k):
        delta += gt[:, s:s + 1] * y[:, s, :]
    return delta, idx, g
