"""Seeded synthetic inputs for the routed-MoE expert FFN.

Shared by the tests, the smoke check and the benchmark. This module holds none of the
method's arithmetic: it draws router logits, activations, fp32 expert weights and random
packed blocks; it never quantises, dequantises, routes, groups or multiplies. Where a
packed block's scale must be a valid fp16 number it is drawn in fp32 and converted with
numpy's own float16 cast.

Recipe (one ``numpy.random.default_rng(seed)`` per workload, draws in this order):
  1. logits L = standard_normal((T, E)) cast to fp32;
  2. bias: "normal" adds normal(0, sigma, E) (fp32); "zipf" adds -s * ln(r) with
     r = permutation(E) + 1, i.e. expert popularity proportional to r^-s;
  3. ties (fraction f of tokens): ids = choice(T, round(f*T), replace=False); for each id
     o = stable argsort(-L[t]); L[t, o[1]] = L[t, o[0]] and L[t, o[k]] = L[t, o[k-1]];
  4. x = standard_normal((T, D)) fp32, rounded to bf16 (nearest-even).
Expert weights come from a counter-based generator (Philox-4x64 as implemented by numpy)
keyed by (seed, expert, matrix), so any expert can be drawn alone: N(0, 0.02) in fp32,
gate/up [F, D] and down [D, F]. Shared-expert weights are drawn the same way with their
own key and rounded to bf16. The workloads stand in for one MoE layer of the pages'
DeepSeek-V4 workload; no public dataset is involved.
"""
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass
import os

import numpy as np

GATE, UP, DOWN = 0, 1, 2
SHARED_KEY = 0xFFFF


@dataclass(frozen=True)
class Workload:
    name: str
    T: int          # tokens
    D: int          # d_model
    F: int          # d_ff
    E: int          # routed experts
    k: int          # experts per token
    seed: int
    bias: tuple = ()        # () | ("normal", sigma) | ("zipf", s)
    tie_frac: float = 0.0   # fraction of tokens with forced exact logit ties
    shared: bool = True     # one always-on bf16 shared expert of the same shape
    slots: int = 0          # > 0: experts stream from host memory into this many device slots
    ring: int = 1           # distinct inputs cycled through, one per step (seeds seed .. seed+ring-1)
    fmt: str = "q2"         # "q2": IQ2-style gate/up + Q2_K-style down; "q4": the 4-bit variant

    def replace(self, **kw):
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


WORKLOADS = {
    w.name: w for w in [
        Workload("tiny_t4", T=4, D=256, F=256, E=8, k=2, seed=0, shared=False),
        Workload("decode_t1", T=1, D=4096, F=2048, E=256, k=8, seed=1),
        Workload("decode_t32", T=32, D=4096, F=2048, E=256, k=8, seed=2, bias=("normal", 0.5)),
        Workload("prefill_t2048", T=2048, D=4096, F=2048, E=256, k=8, seed=3, bias=("zipf", 1.0)),
        Workload("prefill_t8192_d7168", T=8192, D=7168, F=2048, E=256, k=8, seed=4,
                 bias=("zipf", 1.2), tie_frac=0.05),
        # decode with cold experts: 64 of the 256 experts fit in device memory, and each step is
        # a different token, so most of its experts must be copied in from host memory
        Workload("decode_t1_cold", T=1, D=4096, F=2048, E=256, k=8, seed=11, slots=64, ring=64),
        # the 4-bit variant at the decode shape: Q4_K-style gate, up and down
        Workload("decode_t1_q4", T=1, D=4096, F=2048, E=256, k=8, seed=12, fmt="q4"),
        Workload("prefill_t2048_q4", T=2048, D=4096, F=2048, E=256, k=8, seed=13, bias=("zipf", 1.0), fmt="q4"),
        # a profiling stand-in for the tensor-core kernels at d_model 7168: groups of about a
        # thousand tokens (mostly full 256-token tiles, as in the large prefill chunk's big
        # groups) on a device footprint of about 1.5 GB
        Workload("prefill_t2048_d7168_e16", T=2048, D=7168, F=2048, E=16, k=8, seed=14, bias=("zipf", 1.2)),
    ]
}


def f32_to_bf16_bits(a):
    """fp32 -> bf16 bit patterns, round to nearest-even (finite inputs)."""
    u = np.ascontiguousarray(a, np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def draw_inputs(wl):
    """Router logits float32 [T, E] and activations as bf16 bits uint16 [T, D]."""
    rng = np.random.default_rng(wl.seed)
    L = rng.standard_normal((wl.T, wl.E)).astype(np.float32)
    if wl.bias:
        kind, p = wl.bias
        if kind == "normal":
            L += rng.normal(0.0, p, wl.E).astype(np.float32)
        elif kind == "zipf":
            r = rng.permutation(wl.E) + 1
            L += (-p * np.log(r)).astype(np.float32)
        else:
            raise ValueError(kind)
    if wl.tie_frac > 0:
        n = int(round(wl.tie_frac * wl.T))
        ids = rng.choice(wl.T, n, replace=False)
        for t in ids:
            o = np.argsort(-L[t], kind="stable")
            L[t, o[1]] = L[t, o[0]]
            L[t, o[wl.k]] = L[t, o[wl.k - 1]]
    x = f32_to_bf16_bits(rng.standard_normal((wl.T, wl.D)).astype(np.float32))
    return L, x


def router_weights(wl):
    """A seeded router for the workload: bf16 bits [E, D] drawn N(0, 1/sqrt(D)), so that with
    x ~ N(0, 1) the logits spread like the drawn ones (unit variance), and an fp32 bias [E] of the
    workload's per-expert kind (Zipf -s log(rank) over a random expert order, N(0, p), or zero),
    so that routing on the computed logits has the workload's group-size mix."""
    rng = np.random.default_rng(wl.seed + 7919)
    w = f32_to_bf16_bits((rng.standard_normal((wl.E, wl.D)) / np.sqrt(wl.D)).astype(np.float32))
    b = np.zeros(wl.E, np.float32)
    if wl.bias:
        kind, p = wl.bias
        if kind == "normal":
            b = rng.normal(0.0, p, wl.E).astype(np.float32)
        elif kind == "zipf":
            b = (-p * np.log(rng.permutation(wl.E) + 1)).astype(np.float32)
        else:
            raise ValueError(kind)
    return w, b


def _gen(seed, a, b):
    return np.random.Generator(np.random.Philox(key=[int(seed), (int(a) << 8) | int(b)]))


def expert_weight(seed, expert, which, rows, cols, std=0.02):
    """N(0, std) fp32 matrix [rows, cols] for one routed expert's gate/up/down."""
    g = _gen(seed, expert, which)
    return g.standard_normal((rows, cols), dtype=np.float32) * np.float32(std)


def shared_weights(seed, D, F, std=0.02):
    """bf16 bits of the shared expert: gate [F, D], up [F, D], down [D, F]."""
    out = []
    for which, shape in ((GATE, (F, D)), (UP, (F, D)), (DOWN, (D, F))):
        g = _gen(seed, SHARED_KEY, which)
        out.append(f32_to_bf16_bits(g.standard_normal(shape, dtype=np.float32) * np.float32(std)))
    return tuple(out)


def _rand_bytes(seed, expert, which, nbytes):
    g = np.random.Philox(key=[int(seed), (1 << 40) | (int(expert) << 8) | int(which)])
    n64 = (nbytes + 7) // 8
    return g.random_raw(n64).view(np.uint8)[:nbytes].copy(), np.random.Generator(g)


def random_iq2_blob(seed, expert, which, rows, cols):
    """Random IQ2-style blocks (66 B each) with fp16 scales d drawn so that the weights have
    a spread like N(0, 0.02): every field except d is uniform random bits."""
    nb = rows * cols // 256
    b, g = _rand_bytes(seed, expert, which, nb * 66)
    b = b.reshape(nb, 66)
    d = (np.float32(0.0075) * (np.float32(0.5) + g.random(nb, dtype=np.float32))).astype(np.float16)
    b[:, 0:2] = d.view(np.uint8).reshape(nb, 2)
    return b.reshape(-1)


def random_q2k_blob(seed, expert, which, rows, cols):
    """Random Q2_K-style blocks (84 B each) with fp16 d and dmin drawn so that the weights
    have a spread like N(0, 0.02) and roughly zero mean."""
    nb = rows * cols // 256
    b, g = _rand_bytes(seed, expert, which, nb * 84)
    b = b.reshape(nb, 84)
    d = np.float32(0.003) * (np.float32(0.5) + g.random(nb, dtype=np.float32))
    dmin = d * np.float32(1.5) * (np.float32(0.75) + np.float32(0.5) * g.random(nb, dtype=np.float32))
    b[:, 80:82] = d.astype(np.float16).view(np.uint8).reshape(nb, 2)
    b[:, 82:84] = dmin.astype(np.float16).view(np.uint8).reshape(nb, 2)
    return b.reshape(-1)


def random_q4k_blob(seed, expert, which, rows, cols):
    """Random Q4_K-style blocks (144 B each, the 4-bit variant) with fp16 d and dmin drawn so
    that the weights spread like N(0, 0.02) with roughly zero mean (mean code 7.5, mean 6-bit
    scale and min about 31)."""
    nb = rows * cols // 256
    b, g = _rand_bytes(seed, expert, which, nb * 144)
    b = b.reshape(nb, 144)
    d = np.float32(0.7e-4) * (np.float32(0.5) + g.random(nb, dtype=np.float32))
    dmin = d * np.float32(7.5) * (np.float32(0.75) + np.float32(0.5) * g.random(nb, dtype=np.float32))
    b[:, 0:2] = d.astype(np.float16).view(np.uint8).reshape(nb, 2)
    b[:, 2:4] = dmin.astype(np.float16).view(np.uint8).reshape(nb, 2)
    return b.reshape(-1)


def random_q4_expert_blobs(wl, experts=None, seed_offset=0):
    """As random_expert_blobs, for the 4-bit variant: Q4_K-style gate, up and down blobs."""
    experts = range(wl.E) if experts is None else sorted(set(int(e) for e in experts))
    s = wl.seed + seed_offset
    gate, up, down = [None] * wl.E, [None] * wl.E, [None] * wl.E

    def one(e):
        return (e, random_q4k_blob(s, e, GATE, wl.F, wl.D), random_q4k_blob(s, e, UP, wl.F, wl.D),
                random_q4k_blob(s, e, DOWN, wl.D, wl.F))

    for e, a, b, c in parallel_map(one, experts):
        gate[e], up[e], down[e] = a, b, c
    z = np.zeros(wl.F * wl.D // 256 * 144, np.uint8)
    for e in range(wl.E):
        if gate[e] is None:
            gate[e], up[e], down[e] = z, z, z
    return gate, up, down


def parallel_map(fn, items, threads=None):
    """Run fn over items with a thread pool (numpy's generators release the GIL)."""
    threads = threads or min(32, os.cpu_count() or 1)
    with ThreadPoolExecutor(threads) as ex:
        return list(ex.map(fn, items))


def random_expert_blobs(wl, experts=None, seed_offset=0):
    """Random packed blobs for the given experts (default: all). Returns three lists of
    length E (gate, up, down); experts not listed get all-zero blocks."""
    experts = range(wl.E) if experts is None else sorted(set(int(e) for e in experts))
    s = wl.seed + seed_offset
    nbi = wl.F * wl.D // 256 * 66
    nbq = wl.D * wl.F // 256 * 84
    gate = [None] * wl.E
    up = [None] * wl.E
    down = [None] * wl.E

    def one(e):
        return (e, random_iq2_blob(s, e, GATE, wl.F, wl.D), random_iq2_blob(s, e, UP, wl.F, wl.D),
                random_q2k_blob(s, e, DOWN, wl.D, wl.F))

    for e, a, b, c in parallel_map(one, experts):
        gate[e], up[e], down[e] = a, b, c
    zi = np.zeros(nbi, np.uint8)
    zq = np.zeros(nbq, np.uint8)
    for e in range(wl.E):
        if gate[e] is None:
            gate[e], up[e], down[e] = zi, zi, zq
    return gate, up, down
