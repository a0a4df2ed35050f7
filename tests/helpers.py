"""Shared helpers of the GPU parity tests: build a layer from the seeded generators, run the
library through its C ABI, run the oracle on the same inputs, and measure the error."""
import numpy as np

import oracle
import synth

FFN_TOL = 2e-3   # normalised max error: max|delta_gpu - delta_ref| / max|delta_ref|


class Layer:
    """Inputs of one MoE layer: logits, x (bf16 bits), per-expert blobs, shared expert."""

    def __init__(self, wl, quantized=True, experts=None):
        self.wl = wl
        self.L, self.x = synth.draw_inputs(wl)
        if experts is None and not quantized:
            idx, _ = oracle.route(self.L, wl.k)
            experts = np.unique(idx)
        if quantized:
            E = range(wl.E)

            def one(e):
                return (oracle.quantize_iq2(synth.expert_weight(wl.seed, e, synth.GATE, wl.F, wl.D)),
                        oracle.quantize_iq2(synth.expert_weight(wl.seed, e, synth.UP, wl.F, wl.D)),
                        oracle.quantize_q2k(synth.expert_weight(wl.seed, e, synth.DOWN, wl.D, wl.F)))

            res = synth.parallel_map(one, E)
            self.gate = [r[0] for r in res]
            self.up = [r[1] for r in res]
            self.down = [r[2] for r in res]
        else:
            self.gate, self.up, self.down = synth.random_expert_blobs(wl, experts)
        self.shared = synth.shared_weights(wl.seed, wl.D, wl.F) if wl.shared else None

    def oracle_delta(self, tokens=None, mode=0):
        return oracle.moe_ffn(self.x, self.L, self.wl.k, self.gate, self.up, self.down, self.wl.D, self.wl.F,
                              shared=self.shared, mode=mode, tokens=tokens)

    def upload(self, ds4, max_tokens=None, max_k=None):
        return ds4.ds4moe_weights_create(self.gate, self.up, self.down, self.wl.D, self.wl.F, shared=self.shared,
                                         max_tokens=max_tokens or self.wl.T, max_k=max_k or self.wl.k)

    def run(self, ds4, W, out_init=None, mode=0):
        import torch
        x = torch.from_numpy(self.x.view(np.int16)).cuda().view(torch.bfloat16)
        logits = torch.from_numpy(self.L).cuda()
        out = torch.zeros((self.wl.T, self.wl.D), dtype=torch.float32, device="cuda")
        if out_init is not None:
            out.copy_(torch.from_numpy(out_init))
        ds4.ds4moe_expert_ffn(x, W, logits, self.wl.k, out, gate_mode=mode)
        st = ds4.ds4moe_last_status(W)
        assert st == 0, ds4.ds4moe_strerror(st)
        return out.cpu().numpy()


def sample_tokens(L, k, n_pos=64, n_ties=8, gemm_min=7):
    """Tokens for a sampled full-size parity check, chosen to reach the paths the kernels take:
    tokens whose pairs sit at n_pos evenly spread column positions of the largest group's 256-token
    tiles (cycling over its tiles), the first and the last pair of its last (ragged) tile, tokens of
    four one-token groups, four groups below gemm_min tokens and four groups from gemm_min to 64
    tokens, and the first n_ties tokens whose top two logits tie."""
    T, E = L.shape
    idx, _ = oracle.route(L, k)
    counts, offsets, perm, _ = oracle.permute(idx, E)
    big = int(np.argmax(counts))
    n = int(counts[big])
    ntile = (n + 255) // 256
    toks = set()
    for i, c in enumerate(range(0, 256, max(1, 256 // n_pos))):
        for j in range(ntile):
            r = ((i + j) % ntile) * 256 + c
            if r < n:
                toks.add(int(perm[offsets[big] + r]) // k)
                break
    last0 = (ntile - 1) * 256
    toks.add(int(perm[offsets[big] + last0]) // k)
    toks.add(int(perm[offsets[big] + n - 1]) // k)
    for lo, hi in ((1, 1), (2, gemm_min - 1), (gemm_min, 64)):
        for e in np.nonzero((counts >= lo) & (counts <= hi))[0][:4]:
            toks.add(int(perm[offsets[e]]) // k)
    o = np.argsort(-L, axis=1, kind="stable")
    tied = np.nonzero(L[np.arange(T), o[:, 0]] == L[np.arange(T), o[:, 1]])[0]
    toks.update(int(t) for t in tied[:n_ties])
    return sorted(toks)


def norm_max_err(got, ref):
    ref = np.asarray(ref, np.float64)
    return float(np.max(np.abs(np.asarray(got, np.float64) - ref)) / max(np.max(np.abs(ref)), 1e-30))
