"""Streamed experts (pooled handles) on the GPU: results identical bit for bit to a resident
handle of the same weights, the slot table of the documented least-recently-used policy, the
hit and miss counters, and the capacity error."""
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


class LruModel:
    """The slot policy written out on the host: a touched expert that is resident keeps its
    slot; each missing one, in increasing expert order, takes the slot not used by this call
    whose last use is oldest (never used counts as oldest), ties to the lower slot."""

    def __init__(self, n_slots):
        self.expert_of = [-1] * n_slots
        self.last = [0] * n_slots
        self.call = 0
        self.hits = 0
        self.misses = 0

    def step(self, touched):
        touched = sorted(set(int(e) for e in touched))
        if len(touched) > len(self.expert_of):
            return False
        self.call += 1
        slot_of = {e: s for s, e in enumerate(self.expert_of) if e >= 0}
        used = {slot_of[e] for e in touched if e in slot_of}
        free = sorted((self.last[s], s) for s in range(len(self.expert_of)) if s not in used)
        nxt = 0
        for e in touched:
            if e in slot_of:
                self.hits += 1
                self.last[slot_of[e]] = self.call
            else:
                s = free[nxt][1]
                nxt += 1
                self.expert_of[s] = e
                self.last[s] = self.call
                self.misses += 1
        return True


def _handles(ds4, wl, n_slots, single_step=1):
    """A resident and a pooled handle of the same weights, both taking (single_step = 1) or both
    avoiding (0) the fused single-token kernel."""
    gate, up, down = synth.random_expert_blobs(wl)
    shared = synth.shared_weights(wl.seed, wl.D, wl.F) if wl.shared else None
    Wr = ds4.ds4moe_weights_create(gate, up, down, wl.D, wl.F, shared=shared, max_tokens=wl.T, max_k=wl.k)
    Wp = ds4.ds4moe_weights_create(gate, up, down, wl.D, wl.F, shared=shared, max_tokens=wl.T, max_k=wl.k,
                                   n_slots=n_slots)
    for W in (Wr, Wp):
        ds4.ds4moe_set_option(W, ds4.DS4MOE_OPT_SINGLE_STEP, single_step)
    return Wr, Wp, (gate, up, down, shared)


def _logits(rng, wl, favoured):
    """Logits whose top-k falls inside the favoured experts (a bias of +20 on them)."""
    L = rng.standard_normal((wl.T, wl.E)).astype(np.float32)
    L[:, favoured] += 20.0
    return L


@pytest.mark.parametrize("T,S,n_fav,fused,D,F", [(1, 12, 4, 1, 512, 2048), (1, 12, 6, 0, 512, 512),
                                                 (5, 12, 10, 1, 512, 512), (40, 32, 20, 1, 512, 512),
                                                 (300, 32, 32, 1, 512, 512)])
def test_pooled_handle_matches_resident_and_keeps_the_lru_table(ds4, T, S, n_fav, fused, D, F):
    # (the fused single-token kernel needs d_ff = 2048: the first case takes it on both handles)
    import torch
    wl = synth.Workload("pool", T=T, D=D, F=F, E=48, k=4, seed=700 + T + fused, shared=True)
    Wr, Wp, (gate, up, down, shared) = _handles(ds4, wl, S, fused)
    model = LruModel(S)
    rng = np.random.default_rng(wl.seed)
    xb = synth.f32_to_bf16_bits(rng.standard_normal((T, wl.D)).astype(np.float32))
    x = torch.from_numpy(xb.view(np.int16)).cuda().view(torch.bfloat16)
    for call in range(7):
        favoured = rng.choice(wl.E, n_fav, replace=False)
        L = _logits(rng, wl, favoured)
        Ld = torch.from_numpy(L).cuda()
        outs = []
        for W in (Wr, Wp):
            out = torch.zeros((T, wl.D), dtype=torch.float32, device="cuda")
            before = ds4.ds4moe_get_stats(W)["launches"]
            ds4.ds4moe_expert_ffn(x, W, Ld, wl.k, out)
            assert ds4.ds4moe_last_status(W) == 0
            if fused and T == 1 and W is Wr:  # the case meant for the fused kernel really takes it
                assert ds4.ds4moe_get_stats(W)["launches"] - before == 1
            outs.append(out.cpu().numpy())
        assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32)), "call %d" % call
        idx, _ = oracle.route(L, wl.k)
        assert model.step(np.unique(idx))
        n, hits, misses, slots = ds4.ds4moe_pool_info(Wp)
        assert n == S and list(slots) == model.expert_of, "call %d" % call
        assert (hits, misses) == (model.hits, model.misses)
    ref, _, _ = oracle.moe_ffn(xb, L, wl.k, gate, up, down, wl.D, wl.F, shared=shared,
                               tokens=None if T <= 40 else np.arange(0, T, 37))
    got = outs[1] if T <= 40 else outs[1][np.arange(0, T, 37)]
    assert norm_max_err(got, ref) <= FFN_TOL
    Wr.close()
    Wp.close()


def test_pooled_call_beyond_capacity_reports_and_changes_nothing(ds4):
    import torch
    wl = synth.Workload("pool_cap", T=8, D=256, F=256, E=32, k=4, seed=9, shared=False)
    Wr, Wp, _ = _handles(ds4, wl, 8)
    Wr.close()
    rng = np.random.default_rng(3)
    x = torch.from_numpy(synth.f32_to_bf16_bits(rng.standard_normal((8, wl.D)).astype(np.float32)).view(np.int16))
    x = x.cuda().view(torch.bfloat16)
    L = torch.from_numpy(rng.standard_normal((8, wl.E)).astype(np.float32)).cuda()  # touches > 8 experts
    out = torch.zeros((8, wl.D), dtype=torch.float32, device="cuda")
    ds4.ds4moe_expert_ffn(x, Wp, L, wl.k, out)
    assert ds4.ds4moe_last_status(Wp) == ds4.DS4MOE_ECAPACITY
    n, hits, misses, slots = ds4.ds4moe_pool_info(Wp)
    assert (hits, misses) == (0, 0) and list(slots) == [-1] * 8
    # a call that fits works afterwards
    out1 = torch.zeros((1, wl.D), dtype=torch.float32, device="cuda")
    ds4.ds4moe_expert_ffn(x[:1], Wp, L[:1], wl.k, out1)
    assert ds4.ds4moe_last_status(Wp) == 0
    assert ds4.ds4moe_pool_info(Wp)[2] == 4
    Wp.close()


def test_pooled_handle_refuses_the_entries_that_need_resident_experts(ds4):
    import torch
    wl = synth.Workload("pool_unsup", T=2, D=256, F=256, E=8, k=2, seed=5, shared=False)
    Wr, Wp, _ = _handles(ds4, wl, 4)
    dst = torch.empty((wl.F, wl.D), dtype=torch.float32, device="cuda")
    with pytest.raises(ds4.Ds4moeError) as e:
        ds4.ds4moe_weights_dequantize(Wp, 0, ds4.DS4MOE_GATE, dst_f32=dst)
    assert e.value.status == ds4.DS4MOE_EUNSUPPORTED
    with pytest.raises(ds4.Ds4moeError) as e:
        ds4.ds4moe_pool_info(Wr)
    assert e.value.status == ds4.DS4MOE_EINVAL
    Wr.close()
    Wp.close()
