#!/usr/bin/env python
"""Benchmark of the routed-MoE expert FFN over 2-bit experts on one or more GB300s.

A step is one call of ds4moe_expert_ffn over one batch of synthetic input: routing,
grouping, the SwiGLU experts (packed 2-bit routed experts plus the bf16 shared expert) and
the gate-weighted combine. The default workload is the largest single-GPU configuration, the
prefill chunk of 8192 tokens (d_model 7168, d_ff 2048, 256 experts, top-8, Zipf s=1.2 routing
with 5% tied tokens, bf16 shared expert); --workload picks another (decode_t1 is single-token
decode). Under torchrun every rank runs an independent replica (no data-path collective; weak
scaling).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Prints one JSON line. --impl reference times the oracle (the plain fp64 CPU restatement)
on the host cores on the same workload and metric.
"""
import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

L2_BYTES = 129 * 10 ** 6
METRIC = "routed-MoE tokens/s"
IQ2_PER_EXPERT = lambda D, F: 2 * F * D // 256 * 66  # noqa: E731  gate + up
Q2K_PER_EXPERT = lambda D, F: D * F // 256 * 84      # noqa: E731  down
Q4_UP_PER_EXPERT = lambda D, F: 2 * F * D // 256 * 144  # noqa: E731  gate + up, the 4-bit variant
Q4_DOWN_PER_EXPERT = lambda D, F: D * F // 256 * 144    # noqa: E731  down, the 4-bit variant


def up_per_expert(wl):
    return Q4_UP_PER_EXPERT(wl.D, wl.F) if wl.fmt == "q4" else IQ2_PER_EXPERT(wl.D, wl.F)


def down_per_expert(wl):
    return Q4_DOWN_PER_EXPERT(wl.D, wl.F) if wl.fmt == "q4" else Q2K_PER_EXPERT(wl.D, wl.F)


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="prefill_t8192_d7168", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--weights", choices=["quantized", "random"], default=None,
                    help="routed-expert blobs: host-quantised N(0,0.02) (default for decode) or random valid blocks")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--cpu-worker", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--router", action="store_true",
                    help="a step also computes the router logits on the device (bf16 router, fp32 bias) in "
                         "front of routing, instead of taking the workload's logits")
    ap.add_argument("--calls", type=int, default=0,
                    help="run the workload's call this many times (no timing, no JSON line) and exit: "
                         "a fixed launch sequence for profilers")
    return ap.parse_args(argv)


# ------------------------------------------------------------------ multi-rank plumbing

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def reduce_max(value, world, device=None):
    """Max of a float over ranks (a timing reduction, not part of the data path)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def whole_job_rate(units_per_rank, world, max_seconds):
    """Units processed by all ranks divided by the slowest rank's time."""
    return units_per_rank * world / max_seconds


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        # the raw samples (nvidia-smi CSV); the JSON line carries their summary
        self.path = os.path.join(tempfile.gettempdir(), "ds4moe_clocks_%d.csv" % os.getpid())

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if not self.proc:
            return None
        rows = []
        for line in open(self.path):
            p = [s.strip() for s in line.split(",")]
            if len(p) >= 9 and p[1].replace(".", "").isdigit():
                rows.append(p)
        if not rows:
            return None
        mhz = [float(r[1]) for r in rows]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": float(rows[0][2]),
                "reasons": sorted(reasons), "samples": len(rows)}


# ------------------------------------------------------------------ workload set-up

def touched_experts(ds4, wl, L):
    import torch
    idx, _ = ds4.ds4moe_route(torch.from_numpy(L).cuda(), wl.k)
    return sorted(set(idx.cpu().numpy().reshape(-1).tolist()))


def make_weights(ds4, wl, experts, mode):
    """Blobs for every expert: the touched ones quantised from N(0, 0.02) by the library's
    host quantiser (or random valid blocks), the others all-zero blocks (never read)."""
    if wl.fmt == "q4":
        if mode == "random":
            return synth.random_q4_expert_blobs(wl, experts)
        z = np.zeros(ds4.ds4moe_q4k_bytes(wl.F, wl.D), np.uint8)
        gate, up, down = [z] * wl.E, [z] * wl.E, [z] * wl.E
        for e in experts:
            gate[e] = ds4.ds4moe_quantize_q4k(synth.expert_weight(wl.seed, e, synth.GATE, wl.F, wl.D))
            up[e] = ds4.ds4moe_quantize_q4k(synth.expert_weight(wl.seed, e, synth.UP, wl.F, wl.D))
            down[e] = ds4.ds4moe_quantize_q4k(synth.expert_weight(wl.seed, e, synth.DOWN, wl.D, wl.F))
        return gate, up, down
    if mode == "random":
        return synth.random_expert_blobs(wl, experts)
    nbi = ds4.ds4moe_iq2_bytes(wl.F, wl.D)
    nbq = ds4.ds4moe_q2k_bytes(wl.D, wl.F)
    zi, zq = np.zeros(nbi, np.uint8), np.zeros(nbq, np.uint8)
    gate, up, down = [zi] * wl.E, [zi] * wl.E, [zq] * wl.E
    for e in experts:
        gate[e] = ds4.ds4moe_quantize_iq2(synth.expert_weight(wl.seed, e, synth.GATE, wl.F, wl.D))
        up[e] = ds4.ds4moe_quantize_iq2(synth.expert_weight(wl.seed, e, synth.UP, wl.F, wl.D))
        down[e] = ds4.ds4moe_quantize_q2k(synth.expert_weight(wl.seed, e, synth.DOWN, wl.D, wl.F))
    return gate, up, down


def small_path(wl):
    """Whether a multi-token call runs its small groups on the small-group kernels (the library's
    default for d_model <= 4096 and d_ff <= 2048)."""
    return wl.T > 1 and wl.D <= 4096 and wl.F <= 2048 and wl.fmt == "q2"


def gemm_rows(wl, counts):
    """Token rows the tensor-core GEMMs take in one call under the library's default dispatch:
    the routed groups of at least the threshold's tokens (every expert's weights fit fp16 here),
    plus the shared expert's T rows from 2 tokens on (its gate/up on the warp-MMA kernel up to
    48 tokens: (routed rows, shared rows of the up GEMM, shared rows of the down GEMM))."""
    T = wl.T
    if wl.fmt == "q4":
        gm = 0 if T <= 64 else 2
    elif small_path(wl):
        gm = 0 if T <= 64 else 7
    else:
        gm = 2
    routed = int(counts[counts >= gm].sum()) if gm > 0 and T >= gm else 0
    sh_down = T if wl.shared and T >= 2 else 0
    sh_up = 0 if small_path(wl) and T <= 48 else sh_down
    return routed, sh_up, sh_down


def algorithmic(wl, counts):
    """Bytes and FLOPs the method must move / compute for one call, per stage."""
    D, F, T, k = wl.D, wl.F, wl.T, wl.k
    touched = int(np.count_nonzero(counts))
    P = T * k
    sh_up = 2 * F * D * 2 if wl.shared else 0
    sh_down = D * F * 2 if wl.shared else 0
    rows = P + (T if wl.shared else 0)
    up_bytes = touched * up_per_expert(wl) + sh_up + T * D * 2 + rows * F * 4
    down_bytes = touched * down_per_expert(wl) + sh_down + rows * F * 4 + rows * D * 4
    if small_path(wl):
        # the small-group kernels' stages: routed groups below the tensor-core threshold only (the
        # shared expert and larger groups run in the tensor-core stages)
        gm = 0 if T <= 64 else 7
        sel = (counts > 0) & ((counts < gm) if gm else True)
        n_small, p_small = int(np.count_nonzero(sel)), int(counts[sel].sum())
        up_bytes = n_small * IQ2_PER_EXPERT(D, F) + T * D * 2 + p_small * F * 4
        down_bytes = n_small * Q2K_PER_EXPERT(D, F) + p_small * F * 4 + p_small * D * 4
    # the tensor-core stages' FLOPs: the rows those kernels ran, not every pair of the call
    r_tc, sh_up_tc, sh_down_tc = gemm_rows(wl, counts)
    flops_up = 2 * 2 * F * D * (r_tc + sh_up_tc)
    flops_down = 2 * D * F * (r_tc + sh_down_tc)
    flops_call = 6 * D * F * rows
    act_bytes = T * D * 2 + T * wl.E * 4 + 2 * T * D * 4 + 2 * rows * F * 4   # x, logits, out, h
    return {"touched": touched, "up_bytes": up_bytes, "down_bytes": down_bytes, "act_bytes": act_bytes,
            "total_bytes": touched * (up_per_expert(wl) + down_per_expert(wl)) + sh_up + sh_down,
            "flops_up": flops_up, "flops_down": flops_down, "flops_call": flops_call}


def _include_closure(names):
    """The kernel source files and every header they include, directly or through another
    header (quoted includes, resolved against the including file's folder), in a fixed order."""
    csrc = os.path.join(ROOT, "bit_quantized_routed_gb300", "csrc")
    todo = [os.path.normpath(os.path.join(csrc, n)) for n in names]
    seen = []
    while todo:
        f = todo.pop(0)
        if f in seen:
            continue
        seen.append(f)
        with open(f) as fh:
            for line in fh:
                m = re.match(r'\s*#\s*include\s+"([^"]+)"', line)
                if m:
                    todo.append(os.path.normpath(os.path.join(os.path.dirname(f), m.group(1))))
    return sorted(seen)


def src_sha(*names):
    """Hash of a kernel's source file and the headers it includes: a traffic record is reported
    only while this matches the one taken with it."""
    h = hashlib.sha256()
    for f in _include_closure(names):
        h.update(os.path.relpath(f, ROOT).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


STAGE_KERNEL = {"step": ("decode_step_kernel", "decode_step.cu"),
                "up_gemm": ("gemm_kernel<UP>", "gemm_tc.cu"), "down_gemm": ("gemm_kernel<DOWN>", "gemm_tc.cu"),
                "pool": ("pool_fill_kernel", "pool.cu"),
                "up_gemv": ("decode_up_kernel", "decode.cu"), "down_gemv": ("decode_down_kernel", "decode.cu"),
                "combine": ("combine_kernel", "combine.cu"), "route": ("route_kernel", "route_group.cu"),
                "group": ("group_kernel", "route_group.cu")}


SMALL_STAGE_KERNEL = {"up_gemv": ("small_up_kernel", "small_groups.cu"),
                      "down_gemv": ("small_down_kernel", "small_groups.cu")}


Q4_STAGE_KERNEL = {"up_gemv": ("gemv_up_kernel", "gemv.cu"), "down_gemv": ("gemv_down_kernel", "gemv.cu")}
# one token: the streamed GEMV kernels (when their shared-memory ring fits the shape)
Q4_T1_STAGE_KERNEL = {"up_gemv": ("gemv_up_stream_kernel", "gemv.cu"), "down_gemv": ("gemv_down_stream_kernel", "gemv.cu")}


def stage_kernel(stage, wl):
    if wl.fmt == "q4" and wl.T == 1 and stage in Q4_T1_STAGE_KERNEL:
        return Q4_T1_STAGE_KERNEL[stage]
    if wl.fmt == "q4" and stage in Q4_STAGE_KERNEL:
        return Q4_STAGE_KERNEL[stage]
    if small_path(wl) and stage in SMALL_STAGE_KERNEL:
        return SMALL_STAGE_KERNEL[stage]
    return STAGE_KERNEL.get(stage, (stage, None))


def ncu_traffic(stage, workload):
    """dram read+write bytes per launch from the committed ncu summary, if the kernel
    source is unchanged since the capture."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    kern, src = stage_kernel(stage, synth.WORKLOADS[workload])
    if src is None or not os.path.exists(path):
        return None
    rec = json.load(open(path)).get("%s@%s" % (kern, workload))
    if not rec or rec.get("src_sha") != src_sha(src):
        return None
    return rec.get("bytes_per_launch")


def e2e_pipelined(step_on, stream, K, xh, Lh, out_in, out_h, xd, Ld, out, copy_logits):
    """K steps through the public API with their host copies, overlapped across steps: two sets of
    device buffers; step i's inputs (x, the logits unless the router computes them, the residual)
    are copied in on one stream once the read-back of step i-2 (same buffers) is done, the call
    runs on the compute stream once they are in, and its result is read back on a third stream.
    Returns the milliseconds from the first copy-in to the last read-back (CUDA events)."""
    import torch
    bufs = [(xd, Ld, out), (torch.empty_like(xd), torch.empty_like(Ld), torch.empty_like(out))]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    h2d_done = [torch.cuda.Event() for _ in range(K)]
    comp_done = [torch.cuda.Event() for _ in range(K)]
    d2h_done = [torch.cuda.Event() for _ in range(K)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(s_in)
    for i in range(K):
        xb, Lb, ob = bufs[i % 2]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(d2h_done[i - 2])
            xb.copy_(xh, non_blocking=True)
            if copy_logits:
                Lb.copy_(Lh, non_blocking=True)
            ob.copy_(out_in, non_blocking=True)
            h2d_done[i].record(s_in)
        stream.wait_event(h2d_done[i])
        with torch.cuda.stream(stream):
            step_on(xb, Lb, ob)
            comp_done[i].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[i])
            out_h.copy_(ob, non_blocking=True)
            d2h_done[i].record(s_out)
    s_out.wait_event(d2h_done[K - 1])
    t1.record(s_out)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        p = json.load(open(path))
        return p["hbm_gbs"], p["bf16_tflops"], "measured"
    return 6800.0, 1900.0, "fallback"


def default_weights(wl, args):
    """Routed-expert blobs of a run: host-quantised N(0, 0.02) for decode-sized workloads, random
    valid blocks (same kernels, same time) for the large ones, unless --weights says otherwise."""
    return args.weights or ("quantized" if wl.T <= 32 else "random")


def config_dict(wl, mode, touched, flush, world, router):
    """The workload's description in the JSON line (the same for both arms)."""
    return {"workload": wl.name, "tokens": wl.T, "d_model": wl.D, "d_ff": wl.F, "experts": wl.E,
            "top_k": wl.k, "shared_expert": "bf16" if wl.shared else None,
            "routed_weights": ("4-bit Q4_K-style gate/up/down, " if wl.fmt == "q4" else
                               "2-bit IQ2-style gate/up + Q2_K-style down, ") +
                              ("host-quantised N(0,0.02)" if mode == "quantized" else "random valid blocks"),
            "experts_touched": touched,
            "l2": "flushed between steps (write then read 256 MB)" if flush else "working set > 4x L2",
            "parallelism": "replicas" if world > 1 else "single GPU",
            **({"router": "bf16 [E x D] + fp32 bias, logits computed on the device in front of routing"}
               if router else {})}


def reference_config(args, world):
    """Our arm's config dict for the reference arm's line, computed on the host: the experts the
    workload touches come from the oracle's routing of the same logits."""
    import oracle
    wl = synth.WORKLOADS[args.workload]
    if wl.slots:   # the pooled workload's line describes its pool instead; the plain keys are shared
        return {"workload": wl.name, "tokens": wl.T, "d_model": wl.D, "d_ff": wl.F, "experts": wl.E,
                "top_k": wl.k}
    L, _ = synth.draw_inputs(wl)
    idx = oracle.route(L, wl.k)[0]
    touched = int(np.unique(idx).size)
    counts = np.bincount(idx.reshape(-1), minlength=wl.E)
    alg = algorithmic(wl, counts)
    flush = alg["total_bytes"] < 4 * L2_BYTES
    return config_dict(wl, default_weights(wl, args), touched, flush, world, args.router)


# ------------------------------------------------------------------ our arm

def capture(fn):
    """CUDA graph of one call of fn on the current device."""
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def run_ours(args):
    import torch
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    import bit_quantized_routed_gb300 as ds4
    ds4.build()
    wl = synth.WORKLOADS[args.workload]
    if world > 1:
        wl = wl.replace(seed=wl.seed + 1000 * rank)   # each replica its own batch
    if wl.slots:
        return run_pooled(args, wl)
    mode = default_weights(wl, args)
    L, x = synth.draw_inputs(wl)
    xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    if args.router:
        # a seeded bf16 router and fp32 bias with the workload's routing mix; the logits the step
        # routes on are computed on the device from x
        wr, br = synth.router_weights(wl)
        wrd = torch.from_numpy(wr.view(np.int16)).cuda().view(torch.bfloat16)
        brd = torch.from_numpy(br).cuda()
        L = ds4.ds4moe_router_logits(xd, wrd, brd).cpu().numpy()
    experts = touched_experts(ds4, wl, L)
    gate, up, down = make_weights(ds4, wl, experts, mode)
    shared = synth.shared_weights(wl.seed, wl.D, wl.F) if wl.shared else None
    W = ds4.ds4moe_weights_create(gate, up, down, wl.D, wl.F, shared=shared, max_tokens=wl.T, max_k=wl.k,
                                  fmt=wl.fmt)
    del gate, up, down
    Ld = torch.from_numpy(L).cuda()
    out = torch.zeros((wl.T, wl.D), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    counts, _, _, _ = ds4.ds4moe_group(ds4.ds4moe_route(Ld, wl.k)[0], wl.E)
    alg = algorithmic(wl, counts.cpu().numpy())
    if args.router:
        alg["total_bytes"] += wl.E * wl.D * 2 + wl.E * 4   # the router's weights and bias
    flush = alg["total_bytes"] < 4 * L2_BYTES
    if flush:
        fw = torch.empty(256 * 2 ** 20, dtype=torch.uint8, device="cuda")
        fr = torch.ones(64 * 2 ** 20, dtype=torch.float32, device="cuda")

    def l2_flush():
        fw.zero_()           # write more than L2 ...
        fr.sum()             # ... then read more than L2, so no dirty line is left behind

    def step_on(xb, Lb, ob):
        if args.router:
            ds4.ds4moe_router_logits(xb, wrd, brd, logits=Lb)
        ds4.ds4moe_expert_ffn(xb, W, Lb, wl.k, ob)

    def step():
        step_on(xd, Ld, out)

    if args.calls:
        for _ in range(args.calls):
            if flush:
                l2_flush()
            step()
        torch.cuda.synchronize()
        st = ds4.ds4moe_last_status(W)
        W.close()
        if st:
            raise RuntimeError(ds4.ds4moe_strerror(st))
        return
    for _ in range(max(3, args.warmup)):
        if flush:
            l2_flush()
        step()
    st = ds4.ds4moe_last_status(W)
    if st:
        raise RuntimeError(ds4.ds4moe_strerror(st))
    before = ds4.ds4moe_get_stats(W)["launches"]
    step()
    launches_per_call = ds4.ds4moe_get_stats(W)["launches"] - before + (1 if args.router else 0)

    # The call is replayed as a CUDA graph, so the device time of a step is not
    # stretched by host-side launch latency.
    graph = capture(step)
    for _ in range(max(3, args.warmup)):
        if flush:
            l2_flush()
        graph.replay()

    # ---- timed region: K steps, device time from CUDA events on the launching stream
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    with ClockSampler(local) as clocks:
        torch.cuda.synchronize()
        barrier(world)
        for i in range(K):
            if flush:
                l2_flush()
            ev[i][0].record(stream)
            graph.replay()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        barrier(world)
    launches = launches_per_call * K
    dev_ms = sum(a.elapsed_time(b) for a, b in ev)
    max_ms = reduce_max(dev_ms, world, "cuda")
    value = whole_job_rate(K * wl.T, world, max_ms / 1e3)

    # ---- per-stage device times: events at each stage boundary on the launching stream. A
    # short device-side spin ahead of each step lets the host queue all of the step's launches
    # before the GPU reaches them, so no stage waits for the host.
    ds4.ds4moe_set_option(W, ds4.DS4MOE_OPT_PROFILE, 1)
    stage_tot = {n: 0.0 for n in ds4.STAGES}
    for i in range(K):
        if flush:
            l2_flush()
        torch.cuda._sleep(400000)
        step()
        for n, v in ds4.ds4moe_get_stats(W)["stage_ms"].items():
            stage_tot[n] += v
    ds4.ds4moe_set_option(W, ds4.DS4MOE_OPT_PROFILE, 0)
    dom = max(stage_tot, key=stage_tot.get)
    dom_ms = stage_tot[dom] / K
    if launches_per_call == 1:
        # one kernel per call: its launch duration is the timed step itself (CUDA events on the
        # launching stream around each replay of the timed region)
        dom_ms = max_ms / K

    # ---- end to end through the public API: pinned host buffers, copies inside the region
    xh = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory()
    Lh = torch.from_numpy(L).pin_memory()
    out_in = torch.zeros((wl.T, wl.D), dtype=torch.float32).pin_memory()
    out_h = torch.empty((wl.T, wl.D), dtype=torch.float32).pin_memory()
    e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    torch.cuda.synchronize()
    for i in range(K):
        if flush:
            l2_flush()
        e2e_ev[i][0].record(stream)
        xd.copy_(xh, non_blocking=True)
        if not args.router:
            Ld.copy_(Lh, non_blocking=True)
        out.copy_(out_in, non_blocking=True)
        step()
        out_h.copy_(out, non_blocking=True)
        e2e_ev[i][1].record(stream)
    torch.cuda.synchronize()
    e2e_serial_ms = reduce_max(sum(a.elapsed_time(b) for a, b in e2e_ev), world, "cuda")
    e2e_ms, e2e_mode = e2e_serial_ms, "serial: each step's copies, call and read-back in order on one stream"
    if not flush:
        e2e_ms = e2e_pipelined(step_on, stream, K, xh, Lh, out_in, out_h, xd, Ld, out, not args.router)
        e2e_ms = reduce_max(e2e_ms, world, "cuda")
        e2e_mode = ("pipelined: two sets of device buffers; step i's inputs are copied in on one stream while "
                    "step i-1 computes, and its result is read back on another while step i+1 computes; "
                    "the time is the span from the first copy-in to the last read-back")
    h2d = wl.T * wl.D * 2 + (0 if args.router else wl.T * wl.E * 4) + wl.T * wl.D * 4
    d2h = wl.T * wl.D * 4
    st = ds4.ds4moe_last_status(W)
    if st:
        raise RuntimeError(ds4.ds4moe_strerror(st))

    hbm, tflops, peak_src = load_peaks()
    if dom in ("step", "up_gemv", "down_gemv", "combine", "route", "group"):
        b = alg["up_bytes"] if dom == "up_gemv" else alg["down_bytes"] if dom == "down_gemv" else None
        if dom == "step":  # the whole single-token call in one kernel
            b = alg["total_bytes"] + alg["act_bytes"]
        if dom == "combine":
            b = (wl.T * wl.k + wl.T) * wl.D * 4 + 2 * wl.T * wl.D * 4
        achieved = (b / (dom_ms / 1e3) / 1e9) if b else None
        roof = {"bound": "hbm", "kernel": stage_kernel(dom, wl)[0], "achieved": achieved, "peak": hbm,
                "unit": "GB/s", "frac": (achieved / hbm) if achieved else None,
                "traffic": ncu_traffic(dom, wl.name), "algorithmic_bytes": b, "avg_launch_ms": dom_ms,
                "peak_source": peak_src}
    else:
        f = alg["flops_up"] if dom == "up_gemm" else alg["flops_down"]
        achieved = f / (dom_ms / 1e3) / 1e12
        roof = {"bound": "tensor", "kernel": "gemm_kernel<UP>" if dom == "up_gemm" else "gemm_kernel<DOWN>", "achieved": achieved, "peak": tflops, "unit": "TFLOP/s",
                "frac": achieved / tflops, "traffic": ncu_traffic(dom, wl.name), "algorithmic_flops": f, "avg_launch_ms": dom_ms,
                "peak_source": peak_src}
    roof["stage_ms"] = {n: round(v / K, 5) for n, v in stage_tot.items() if v > 0}
    roof["call_hbm_gbs"] = alg["total_bytes"] / (max_ms / K / 1e3) / 1e9
    roof["call_hbm_frac"] = roof["call_hbm_gbs"] / hbm

    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
            "warmup": max(3, args.warmup), "ms_per_step": max_ms / K, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            # the arithmetic of the dominant stage: fp16 tensor-core operands (fp32 accumulate), or fp32
            "dtype": "f16" if roof["bound"] == "tensor" else "f32", "data": "synthetic",
            "config": config_dict(wl, mode, alg["touched"], flush, world, args.router),
            "gpu_launches": int(launches),
            "e2e": {"value": whole_job_rate(K * wl.T, world, e2e_ms / 1e3), "unit": "tokens/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "mode": e2e_mode,
                    "serial_value": whole_job_rate(K * wl.T, world, e2e_serial_ms / 1e3)},
            "roofline": roof, "clocks": clocks.summary()}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload, args.cpu_seconds)
    W.close()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_pooled(args, wl):
    """Decode with cold experts: a pooled handle (wl.slots expert slots in device memory in front
    of the host-resident store) and a ring of wl.ring seeded tokens, step i taking token i mod
    ring, so successive steps route to different experts and each step copies its missing experts
    in from host memory before computing. Expert blocks are random valid blocks (the kernels'
    time does not depend on their values); every expert is in the store."""
    import torch
    import bit_quantized_routed_gb300 as ds4
    rank, world, local = dist_env()
    R = wl.ring
    draws = [synth.draw_inputs(wl.replace(seed=wl.seed + i)) for i in range(R)]
    Ls = np.stack([d[0] for d in draws])
    xs = np.stack([d[1] for d in draws])
    gate, up, down = synth.random_expert_blobs(wl)
    shared = synth.shared_weights(wl.seed, wl.D, wl.F) if wl.shared else None
    W = ds4.ds4moe_weights_create(gate, up, down, wl.D, wl.F, shared=shared, max_tokens=wl.T, max_k=wl.k,
                                  n_slots=wl.slots)
    del gate, up, down
    xd = torch.from_numpy(xs.view(np.int16)).cuda().view(torch.bfloat16)
    Ld = torch.from_numpy(Ls).cuda()
    out = torch.zeros((wl.T, wl.D), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    fw = torch.empty(256 * 2 ** 20, dtype=torch.uint8, device="cuda")
    fr = torch.ones(64 * 2 ** 20, dtype=torch.float32, device="cuda")

    def l2_flush():
        fw.zero_()
        fr.sum()

    def step(i):
        ds4.ds4moe_expert_ffn(xd[i % R], W, Ld[i % R], wl.k, out)

    if args.calls:  # a fixed launch sequence for profilers: calls over the ring, then exit
        for i in range(args.calls):
            l2_flush()
            step(i)
        torch.cuda.synchronize()
        st = ds4.ds4moe_last_status(W)
        W.close()
        if st:
            raise RuntimeError(ds4.ds4moe_strerror(st))
        return
    for i in range(R):  # one pass over the ring fills the pool
        l2_flush()
        step(i)
    st = ds4.ds4moe_last_status(W)
    if st:
        raise RuntimeError(ds4.ds4moe_strerror(st))
    before = ds4.ds4moe_get_stats(W)["launches"]
    step(0)
    launches_per_call = ds4.ds4moe_get_stats(W)["launches"] - before
    graphs = [capture(lambda i=i: step(i)) for i in range(R)]
    pos = 1
    for _ in range(max(3, args.warmup)):
        l2_flush()
        graphs[pos % R].replay()
        pos += 1

    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    _, h0, m0, _ = ds4.ds4moe_pool_info(W)
    with ClockSampler(local) as clocks:
        torch.cuda.synchronize()
        barrier(world)
        for i in range(K):
            l2_flush()
            ev[i][0].record(stream)
            graphs[(pos + i) % R].replay()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        barrier(world)
    pos += K
    _, h1, m1, _ = ds4.ds4moe_pool_info(W)
    dev_ms = sum(a.elapsed_time(b) for a, b in ev)
    max_ms = reduce_max(dev_ms, world, "cuda")
    value = whole_job_rate(K * wl.T, world, max_ms / 1e3)
    expert_bytes = IQ2_PER_EXPERT(wl.D, wl.F) + Q2K_PER_EXPERT(wl.D, wl.F)
    misses_per_step = (m1 - m0) / K
    hit_rate = (h1 - h0) / max(1, (h1 - h0) + (m1 - m0))

    # per-stage device times (the pool stage: slot assignment + the copies of the missing experts)
    ds4.ds4moe_set_option(W, ds4.DS4MOE_OPT_PROFILE, 1)
    stage_tot = {n: 0.0 for n in ds4.STAGES}
    _, _, mp0, _ = ds4.ds4moe_pool_info(W)
    for i in range(K):
        l2_flush()
        torch.cuda._sleep(400000)
        step(pos + i)
        for n, v in ds4.ds4moe_get_stats(W)["stage_ms"].items():
            stage_tot[n] += v
    _, _, mp1, _ = ds4.ds4moe_pool_info(W)
    pos += K
    ds4.ds4moe_set_option(W, ds4.DS4MOE_OPT_PROFILE, 0)
    pool_ms = stage_tot["pool"] / K
    fill_bytes = (mp1 - mp0) / K * expert_bytes

    # host-to-device bandwidth of the copy engine on this machine: the fill kernel's reference
    src = torch.empty(256 * 2 ** 20, dtype=torch.uint8).pin_memory()
    dst = torch.empty(256 * 2 ** 20, dtype=torch.uint8, device="cuda")
    dst.copy_(src, non_blocking=True)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(4):
        dst.copy_(src, non_blocking=True)
    b.record(stream)
    torch.cuda.synchronize()
    h2d_gbs = 4 * src.numel() / (a.elapsed_time(b) / 1e3) / 1e9
    del src, dst

    # end to end through the public API: each step's token copied in, the result copied out
    xh = torch.from_numpy(xs.view(np.int16)).view(torch.bfloat16).pin_memory()
    Lh = torch.from_numpy(Ls).pin_memory()
    x1 = torch.empty((wl.T, wl.D), dtype=torch.bfloat16, device="cuda")
    L1 = torch.empty((wl.T, wl.E), dtype=torch.float32, device="cuda")
    out_h = torch.empty((wl.T, wl.D), dtype=torch.float32).pin_memory()
    e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    torch.cuda.synchronize()
    for i in range(K):
        l2_flush()
        e2e_ev[i][0].record(stream)
        x1.copy_(xh[(pos + i) % R], non_blocking=True)
        L1.copy_(Lh[(pos + i) % R], non_blocking=True)
        ds4.ds4moe_expert_ffn(x1, W, L1, wl.k, out)
        out_h.copy_(out, non_blocking=True)
        e2e_ev[i][1].record(stream)
    torch.cuda.synchronize()
    e2e_ms = reduce_max(sum(a.elapsed_time(b) for a, b in e2e_ev), world, "cuda")
    st = ds4.ds4moe_last_status(W)
    if st:
        raise RuntimeError(ds4.ds4moe_strerror(st))
    achieved = fill_bytes / (pool_ms / 1e3) / 1e9 if pool_ms > 0 else None
    roof = {"bound": "c2c", "kernel": "pool_fill_kernel (+ pool_assign_kernel)", "achieved": achieved,
            "peak": h2d_gbs, "unit": "GB/s", "frac": achieved / h2d_gbs if achieved else None,
            "traffic": ncu_traffic("pool", wl.name),
            "algorithmic_bytes": fill_bytes, "avg_launch_ms": pool_ms,
            "peak_source": "measured in this run: copy-engine host-to-device rate of 256 MB of pinned memory",
            "stage_ms": {n: round(v / K, 5) for n, v in stage_tot.items() if v > 0}}
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
            "warmup": max(3, args.warmup), "ms_per_step": max_ms / K, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": wl.name, "tokens": wl.T, "d_model": wl.D, "d_ff": wl.F, "experts": wl.E,
                       "top_k": wl.k, "shared_expert": "bf16" if wl.shared else None,
                       "routed_weights": "2-bit IQ2-style gate/up + Q2_K-style down, random valid blocks",
                       "device_slots": wl.slots, "store": "pinned host memory, read by the GPU",
                       "token_ring": R, "hit_rate": hit_rate, "misses_per_step": misses_per_step,
                       "copied_bytes_per_step": misses_per_step * expert_bytes,
                       "l2": "flushed between steps (write then read 256 MB)",
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "gpu_launches": int(launches_per_call * K),
            "e2e": {"value": whole_job_rate(K * wl.T, world, e2e_ms / 1e3), "unit": "tokens/s",
                    "h2d_bytes_per_step": wl.T * wl.D * 2 + wl.T * wl.E * 4, "d2h_bytes_per_step": wl.T * wl.D * 4},
            "roofline": roof, "clocks": clocks.summary()}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload, args.cpu_seconds)
    W.close()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ the oracle on the host

def cpu_baseline(workload, seconds):
    """Runs the oracle in a fresh single-threaded process (spawned, not forked)."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    out = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-worker", "--workload", workload,
                          "--cpu-seconds", str(seconds)], capture_output=True, text=True, env=env, timeout=900)
    if out.returncode:
        return {"value": None, "error": out.stderr.strip().splitlines()[-1:] or ["failed"]}
    return json.loads(out.stdout.strip().splitlines()[-1])


def cpu_worker(workload, seconds):
    import oracle
    oracle.build()
    wl = synth.WORKLOADS[workload]
    L, x = synth.draw_inputs(wl)
    # the oracle's FFN cost does not depend on block contents: random valid blocks stand in
    # for the quantised experts so that the baseline does not time quantisation
    per = max(1, min(wl.T, 4))
    n_tok, calls, el = 0, 0, 0.0
    rng = np.random.default_rng(0)
    sh = synth.shared_weights(wl.seed, wl.D, wl.F) if wl.shared else None
    while el < seconds:
        toks = np.sort(rng.choice(wl.T, per, replace=False)) if wl.T > per else np.arange(wl.T)
        idx, _ = oracle.route(L[toks], wl.k)
        blobs = synth.random_q4_expert_blobs if wl.fmt == "q4" else synth.random_expert_blobs
        gate, up, down = blobs(wl, np.unique(idx))
        t1 = time.perf_counter()
        oracle.moe_ffn(x[toks], L[toks], wl.k, gate, up, down, wl.D, wl.F, shared=sh, fmt=wl.fmt, threads=1)
        el += time.perf_counter() - t1
        n_tok += len(toks)
        calls += 1
    print(json.dumps({"value": n_tok / el, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                      "sample": "%d oracle call(s) of %d token(s) each from %s, %.1f s of oracle time "
                                "(fp64, one thread; random valid 2-bit blocks; input generation excluded)"
                                % (calls, per, workload, el)}))


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    wl = synth.WORKLOADS[args.workload]
    cb = cpu_baseline(args.workload, max(5.0, min(60.0, args.cpu_seconds)))
    v = cb.get("value")
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": (1e3 * wl.T / v) if v else None,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": reference_config(args, world),
            "cpu_baseline": cb, "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                                        "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.cpu_worker:
        cpu_worker(args.workload, args.cpu_seconds)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
