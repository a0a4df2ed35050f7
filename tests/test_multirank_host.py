"""The benchmark's multi-rank plumbing on CPU: two ranks over gloo (no GPU). The path shards by
tokens with no exchange step, so N GPUs run N independent replicas; what must hold is the rank
bookkeeping, the max-over-ranks timing, the whole-job rate, per-rank inputs, and that only rank 0
of the reference arm does any work."""
import contextlib
import io
import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    import synth
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        m = bench.reduce_max(float(10 * (rank + 1)), w)   # rank r reports 10 (r + 1) "ms"
        bench.barrier(w)
        wl = synth.WORKLOADS["tiny_t4"]
        mine = synth.draw_inputs(wl.replace(seed=wl.seed + 1000 * r))[0]
        # the reference arm: every rank but 0 returns at once and prints nothing
        buf = io.StringIO()
        if r != 0:
            with contextlib.redirect_stdout(buf):
                bench.run_reference(bench.parse_args(["--impl", "reference", "--workload", "tiny_t4"]))
        out.put((rank, r, w, local, m, bench.whole_job_rate(4, w, m / 1e3), mine.tolist(), buf.getvalue()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_replica_bookkeeping():
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, r, w, local, m, rate, _, printed in res:
        assert (r, w, local) == (rank, 2, rank)
        assert m == 20.0                               # the slowest rank's time, on every rank
        assert rate == pytest.approx(4 * 2 / 0.020)    # all ranks' tokens over the slowest time
    assert res[1][7] == ""                              # rank 1 of the reference arm printed nothing
    assert not np.array_equal(np.array(res[0][6]), np.array(res[1][6]))  # each replica its own batch


def test_single_rank_defaults():
    sys.path.insert(0, ROOT)
    import bench
    env = {k: os.environ.pop(k) for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK") if k in os.environ}
    try:
        assert bench.dist_env() == (0, 1, 0)
        assert bench.reduce_max(3.5, 1) == 3.5
        bench.barrier(1)   # no process group needed
    finally:
        os.environ.update(env)
