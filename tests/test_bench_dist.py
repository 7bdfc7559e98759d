"""The multi-process side of bench.py on CPU: two gloo ranks, as torchrun
would start them on two GPUs.  Replicas only (no collective on the data
path): the ranks meet at barriers, agree on the slowest rank's time, and
report the whole job's tokens; each rank draws its own tokens; the reference
arm prints from rank 0 only."""
import contextlib
import io
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import bench
    from workloads import CONFIGS, make_tokens
    w, r, local = bench.dist_setup(world)
    assert (w, r, local) == (world, rank, rank) and dist.get_backend() == "gloo"
    bench.barrier(w)
    # every rank's elapsed time; all agree on the maximum
    my_ms = 10.0 + 5.0 * rank
    ms_max = bench.max_over_ranks(w, my_ms)
    value = bench.whole_job_tokens_per_s(w, 8, 100, ms_max)
    # each replica's first token batch, compared across ranks
    x = make_tokens(CONFIGS["tiny"], T=4, batch=bench.replica_batch(r, 0))
    t = torch.tensor([float(np.abs(x).sum())], dtype=torch.float64)
    got = [torch.zeros(1, dtype=torch.float64) for _ in range(w)]
    dist.all_gather(got, t)
    bench.barrier(w)
    dist.destroy_process_group()
    q.put((rank, ms_max, value, [float(g.item()) for g in got]))


def test_two_gloo_ranks_agree_on_time_and_whole_job_tokens():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    out.sort()
    for rank, ms_max, value, sums in out:
        assert ms_max == 15.0                          # the slowest rank's time, on every rank
        assert value == pytest.approx(2 * 8 * 100 / 0.015)  # all ranks' tokens / that time
        assert sums[0] != sums[1]                      # replicas draw different tokens


def test_reference_arm_prints_on_rank_zero_only():
    sys.path.insert(0, ROOT)
    import bench
    args = type("A", (), {"steps": 1, "warmup": 3})()
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(args, "dsv2lite-decode-T8", 1, with_prefill=True)
    assert buf.getvalue() == ""
