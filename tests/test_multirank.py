"""The multi-rank path of the benchmark on two gloo ranks (CPU, no GPU).

Sequences are independent, so N ranks each verify their own batch (weak
scaling) with no collective on the data path; the only exchange is the
max-over-ranks reduction of the step time.  These tests run that host logic
on world_size 2: per-rank shards are distinct and each is a pure function of
its rank, the reduction returns the slowest rank's time on every rank, the
aggregate counts every rank's units, and the reference arm prints on rank 0
only.
"""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

from tests.conftest import ROOT  # noqa: E402

sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import oracle
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        slowest = bench.reduce_max(1.5 + rank, world)
        case = bench.make_workload(1, rank)
        toks, n, _ = oracle.verify(case.target, case.draft, case.tokens, case.u_accept,
                                   case.u_resample, case.temperature)
        shards = [None] * world
        dist.all_gather_object(shards, (case.target[0, 0, :8].tolist(), n.tolist(),
                                        toks.tolist()))

        class A:
            config, batch, steps, warmup = 1, None, 1, 0
        buf = io.StringIO()
        with redirect_stdout(buf):
            bench.run_reference(A)
        q.put((rank, slowest, shards, buf.getvalue()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = dict()
    for _ in procs:
        r, slowest, shards, printed = q.get(timeout=300)
        out[r] = (slowest, shards, printed)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # the reduction gives every rank the slowest rank's time
    assert out[0][0] == out[1][0] == 2.5
    # the shards differ, and each equals what one process computes for that rank
    (t0, n0, k0), (t1, n1, k1) = out[0][1]
    assert t0 != t1
    import oracle
    for rank, (_, n, toks) in enumerate(out[0][1]):
        case = bench.make_workload(1, rank)
        rt, rn, _ = oracle.verify(case.target, case.draft, case.tokens, case.u_accept,
                                  case.u_resample, case.temperature)
        assert rn.tolist() == n and rt.tolist() == toks
    # the reference arm prints one line on rank 0 and nothing on rank 1
    assert out[0][2].count("\n") == 1 and '"impl": "reference"' in out[0][2]
    assert out[1][2] == ""


def test_aggregate_rate_counts_every_rank():
    assert bench.aggregate_rate(2048, 10, 4, 2.0) == 4 * 2048 * 10 / 2.0
    assert bench.reduce_max(3.25, 1) == 3.25
