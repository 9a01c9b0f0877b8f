"""The multi-process path of bench.py on CPU (gloo, world size 2): the
barrier, the max-over-ranks step time and the all-rank work sum that
`value` divides, and the reference arm's rank-0-only rule."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    bench.barrier(ws)
    step_ms = 10.0 + 5.0 * rank          # rank 1 is the slow one
    work = 100.0 * (rank + 1)
    mx = bench.max_over_ranks(step_ms, ws)
    tot = bench.sum_over_ranks(work, ws)
    out[rank] = (mx, tot, bench.dist_env())
    dist.destroy_process_group()


def test_gloo_world_size_two():
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    for rank in (0, 1):
        mx, tot, env = res[rank]
        assert mx == 15.0 and tot == 300.0
        assert env == (2, rank, rank)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        workload = "tiny"
        steps = 1
        warmup = 0
        cpu_seconds = 1.0

    # a rank other than 0 returns before any work (no output, no workload)
    assert bench.run_reference(Args()) is None
