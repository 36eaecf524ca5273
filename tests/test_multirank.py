"""The benchmark's multi-rank plumbing on CPU (gloo, world size 2).

Each rank runs its own replica; the only cross-rank steps are the barrier
around the timed region and the max over ranks of the step time.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench

    r, w, local = bench.dist_setup()
    assert (r, w, local) == (rank, world, rank)
    bench.barrier(w)
    got = bench.max_over_ranks(1.5 + rank, w)
    import torch.distributed as dist

    dist.destroy_process_group()
    q.put((rank, got))


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    results = dict(q.get(timeout=5) for _ in range(2))
    assert results == {0: 2.5, 1: 2.5}


def test_single_rank_defaults(monkeypatch):
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    sys.path.insert(0, ROOT)
    import bench

    assert bench.dist_setup() == (0, 1, 0)
    assert bench.max_over_ranks(3.0, 1) == 3.0


def test_flop_count():
    sys.path.insert(0, ROOT)
    import bench
    from attention_backward_tcgen05_gb300 import inputs

    w = inputs.WORKLOADS["gqa_causal_d128"]
    assert bench.backward_flops(w) == pytest.approx(343.597e9, rel=1e-4)
    assert bench.backward_flops(inputs.WORKLOADS["long_seq"]) == pytest.approx(2748.8e9, rel=1e-4)
