"""The N > 1 path of bench.py on CPU: two gloo ranks (one per would-be GPU).
BitLinear shards by replicas with no data-path exchange; across ranks only the
timing is combined (the slowest replica sets the step time, the value is the
aggregate), and the reference arm runs on rank 0 alone."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      LOCAL_RANK=str(rank), WORLD_SIZE=str(world))
    import sys
    sys.path.insert(0, ROOT)
    import bench
    r, lr, w = bench.dist_env()
    dist.init_process_group("gloo", rank=r, world_size=w)
    try:
        step_ms = 1.0 + 0.5 * r                      # rank 1 is the slower replica
        ms = bench.max_over_ranks(step_ms, dist, "cpu")
        value = bench.aggregate_gbs(w, 10 ** 9, ms)
        # rank != 0 leaves the reference arm without doing any work
        ref = bench.reference_arm(type("A", (), {"steps": 1, "warmup": 0, "ref_seconds": 0.1})()) if r != 0 else None
        out[r] = (r, lr, w, ms, value, ref)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_combine_timing():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert sorted(res) == [0, 1]
    for r in (0, 1):
        rank, local_rank, w, ms, value, ref = res[r]
        assert (rank, local_rank, w) == (r, r, 2)
        assert ms == 1.5                               # max over ranks
        assert value == pytest.approx(2 * 1e9 / 1.5e-3 / 1e9)
    assert res[1][5] == 0                             # reference arm: rank 1 exits at once


def test_single_process_helpers():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.5, None, "cpu") == 2.5
    assert bench.aggregate_gbs(1, 520 * 10 ** 6, 2.0) == pytest.approx(260.0)
