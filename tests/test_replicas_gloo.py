"""The multi-rank path of bench.py on the CPU: two gloo ranks as separate processes.

The layer forward does not shard; N GPUs run N independent replicas with no collective on the
data path. The only cross-rank steps are the barriers around the timed region and the max over
ranks of the elapsed time. Whole-job throughput is the tokens of all ranks divided by that max.
The reference arm runs on rank 0 only, and the other ranks exit without work.
"""
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    ws, r, _ = bench.init_dist("gloo")
    assert (ws, r) == (world, rank)
    bench.barrier(None)
    # each rank "measured" a different time; every rank must see the slowest one
    slowest = bench.max_over_ranks(0.5 + rank, torch.device("cpu"))
    value = bench.weak_scaling_value(tokens_per_rank_step=2048, steps=10, n_ranks=ws, max_seconds=slowest)
    # the reference arm: rank 0 alone would run the oracle; the others return 0 at once
    ref_rc = None
    if rank != 0:
        ref_rc = bench.run_reference(type("A", (), {"steps": 1, "warmup": 3, "reference_budget_s": 1.0})(),
                                     bench.W.TINY_FP32)
    bench.barrier(None)
    torch.distributed.destroy_process_group()
    out.put((rank, slowest, value, ref_rc))


def test_two_gloo_ranks_take_the_max_time_and_sum_the_tokens():
    world = 2
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    results = sorted(out.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, value, ref_rc in results:
        assert slowest == pytest.approx(1.5)
        assert value == pytest.approx(2048 * 10 * world / 1.5)
        if rank != 0:
            assert ref_rc == 0
