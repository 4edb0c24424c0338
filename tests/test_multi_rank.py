"""The N > 1 bench path on CPU: two gloo ranks (127.0.0.1) run the timing reduction and
the whole-job aggregate that bench.py uses under torchrun; each rank verifies its own
replica of the workload (sequences are independent: replicas only, no data collective)."""
import os
import socket
import sys

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
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import workloads
    dist.barrier()
    elapsed = 10.0 + 3.0 * rank  # the ranks' own timed intervals
    job_ms = bench.max_over_ranks(elapsed, dist, "cpu")
    steps, units = 5, 2048.0
    value = bench.job_value(units, world, job_ms / steps)
    x = workloads.chain_workload("chain_b1_v1000", bench.replica_round(rank, 0), "cpu")
    dist.barrier()
    out.put((rank, job_ms, value, float(x["logits"].sum())))
    dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_gloo_ranks_take_the_slowest_interval_and_aggregate():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=240) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    want_ms = 10.0 + 3.0 * (world - 1)
    for rank, job_ms, value, _ in res:
        assert job_ms == want_ms
        assert value == pytest.approx(2048.0 * world / (want_ms / 5 / 1e3))
    assert res[0][3] != res[1][3]  # each replica verifies its own data


def test_single_process_reduction_is_the_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(12.5) == 12.5
    assert bench.job_value(100.0, 1, 2.0) == pytest.approx(50000.0)
