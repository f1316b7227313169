"""The N > 1 path of bench.py without GPUs: two gloo ranks on the CPU run the
same barrier / max-over-ranks / sum-over-ranks helpers the GPU replicas use,
so `value` = bytes of all ranks / the slowest rank's time."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench

    r, lr, w = bench.dist_env()
    assert (r, lr, w) == (rank, rank, world)
    bench.init_dist(w, "gloo")
    bench.barrier(w)
    elapsed_ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
    step_bytes = 1000.0 * (rank + 1)
    mx = bench.allreduce_max(elapsed_ms, w)
    tot = bench.allreduce_sum(step_bytes, w)
    out[rank] = (mx, tot)
    import torch.distributed as dist

    dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_like_bench():
    world, port = 2, _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == out[1] == (15.0, 3000.0)


def test_single_rank_helpers_are_identity():
    import bench

    assert bench.allreduce_max(3.5, 1) == 3.5 and bench.allreduce_sum(2.0, 1) == 2.0
    bench.barrier(1)


@pytest.mark.parametrize("argv", [[], ["--gpus", "2", "--steps", "7", "--warmup", "3"]])
def test_bench_arguments(argv):
    import bench

    a = bench.parse_args(argv)
    assert a.warmup >= 3 and a.steps >= 1 and a.impl == "ours"
