"""The multi-rank plumbing of bench.py on CPU: two gloo ranks (world size 2)
go through the same helpers the benchmark uses under torchrun -- process
group set-up from the environment, the barrier, the max over ranks of a
step time (the reported time is the slowest rank's) and the sum over ranks
of a throughput -- and the reference arm leaves every rank but 0 idle.

The decode path itself has no exchange between GPUs (streams are
independent), so these helpers are the whole multi-GPU logic."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    r, w, local = bench.init_dist(world)
    assert (r, w, local) == (rank, world, rank)
    bench.barrier()
    step_ms = 1.0 + rank                      # rank 1 is the slow one
    slowest = bench.max_over_ranks(step_ms)
    total = bench.sum_over_ranks(100.0 * (rank + 1))
    bench.barrier()
    results[rank] = (slowest, total)
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_max_and_sum():
    port = _free_port()
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_rank_main, args=(2, port, results), nprocs=2, join=True)
        got = dict(results)
    assert got[0] == got[1] == (2.0, 300.0)


def test_single_process_helpers_are_identities():
    import bench
    assert not bench._DIST["on"]
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.sum_over_ranks(7.0) == 7.0
    bench.barrier()  # no process group: returns at once


def _ref_rank_main(rank: int, world: int, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world))
    import bench

    class Args:
        workload = "toy_k4v2_t1k"
        steps = 1
        warmup = 0

    called = []
    bench.oracle_sample = lambda *a, **k: called.append(1) or {"value": 1.0, "unit": "us/step", "cores": 1,
                                                                 "kind": "oracle", "sample": "stub",
                                                                 "streams": 3, "seconds": 0.1}
    bench.run_reference(Args())
    out[rank] = len(called)


@pytest.mark.parametrize("world", [2])
def test_reference_arm_runs_on_rank0_only(world):
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_ref_rank_main, args=(world, out), nprocs=world, join=True)
        got = dict(out)
    assert got[0] >= 1 and all(got[r] == 0 for r in range(1, world))


def test_all_cores_oracle_timing_runs_workers():
    """The all-cores CPU baseline: spawned oracle workers, one stream each;
    the reported step time is positive and names the process count."""
    import bench
    r = bench.oracle_sample_all_cores("toy_k4v2_t1k", 0.2, procs=2)
    assert r is not None and "unavailable" not in r, r
    assert r["cores"] == 2 and r["kind"] == "oracle" and r["value"] > 0
