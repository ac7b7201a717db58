"""The multi-GPU path of bench.py is replicas only: every rank runs the same
per-GPU workload on its own sequences, with no collective on the data path.
What crosses ranks is the measurement: a barrier around the timed region, the
maximum step time and the total query count. These run here as two gloo ranks
on the CPU (rendezvous on 127.0.0.1)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        r, w, loc = bench.dist_env()
        bench.barrier(w)
        # Each rank's step time and query count, as run_ours reports them.
        ms = 1.0 + rank          # rank 1 is the slowest
        q = 8.0 * (rank + 1)     # queries this rank processed per step
        ms_max = bench.max_over_ranks(ms, w)
        total_q = bench.sum_over_ranks(q, w)
        bench.barrier(w)
        out[rank] = (r, w, loc, ms_max, total_q, total_q / (ms_max * 1e-3))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_like_the_bench():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
        assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
        res = dict(out)
    for rank in range(2):
        r, w, loc, ms_max, total_q, value = res[rank]
        assert (r, w, loc) == (rank, 2, rank)
        assert ms_max == pytest.approx(2.0)       # the slowest rank sets the step time
        assert total_q == pytest.approx(24.0)     # queries of all ranks
        assert value == pytest.approx(24.0 / 2e-3)  # whole-job queries per second


def _reference_rank(rank, world, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    from synth.workloads import WORKLOADS

    class Args:
        steps, warmup = 1, 1

    # Ranks other than 0 do no work and print nothing in the reference arm.
    out[rank] = bench.run_reference(Args(), WORKLOADS[0], rank, world) if rank != 0 else "skipped"


def test_reference_arm_runs_on_rank_zero_only():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        p = ctx.Process(target=_reference_rank, args=(1, 2, out))
        p.start()
        p.join(120)
        assert p.exitcode == 0
        assert out[1] is None
