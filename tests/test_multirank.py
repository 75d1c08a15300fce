"""Host logic of the multi-GPU run (replicas only): two gloo ranks on CPU.

Each rank runs its own replica of the step; the job's time is the slowest
rank's, its rate the units of all ranks over that time, and only rank 0 runs
the reference arm.  No GPU is involved.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import sys
    import torch.distributed as dist
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = bench.max_over_ranks(1.5 + rank, "cpu")          # rank 1 is the slow one
    rate = bench.whole_job_rate(world, 4, ms)
    ws, r, _ = bench._dist()
    ref = bench.run_reference(None, None, None) if r != 0 else "rank0"
    out.put((rank, ms, rate, ws, ref))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_time_and_rate():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, rate, ws, ref in res:
        assert ws == 2
        assert ms == pytest.approx(2.5)                   # max over ranks, on every rank
        assert rate == pytest.approx(2 * 4 / 2.5e-3)      # whole-job units / slowest time
    assert res[0][4] == "rank0" and res[1][4] is None     # only rank 0 runs the reference arm


def test_single_process_is_its_own_max():
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.whole_job_rate(1, 4, 0.1) == pytest.approx(40000.0)
