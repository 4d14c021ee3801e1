"""The multi-rank host logic of bench.py (replicas: one process per GPU,
barrier, slowest rank's time, rank 0 reports) on CPU with two gloo ranks."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    slowest = bench.max_over_ranks(10.0 + 5.0 * rank)  # rank 1 is the slow one
    dist.barrier()
    # the reference arm: rank 0 alone runs and prints; the others exit 0 without work
    args = type("A", (), dict(config="single_linear", warmup=0, steps=1, gpus=world))()
    buf = io.StringIO()
    with redirect_stdout(buf):
        rc = bench.run_reference(args)
    out[rank] = (slowest, bench.job_ms_per_step(slowest, world), rc, buf.getvalue())
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_and_rank0_reports():
    world = 2
    with mp.Manager() as man:
        out = man.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world, start_method="spawn",
                           join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 15.0
    assert res[0][1] == res[1][1] == 7.5  # two replicas' steps in the slowest rank's time
    assert res[0][2] == res[1][2] == 0
    import json

    line = json.loads(res[0][3].strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert res[1][3] == ""


def test_single_process_without_group_is_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert not dist.is_initialized()
    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.job_ms_per_step(8.0, 1) == 8.0


def test_bench_tables_cover_every_profiled_kernel_kind():
    # the bench reads every kind of the library's launch profile: each needs a
    # kernel name for the roofline line and, if tensor-bound, its MMA count
    sys.path.insert(0, ROOT)
    import bench
    from infra_fac_factors_gb300 import capi

    assert set(bench.KERNEL_NAMES) == set(capi.KERNEL_KINDS)
    assert set(bench.ISSUED_PER_ALGORITHMIC) == set(capi.KERNEL_KINDS) - {"running"}
