"""The multi-rank path of the benchmark, on CPU with the gloo backend and two
ranks: the layer runs as independent replicas (no data-path exchange), the
job's step time is the maximum over ranks and the throughput counts every
rank's tokens; the reference arm does its work on rank 0 only."""
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


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(1.5 + rank, "cpu")        # rank 1 is the slow one
        dist.barrier()
        ref_rc = None
        if rank != 0:
            # the reference arm: ranks other than 0 exit at once without work
            ref_rc = bench.run_reference(bench.parse_args(["--impl", "reference"]), None)
        out.put((rank, ms, bench.job_tokens_per_s(world, 4096, ms), ref_rc))
    finally:
        dist.destroy_process_group()


def test_two_replicas_max_over_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(out.get(timeout=10) for _ in range(world))
    for rank, ms, tps, ref_rc in res:
        assert ms == 2.5                                   # both ranks see the slowest time
        assert tps == pytest.approx(2 * 4096 / 2.5e-3)     # every rank's tokens count
        if rank == 1:
            assert ref_rc == 0


def test_single_process_is_a_no_op():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, "cpu") == 3.25
    assert bench.job_tokens_per_s(1, 4096, 2.0) == pytest.approx(2048000.0)
