"""The benchmark's multi-rank plumbing on CPU (gloo, world_size 2): every rank runs an
independent replica of the workload - sequences never exchange data - so the only
collectives are the timing barrier and the max over ranks of the elapsed time; the
reference (CPU oracle) leg runs on rank 0 only."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        m = bench.max_over_ranks(float(10 + rank * 5), world)

        class A:  # the reference leg's arguments
            workload, steps, warmup, gpus = "tiny", 1, 0, world
        import io
        import contextlib
        buf = io.StringIO()
        with contextlib.redirect_stdout(buf):
            bench.run_reference(A, rank, world)
        out[rank] = (m, buf.getvalue())
    finally:
        dist.destroy_process_group()


def test_two_ranks_max_timing_and_rank0_only_reference():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out[0][0] == 15.0 and out[1][0] == 15.0
    assert '"impl": "reference"' in out[0][1]
    assert out[1][1] == ""
