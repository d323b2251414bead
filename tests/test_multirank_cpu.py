"""The benchmark's multi-GPU host logic on CPU: two gloo ranks (no GPU), as
torchrun would launch them. Each rank owns an independent workload, so the
only cross-rank traffic is the barrier and the max/sum of the step timings;
the reference arm runs on rank 0 only."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench

    dist = bench.init_dist(world)
    bench.barrier(dist)
    mx = bench.reduce_over_ranks(dist, 1.5 + rank, "max")
    sm = bench.reduce_over_ranks(dist, 10.0 * (rank + 1), "sum")
    import contextlib
    import io
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        rc = bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3"]) if rank == 1 else 0
    dist.destroy_process_group()
    q.put((rank, mx, sm, rc, buf.getvalue()))


@pytest.mark.parametrize("world", [2])
def test_two_gloo_ranks(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, mx, sm, rc, text in out:
        assert mx == 1.5 + (world - 1)
        assert sm == sum(10.0 * (r + 1) for r in range(world))
        assert rc == 0
    assert out[1][4] == ""  # the reference arm prints nothing off rank 0
