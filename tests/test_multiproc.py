"""The bench's multi-process path on the CPU: two gloo ranks on 127.0.0.1 check
the barrier, the max-over-ranks timing reduction, and that only rank 0 runs
the reference arm (every GPU runs an independent replica: no data-path
collective exists to test)."""
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


def _worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), BEP_DIST_BACKEND="gloo")
    sys.path.insert(0, ROOT)
    import bench
    r, w, local = bench.dist_init()
    bench.dist_barrier(w)
    mx = bench.dist_max(w, float(10 * (r + 1)))

    class Args:
        steps, warmup = 1, 0

    ref = bench.run_reference(Args, r, w) if r == 1 else "skipped"
    bench.dist_barrier(w)
    import torch.distributed as dist
    dist.destroy_process_group()
    q.put((r, w, local, mx, ref))


def test_two_gloo_ranks_barrier_and_max():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[0] for o in out] == [0, 1]
    assert all(o[1] == 2 for o in out)
    assert [o[2] for o in out] == [0, 1]
    assert all(o[3] == 20.0 for o in out)       # max over ranks of 10, 20
    assert out[1][4] is None                    # rank 1 does no reference work
