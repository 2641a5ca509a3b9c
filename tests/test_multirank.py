"""Multi-rank host logic of bench.py on CPU: gloo, world size 2 (no GPU).

Each rank runs its own replica of the workload; the only cross-rank steps are a
barrier around the timed region and the max over ranks of the elapsed time.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench
    import torch.distributed as dist
    w, r, local = bench.dist_init()
    assert (w, r) == (world, rank) and dist.get_backend() == "gloo"
    bench.barrier(w)
    m = bench.max_over_ranks(w, 1.0 + rank * 2.5)

    class Args:  # the reference arm: only rank 0 works, the others return at once
        layers, tokens, steps, warmup, gpus = 1, 2, 1, 0, world

    rc = bench.run_reference(Args(), w, r) if r != 0 else 0
    out.put((rank, m, rc))
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_barrier_and_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(90)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    assert [m for _, m, _ in res] == [3.5, 3.5]
    assert [rc for _, _, rc in res] == [0, 0]
