"""The multi-process side of bench.py on CPU: two gloo ranks launched the way torchrun
sets them up (RANK, WORLD_SIZE, LOCAL_RANK, MASTER_ADDR=127.0.0.1, MASTER_PORT). The
replicas exchange no data; the bench only needs the process group, a barrier around the
timed region and the max over ranks of the timings, which these tests pin."""
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, q):
    # CPU ranks even on a GPU machine: the bench then picks gloo
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(ws), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
    sys.path.insert(0, ROOT)
    try:
        import torch.distributed as dist

        import bench
        got_ws, got_rank, got_local = bench.dist_init()
        # per-rank timings: rank r is slower in the first entry, faster in the second
        vals = bench.reduce_max([1.0 + rank, 10.0 - rank, 0.5], got_ws)
        bench.barrier(got_ws)
        q.put((rank, got_ws, got_rank, got_local, dist.get_backend(), vals))
        dist.destroy_process_group()
    except Exception as e:  # reported to the parent, which fails the test
        q.put((rank, "error", repr(e)))


@pytest.mark.timeout(120)
def test_two_gloo_ranks_take_the_max_over_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=100) for _ in range(2)]
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    by_rank = {r[0]: r for r in res}
    assert set(by_rank) == {0, 1}
    for r in (0, 1):
        rank, ws, got_rank, local, backend, vals = by_rank[r]
        assert (ws, got_rank, local, backend) == (2, r, r, "gloo")
        assert vals == [2.0, 10.0, 0.5]


def test_single_process_needs_no_process_group(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    sys.path.insert(0, ROOT)
    import bench
    assert bench.dist_init() == (1, 0, 0)
    assert bench.reduce_max([3.0, 4.0], 1) == [3.0, 4.0]
    bench.barrier(1)  # a no-op for one process
