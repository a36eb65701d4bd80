"""bench.py's multi-rank path on CPU: two gloo ranks (replicas only: the
only collectives are the timing barrier and the max over ranks)."""
import os
import socket

import pytest
import torch.multiprocessing as mp

pytestmark = pytest.mark.cpu


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, ws, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(ws),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    import bench
    import torch.distributed as dist
    got_ws, got_rank, _ = bench.dist_setup()
    try:
        bench.barrier(got_ws)
        span = 10.0 + 5.0 * got_rank          # ms: rank 1 is the slowest
        ms_max = bench.max_over_ranks(span, got_ws)
        value = bench.weak_scaling_value(1.0e9, got_ws, ms_max)
        out.put((got_rank, got_ws, ms_max, value, dist.get_backend()))
        bench.barrier(got_ws)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_time_and_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for rank, ws, ms_max, value, backend in res:
        assert ws == 2 and backend == "gloo"
        assert ms_max == 15.0                   # the slowest rank's span, on every rank
        assert value == pytest.approx(2 * 1.0e9 / 15.0e-3)   # all ranks' units over that span
    assert [r[0] for r in res] == [0, 1]


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.weak_scaling_value(2.0e9, 1, 4.0) == pytest.approx(5.0e11)
