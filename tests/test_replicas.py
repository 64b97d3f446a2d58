"""The multi-rank path of bench.py on CPU: two gloo ranks, each an
independent replica with its own step time, agree on the slowest step and
report the bytes of both ranks over it (no data-path collective; the one
all-reduce is the timing's max over ranks)."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    torch.distributed.init_process_group("gloo")
    try:
        assert bench.dist_env() == (ws, rank, rank)
        step, value = bench.replica_value(1e-3 * (rank + 1), 10 ** 9, ws, "cpu")
        q.put((rank, step, value))
    finally:
        torch.distributed.destroy_process_group()


def test_two_gloo_replicas_take_the_slowest_step():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, step, value in got:
        assert step == pytest.approx(2e-3)            # rank 1 is the slower one
        assert value == pytest.approx(2 * 1.0 / 2e-3)  # 2 ranks x 1 GB per 2 ms
