"""The N > 1 path of bench.py on CPU: two gloo ranks, each with its own batch
(weak scaling), take the max of their times and report all ranks' units over it."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, ws: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    import bench
    import synth
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        w, r, loc = bench.dist_env()
        assert (w, r, loc) == (ws, rank, rank)
        bench.barrier(ws)
        t_local = 0.010 * (rank + 1)  # rank 1 is the slowest
        t = bench.reduce_max(t_local, ws)
        value = bench.whole_job_value(ws, 36, t)
        wl = synth.WORKLOADS["tiny"]
        x = bench.rank_x(wl, 0, rank)
        out[rank] = (t, value, x.tobytes())
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_weak_scaling():
    ws = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank, args=(ws, port, out), nprocs=ws, join=True, start_method="spawn")
    assert out[0][0] == out[1][0] == pytest.approx(0.020)  # both ranks see the max
    assert out[0][1] == out[1][1] == pytest.approx(2 * 36 / 0.020)  # all ranks' units / slowest time
    assert out[0][2] != out[1][2]  # each rank has its own batch
