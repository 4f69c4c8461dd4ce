"""The multi-GPU mode of bench.py runs independent replicas (the path shards
by output rows with no exchange step): ranks meet at a barrier around the
timed region and the job's time is the slowest rank's.  These checks run the
host side of that with two gloo ranks on the CPU."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
mp = pytest.importorskip("torch.multiprocessing")


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, ws: int, port: int, out) -> None:
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=ws)
    bench._barrier(ws)
    ms = bench._max_over_ranks(10.0 + rank, ws)          # rank 1 is the slower one
    out[rank] = (ms, bench._job_value(ws, 1, 100, ms))
    bench._barrier(ws)
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    port = _free_port()
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    assert res[0] == res[1]                                 # every rank reports the same job time
    ms, value = res[0]
    assert ms == 11.0
    assert value == pytest.approx(2 * 1 * 100 / 0.011)       # both replicas' tokens over the slowest time


def test_single_rank_is_unchanged():
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    assert bench._max_over_ranks(3.5, 1) == 3.5
    assert bench._job_value(1, 4, 10, 20.0) == pytest.approx(4 * 10 / 0.02)


def test_reference_arm_does_no_work_off_rank_0(capsys):
    import sys
    import types
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    args = types.SimpleNamespace(ntok=1, steps=1, warmup=0, gpus=2)
    assert bench.run_reference(args, 2, 1) is None
    assert capsys.readouterr().out == ""
