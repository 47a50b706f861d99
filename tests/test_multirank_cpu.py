"""Multi-process (gloo, world size 2) checks of the benchmark's N > 1 logic:
every rank runs its own batches (replicas, no data-path collective) and the
whole-job figure is all ranks' tokens over the slowest rank's time."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        import bench
        assert bench.dist_env() == (ws, rank, rank)
        ms_local = 10.0 + 5.0 * rank          # rank 1 is the slower one
        tokens_local = 1000 * (rank + 1)
        ms, tokens, value = bench.aggregate(ms_local, tokens_local, ws)
        out[rank] = (ms, tokens, value)
    finally:
        dist.destroy_process_group()


def test_aggregate_two_ranks():
    ws = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(ws, port, out), nprocs=ws, join=True)
        res = dict(out)
    for r in range(ws):
        ms, tokens, value = res[r]
        assert ms == 15.0                     # max over ranks
        assert tokens == 3000.0               # sum over ranks
        assert value == pytest.approx(3000.0 / 0.015)


def test_aggregate_single_rank():
    import bench
    assert bench.aggregate(20.0, 500, 1) == (20.0, 500.0, 500.0 / 0.02)


def _ref_worker(rank, ws, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    import contextlib
    import io
    import bench

    class Args:
        steps, warmup, ref_budget_s = 1, 1, 0.5
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.main_reference(Args())
    out[rank] = buf.getvalue()


def test_reference_arm_prints_on_rank0_only():
    ws = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_ref_worker, args=(ws, _free_port(), out), nprocs=ws, join=True)
        res = dict(out)
    import json
    line = json.loads(res[0].strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert res[1] == ""
