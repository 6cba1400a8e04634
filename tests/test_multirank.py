"""The benchmark's multi-rank host logic on two gloo ranks (CPU only).

Each rank runs its own batch of independent sequences (weak scaling, no
collective on the data path); the only communication is the barrier around
the timed region and the max over ranks of the step time. This checks those
pieces and the whole-job throughput formula without a GPU.
"""
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    torch.cuda.is_available = lambda: False  # force the gloo backend on any host
    import bench
    import torch.distributed as dist
    r, w, local = bench.dist_setup(world)
    step_ms = [3.0, 5.0][r]
    m = bench.max_over_ranks(step_ms, w, "cpu")
    bench.barrier(w)
    out.put((r, w, local, m, bench.rank_seed(2, r), bench.job_value(65536, m, w)))
    dist.destroy_process_group()


def test_two_rank_weak_scaling_logic():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [x[0] for x in res] == [0, 1] and all(x[1] == 2 for x in res)
    assert [x[2] for x in res] == [0, 1]                 # one GPU per local rank
    assert all(x[3] == 5.0 for x in res)                 # max over ranks
    assert res[0][4] != res[1][4]                        # distinct seeded batches
    assert res[0][5] == pytest.approx(2 * 65536 / 5e-3)  # all ranks' tokens / slowest step


def test_reference_arm_runs_on_rank_zero_only(capsys, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    args = type("A", (), {"gpus": 2, "steps": 1, "warmup": 3})()
    bench.run_reference(args)
    assert capsys.readouterr().out == ""
