"""bench.py's multi-rank plumbing on CPU (gloo, world size 2): the timing is
the maximum over ranks, barriers pass, and the reference arm runs on rank 0
only.  (bench.py --gpus N runs N independent replicas of the decode pass; the
path has no collective of its own.)"""
import importlib.util
import os
import socket

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _load_bench():
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _worker(rank, ws, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    bench = _load_bench()
    ws_, rank_, _ = bench.dist_setup()
    bench.dist_barrier(ws_)
    m = bench.dist_max(1.5 + rank_, ws_)
    bench.dist_barrier(ws_)
    dist.destroy_process_group()
    out.put((rank_, ws_, m))


def test_two_gloo_ranks_take_the_max_time():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == [(0, 2, 2.5), (1, 2, 2.5)]


def test_reference_arm_runs_on_rank_zero_only(capsys):
    bench = _load_bench()

    class A:
        steps, warmup, layers, gpus, cpu_seconds = 2, 1, 1, 2, 0.05
    assert bench.run_reference(A, 2, 1) == 0
    assert capsys.readouterr().out == ""


def test_reference_arm_line(capsys):
    import json
    bench = _load_bench()

    class A:
        steps, warmup, layers, gpus, cpu_seconds = 2, 1, 1, 1, 0.05
    assert bench.run_reference(A, 1, 0) == 0
    line = json.loads(capsys.readouterr().out.strip())
    assert line["impl"] == "reference" and line["steps"] == 2 and line["warmup"] == 1
    assert line["cpu_baseline"]["kind"] == "oracle" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0
