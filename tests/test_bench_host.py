"""Host-side pieces of bench.py: the reference (oracle) arm's JSON line, and the
multi-process plumbing (max over ranks, rank-0-only output) on gloo, world size 2."""
import json
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_reference_arm_prints_contract_line(capsys):
    rc = bench.main(["--impl", "reference", "--workload", "tiny_f32", "--steps", "2", "--warmup", "3"])
    assert rc == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert k in line, k
    assert line["impl"] == "reference"
    assert line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["config"]["workload"] == "tiny_f32"


def test_warmup_is_at_least_three(capsys):
    bench.main(["--impl", "reference", "--workload", "tiny_f32", "--steps", "1", "--warmup", "1"])
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["warmup"] == 3


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    bench.init_dist(world, "gloo")
    m = bench.reduce_max(float(rank + 1) * 1.5, world)
    bench.barrier(world)
    q.put((rank, m))
    dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == {0: 3.0, 1: 3.0}


def _ref_worker(rank, world, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import io
    import contextlib
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        rc = bench.main(["--impl", "reference", "--workload", "tiny_f32", "--steps", "1", "--warmup", "3"])
    q.put((rank, rc, buf.getvalue()))


def test_reference_arm_only_rank0_prints():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_ref_worker, args=(r, 2, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = {r: (rc, s) for r, rc, s in (q.get(timeout=120) for _ in range(2))}
    for p in procs:
        p.join(timeout=60)
    assert out[0][0] == 0 and out[1][0] == 0
    assert json.loads(out[0][1].strip())["impl"] == "reference"
    assert out[1][1].strip() == ""
