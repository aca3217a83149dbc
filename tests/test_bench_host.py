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


def test_oracle_sample_weight_gradients_sum_over_the_batch():
    """The bench's sampled-error reference: per sampled head, batch 0's out / lse
    / dq rows and the head's dW_UK / dW_UV columns summed over every batch
    element (the library's weight gradients are batch sums), checked against the
    oracle's full forward and backward on a B = 2 problem."""
    import numpy as np
    import oracle
    from mla_attention_sequence_gb300.configs import Problem
    from mla_attention_sequence_gb300.synth import make_inputs
    p = Problem(B=2, Sq=6, S=11, n_h=3, d_c=8, d_nope=4, d_rope=2, d_v=5, q_offset=5, dtype="f32")
    x = {k: v.astype(np.float64) for k, v in make_inputs(p, seed=3).items()}
    keep = {}
    flops = bench.oracle_sample(p, x, [0, 2], keep)
    assert flops == p.with_(n_h=2).flops_step()
    g = oracle.mla_backward(x["q"], x["c_kv"], x["k_rope"], x["W_UK"], x["W_UV"], x["dout"], p.q_offset, True)
    out, lse = oracle.mla_forward(x["q"], x["c_kv"], x["k_rope"], x["W_UK"], x["W_UV"], p.q_offset, True)
    for h in (0, 2):
        k = keep[h]
        np.testing.assert_allclose(k["dW_UK_h"], g["dW_UK"][:, h * 4:(h + 1) * 4], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(k["dW_UV_h"], g["dW_UV"][:, h * 5:(h + 1) * 5], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(k["dq_h"], g["dq"][0, :, h], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(k["out_h"], out[0, :, h], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(k["lse_h"], lse[0, h], rtol=1e-12, atol=1e-14)


def test_flop_conventions_at_the_dsv3_shard():
    """The algorithmic step count and the FlashAttention convention at the DSV3 SP=8
    last-rank shard, against the closed forms: 2048 queries at offset 14336 see
    2048 * 14336 + 2048 * 2049 / 2 = 31,458,304 keys in all; the step is three times
    the forward (attention 2 * P * n_h * 320, reconstruction 2 * 16384 * 512 * n_h * 256),
    and the FlashAttention convention adds the backward's score recompute 2 * P * n_h * 192."""
    from mla_attention_sequence_gb300.configs import dsv3_rank
    p = dsv3_rank(7)
    P = 2048 * 14336 + 2048 * 2049 // 2
    assert p.pairs == P == 31_458_304
    fwd = 2 * P * 128 * 320 + 2 * 16384 * 512 * 128 * 256
    assert p.flops_step() == 3 * fwd
    assert p.flops_step_fa() - p.flops_step() == 2 * P * 128 * 192
