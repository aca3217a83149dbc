"""The sequence-parallel exchange on the GPU with its default local op (the C
ABI) and NCCL, in a one-rank group: the collectives run on device tensors and
the results equal direct calls of laga_mla_fwd / laga_mla_bwd. The two-rank
exchange logic is tested on CPU ranks (test_sp_gloo.py); this run has one GPU.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist

from mla_attention_sequence_gb300 import laga
from mla_attention_sequence_gb300.configs import Problem
from mla_attention_sequence_gb300.sp import Layout, SPAttention
from mla_attention_sequence_gb300.synth import make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nccl_group():
    from mla_attention_sequence_gb300 import build
    build.build()
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    torch.cuda.set_device(0)
    dist.init_process_group("nccl", rank=0, world_size=1)
    yield
    dist.destroy_process_group()


@pytest.mark.parametrize("kind", ["contiguous", "zigzag"])
def test_sp_exchange_on_gpu_matches_direct_calls(nccl_group, kind):
    p = Problem(B=1, Sq=512, S=512, n_h=2, d_c=512, d_nope=128, d_rope=64, d_v=128, causal=True, dtype="bf16")
    x = make_inputs(p, seed=91)
    dev = torch.device("cuda", 0)
    t = {k: torch.from_numpy(v).to(dev).to(torch.bfloat16) for k, v in x.items()}
    lay = Layout(seq=p.S, sp=1, kind=kind)  # zigzag at SP=1: two segments, chunks 0 and 1
    att = SPAttention(lay)
    rows = lay.rows(0).to(dev)
    out, lse = att.forward(t["q"][:, rows].contiguous(), t["c_kv"][:, rows].contiguous(),
                           t["k_rope"][:, rows].contiguous(), t["W_UK"], t["W_UV"])
    g = att.backward(t["dout"][:, rows].contiguous())
    laga.check(dev)
    ref_out, ref_lse = laga.fwd(t["q"], t["c_kv"], t["k_rope"], t["W_UK"], t["W_UV"], 0, True)
    ref = laga.bwd(t["q"], t["c_kv"], t["k_rope"], t["W_UK"], t["W_UV"], ref_out, ref_lse, t["dout"], 0, True)
    laga.check(dev)
    got = {"out": out, "lse": lse, **g}
    want = {"out": ref_out, "lse": ref_lse, **ref}
    for k in want:
        a = got[k].float().cpu().numpy().astype(np.float64)
        r = want[k].float().cpu().numpy().astype(np.float64)
        assert np.abs(a - r).max() <= 2e-2 * np.abs(r).max(), k
    if kind == "contiguous":  # the same call on the same tensors: bitwise
        for k in want:
            assert torch.equal(got[k], want[k]), k


@pytest.mark.parametrize("kind", ["contiguous", "zigzag"])
def test_sp_overlapped_exchange_on_gpu_matches_direct_calls(nccl_group, kind):
    """The overlapped forward (per-source broadcast, rows rebuilt chunk by chunk
    with laga_mla_reconstruct_rows, attention on the prebuilt K/V, backward
    reusing them) in a one-rank group equals direct laga_mla_fwd / laga_mla_bwd."""
    p = Problem(B=1, Sq=512, S=512, n_h=2, d_c=512, d_nope=128, d_rope=64, d_v=128, causal=True, dtype="bf16")
    x = make_inputs(p, seed=92)
    dev = torch.device("cuda", 0)
    t = {k: torch.from_numpy(v).to(dev).to(torch.bfloat16) for k, v in x.items()}
    lay = Layout(seq=p.S, sp=1, kind=kind)
    att = SPAttention(lay, overlap=True)
    rows = lay.rows(0).to(dev)
    out, lse = att.forward(t["q"][:, rows].contiguous(), t["c_kv"][:, rows].contiguous(),
                           t["k_rope"][:, rows].contiguous(), t["W_UK"], t["W_UV"])
    g = att.backward(t["dout"][:, rows].contiguous())
    laga.check(dev)
    pos = lay.query_args(0)
    ref_out, ref_lse = laga.fwd(t["q"][:, rows].contiguous(), t["c_kv"], t["k_rope"], t["W_UK"], t["W_UV"],
                                pos["q_offset"], True, q_split=pos["q_split"], q_offset2=pos["q_offset2"])
    ref = laga.bwd(t["q"][:, rows].contiguous(), t["c_kv"], t["k_rope"], t["W_UK"], t["W_UV"], ref_out, ref_lse,
                   t["dout"][:, rows].contiguous(), pos["q_offset"], True, q_split=pos["q_split"],
                   q_offset2=pos["q_offset2"])
    laga.check(dev)
    got = {"out": out, "lse": lse, **g}
    want = {"out": ref_out, "lse": ref_lse, **ref}
    for k in want:  # the same kernels on the same rows and inputs: bitwise
        assert torch.equal(got[k], want[k]), k


def test_reconstruct_rows_in_chunks_then_prebuilt_forward_is_bitwise():
    """K_nope / V rebuilt by laga_mla_reconstruct_rows over ragged, out-of-order row
    ranges (the last one past the padded prefix), then laga_mla_fwd with
    LAGA_FLAG_KV_PREBUILT, equals the plain forward bit for bit; B = 2 covers the
    per-batch row offsets."""
    from mla_attention_sequence_gb300 import build
    build.build()
    p = Problem(B=2, Sq=300, S=900, n_h=3, d_c=512, d_nope=128, d_rope=64, d_v=128, q_offset=500, causal=True,
                dtype="bf16")
    x = make_inputs(p, seed=93)
    dev = torch.device("cuda", 0)
    t = {k: torch.from_numpy(v).to(dev).to(torch.bfloat16) for k, v in x.items()}
    args = (t["q"], t["c_kv"], t["k_rope"], t["W_UK"], t["W_UV"])
    ws = torch.empty(laga.fwd_workspace_bytes(p), dtype=torch.uint8, device=dev)
    for row0, rows in ((384, 256), (0, 128), (640, 4096), (128, 256)):
        laga.reconstruct_rows(*args, row0, rows, ws, q_offset=p.q_offset)
    out, lse = laga.fwd(*args, p.q_offset, True, workspace=ws, kv_prebuilt=True)
    ref_out, ref_lse = laga.fwd(*args, p.q_offset, True)
    laga.check(dev)
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)
    with pytest.raises(laga.LagaError):  # a range not ending on a tile boundary before the prefix end
        laga.reconstruct_rows(*args, 0, 100, ws, q_offset=p.q_offset)
