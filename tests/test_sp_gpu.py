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
