"""The sequence-parallel exchange (mla_attention_sequence_gb300.sp) on CPU ranks.

Two gloo ranks, each holding its shard of the latent, the RoPE key, the queries
and dout. The local op is the fp64 oracle (test side only), so the collectives'
plumbing is checked exactly: the gathered latent equals the full one, every
rank's out / lse / dq rows equal the SP=1 oracle's rows, the reduce-scattered
dc_kv / dk_rope rows and the all-reduced dW_UK / dW_UV equal the SP=1 oracle's
gradients. Contiguous and zigzag shard layouts.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from mla_attention_sequence_gb300.configs import Problem
from mla_attention_sequence_gb300.sp import Layout, SPAttention
from mla_attention_sequence_gb300.synth import make_inputs


def _oracle_fwd(q, c_kv, k_rope, W_UK, W_UV, q_offset, causal, q_split, q_offset2):
    import oracle
    f = lambda t: t.numpy()
    out, lse = oracle.mla_forward(f(q), f(c_kv), f(k_rope), f(W_UK), f(W_UV), q_offset, causal, None, q_split,
                                  q_offset2)
    return torch.from_numpy(out), torch.from_numpy(lse)


def _oracle_bwd(q, c_kv, k_rope, W_UK, W_UV, out, lse, dout, q_offset, causal, q_split, q_offset2):
    import oracle
    f = lambda t: t.numpy()
    g = oracle.mla_backward(f(q), f(c_kv), f(k_rope), f(W_UK), f(W_UV), f(dout), q_offset, causal, None, q_split,
                            q_offset2)
    return {k: torch.from_numpy(v) for k, v in g.items()}


PROBLEM = Problem(B=2, Sq=16, S=16, n_h=2, d_c=6, d_nope=3, d_rope=2, d_v=4, dtype="f32")


def _rank_main(rank, world, port, kind, errfile):
    try:
        os.environ["MASTER_ADDR"] = "127.0.0.1"
        os.environ["MASTER_PORT"] = str(port)
        dist.init_process_group("gloo", rank=rank, world_size=world)
        import oracle
        p = PROBLEM
        x = {k: torch.from_numpy(v.astype(np.float64)) for k, v in make_inputs(p, seed=77).items()}
        lay = Layout(seq=p.S, sp=world, kind=kind)
        rows = lay.rows(rank)
        att = SPAttention(lay, causal=True, local_fwd=_oracle_fwd, local_bwd=_oracle_bwd)
        # the gathered latent is the full one, in sequence order
        c_full, r_full = att.gather_latent(x["c_kv"][:, rows].contiguous(), x["k_rope"][:, rows].contiguous())
        assert torch.equal(c_full, x["c_kv"]) and torch.equal(r_full, x["k_rope"])
        out, lse = att.forward(x["q"][:, rows].contiguous(), x["c_kv"][:, rows].contiguous(),
                               x["k_rope"][:, rows].contiguous(), x["W_UK"], x["W_UV"])
        g = att.backward(x["dout"][:, rows].contiguous())
        # SP=1 reference over the whole sequence
        n = {k: v.numpy() for k, v in x.items()}
        ro, rl = oracle.mla_forward(n["q"], n["c_kv"], n["k_rope"], n["W_UK"], n["W_UV"], 0, True)
        rg = oracle.mla_backward(n["q"], n["c_kv"], n["k_rope"], n["W_UK"], n["W_UV"], n["dout"], 0, True)
        r = rows.numpy()
        np.testing.assert_allclose(out.numpy(), ro[:, r], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse.numpy(), rl[:, :, r], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(g["dq"].numpy(), rg["dq"][:, r], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(g["dc_kv"].numpy(), rg["dc_kv"][:, r], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(g["dk_rope"].numpy(), rg["dk_rope"][:, r], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(g["dW_UK"].numpy(), rg["dW_UK"], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(g["dW_UV"].numpy(), rg["dW_UV"], rtol=1e-10, atol=1e-12)
        dist.barrier()
        dist.destroy_process_group()
    except BaseException as e:  # report to the parent, which fails the test
        with open(f"{errfile}.{rank}", "w") as f:
            f.write(repr(e))
        raise


class _OracleOps:
    """The overlapped path's local steps on CPU: the rebuild records each row range
    with the latent rows it saw at that moment; the forward checks that the
    ranges cover the sequence and runs the oracle on the gathered latent."""

    def prepare(self, q, c_kv, k_rope, W_UK, W_UV, pos, causal):
        return {"rebuilt": []}

    def rebuild(self, q, c_kv, k_rope, W_UK, W_UV, pos, causal, row0, rows, ws):
        end = min(row0 + rows, c_kv.shape[1])
        ws["rebuilt"].append((row0, end, c_kv[:, row0:end].clone(), k_rope[:, row0:end].clone()))

    def fwd_prebuilt(self, q, c_kv, k_rope, W_UK, W_UV, pos, causal, ws):
        covered = sorted((a, e) for a, e, _, _ in ws["rebuilt"])
        assert covered[0][0] == 0 and covered[-1][1] == c_kv.shape[1]
        assert all(covered[k][1] == covered[k + 1][0] for k in range(len(covered) - 1)), covered
        return _oracle_fwd(q, c_kv, k_rope, W_UK, W_UV, pos["q_offset"], causal, pos["q_split"], pos["q_offset2"])

    def bwd_reuse(self, q, c_kv, k_rope, W_UK, W_UV, out, lse, dout, pos, causal, ws):
        return _oracle_bwd(q, c_kv, k_rope, W_UK, W_UV, out, lse, dout, pos["q_offset"], causal, pos["q_split"],
                           pos["q_offset2"])


def _rank_main_overlap(rank, world, port, kind, errfile):
    try:
        os.environ["MASTER_ADDR"] = "127.0.0.1"
        os.environ["MASTER_PORT"] = str(port)
        dist.init_process_group("gloo", rank=rank, world_size=world)
        import oracle
        p = PROBLEM
        x = {k: torch.from_numpy(v.astype(np.float64)) for k, v in make_inputs(p, seed=78).items()}
        lay = Layout(seq=p.S, sp=world, kind=kind)
        rows = lay.rows(rank)
        ops = _OracleOps()
        att = SPAttention(lay, causal=True, overlap=True, ops=ops)
        captured = {}
        orig_prepare = ops.prepare

        def prepare(*a):
            captured["ws"] = orig_prepare(*a)
            return captured["ws"]
        ops.prepare = prepare
        out, lse = att.forward(x["q"][:, rows].contiguous(), x["c_kv"][:, rows].contiguous(),
                               x["k_rope"][:, rows].contiguous(), x["W_UK"], x["W_UV"])
        # every chunk was rebuilt after its rows had arrived, own rows first
        rebuilt = captured["ws"]["rebuilt"]
        for a, e, c, r in rebuilt:
            assert torch.equal(c, x["c_kv"][:, a:e]) and torch.equal(r, x["k_rope"][:, a:e]), (a, e)
        own = [(a, a + n) for a, n in lay.segments(rank)]
        assert [(a, e) for a, e, _, _ in rebuilt[:len(own)]] == own
        g = att.backward(x["dout"][:, rows].contiguous())
        n = {k: v.numpy() for k, v in x.items()}
        ro, rl = oracle.mla_forward(n["q"], n["c_kv"], n["k_rope"], n["W_UK"], n["W_UV"], 0, True)
        rg = oracle.mla_backward(n["q"], n["c_kv"], n["k_rope"], n["W_UK"], n["W_UV"], n["dout"], 0, True)
        r = rows.numpy()
        np.testing.assert_allclose(out.numpy(), ro[:, r], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse.numpy(), rl[:, :, r], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(g["dq"].numpy(), rg["dq"][:, r], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(g["dc_kv"].numpy(), rg["dc_kv"][:, r], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(g["dk_rope"].numpy(), rg["dk_rope"][:, r], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(g["dW_UK"].numpy(), rg["dW_UK"], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(g["dW_UV"].numpy(), rg["dW_UV"], rtol=1e-10, atol=1e-12)
        dist.barrier()
        dist.destroy_process_group()
    except BaseException as e:  # report to the parent, which fails the test
        with open(f"{errfile}.{rank}", "w") as f:
            f.write(repr(e))
        raise


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("kind", ["contiguous", "zigzag"])
def test_sp_exchange_two_gloo_ranks(kind, tmp_path):
    errfile = str(tmp_path / "err")
    mp.start_processes(_rank_main, args=(2, _free_port(), kind, errfile), nprocs=2, join=True,
                       start_method="spawn")
    for r in range(2):
        assert not os.path.exists(f"{errfile}.{r}"), open(f"{errfile}.{r}").read()


def test_layout_rows_cover_the_sequence_once():
    for kind in ("contiguous", "zigzag"):
        for sp in (1, 2, 4, 8):
            lay = Layout(seq=64 * sp, sp=sp, kind=kind)
            allrows = torch.cat([lay.rows(r) for r in range(sp)])
            assert torch.equal(torch.sort(allrows).values, torch.arange(lay.seq))
            order = lay.gather_order()
            assert torch.equal(allrows[order], torch.arange(lay.seq))


def test_zigzag_query_arguments():
    lay = Layout(seq=16384, sp=8, kind="zigzag")
    assert lay.query_args(0) == {"q_offset": 0, "q_split": 1024, "q_offset2": 15 * 1024}
    assert lay.query_args(7) == {"q_offset": 7 * 1024, "q_split": 1024, "q_offset2": 8 * 1024}
    assert Layout(seq=16384, sp=8).query_args(7) == {"q_offset": 14336, "q_split": 0, "q_offset2": 0}


def test_bytes_per_step_of_the_dsv3_layer():
    """Per rank and step at SP=8, S=16384: the latent all-gather and the gradient
    reduce-scatter each move 7/8 of the 576-wide bf16 latent (18.9 MB)."""
    att = SPAttention.__new__(SPAttention)  # no process group needed for the arithmetic
    att.layout = Layout(seq=16384, sp=8)
    b = att.bytes_per_step(B=1, d_c=512, d_rope=64, n_h=128, d_nope=128, d_v=128)
    assert b["all_gather"] == pytest.approx(16384 * 576 * 2 * 7 / 8)
    assert b["reduce_scatter"] == b["all_gather"]


@pytest.mark.parametrize("kind", ["contiguous", "zigzag"])
def test_sp_overlapped_gather_two_gloo_ranks(kind, tmp_path):
    """The overlapped forward: per-source broadcasts, each chunk rebuilt once its
    rows have arrived (own rows first), then the attention on the prebuilt K/V;
    results equal the SP = 1 oracle's."""
    errfile = str(tmp_path / "err")
    mp.start_processes(_rank_main_overlap, args=(2, _free_port(), kind, errfile), nprocs=2, join=True,
                       start_method="spawn")
    for r in range(2):
        assert not os.path.exists(f"{errfile}.{r}"), open(f"{errfile}.{r}").read()
