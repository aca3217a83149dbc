"""The fp64 oracle over many heads at once, for the full-size parity tests.

Test helper only (not a test module). The oracle itself runs one (batch, head)
at a time; here the heads are dealt out to worker processes, each worker calls
the per-head oracle for its heads and adds up the contributions that sum over
heads (dc_kv, dk_rope), and the parent stitches the per-head outputs together.
Nothing of the method's arithmetic lives here: every number comes from
oracle.mla_backward_head.

The workers are started with the "spawn" method: a process forked after the
parent has made CUDA calls can hang.
"""
from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np


def _worker(args):
    import oracle
    xs, heads, q_offset, causal, scale = args
    # this worker's heads only, renumbered 0..len(heads)-1 (the per-head oracle reads
    # the head count and widths off the arrays it is given)
    x = {k: np.asarray(v, dtype=np.float64) for k, v in xs.items()}
    B, Sq, n_h, d_qk = x["q"].shape
    S, d_c = x["c_kv"].shape[1], x["c_kv"].shape[2]
    d_nope = x["W_UK"].shape[1] // n_h
    d_v = x["W_UV"].shape[1] // n_h
    res = {"heads": heads, "dc_kv": np.zeros((B, S, d_c)), "dk_rope": np.zeros((B, S, d_qk - d_nope)),
           "dq": {}, "out": {}, "lse": {}, "dW_UK": {}, "dW_UV": {}}
    for hl, h in enumerate(heads):
        dWk = np.zeros((d_c, d_nope))
        dWv = np.zeros((d_c, d_v))
        for b in range(B):
            g = oracle.mla_backward_head(x["q"], x["c_kv"], x["k_rope"], x["W_UK"], x["W_UV"], x["dout"], b, hl,
                                         q_offset, causal, scale)
            res["dq"][(b, h)] = g["dq_h"]
            res["out"][(b, h)] = g["out_h"]
            res["lse"][(b, h)] = g["lse_h"]
            res["dc_kv"][b] += g["dc_kv_h"]
            res["dk_rope"][b] += g["dK_rope_h"]
            dWk += g["dW_UK_h"]
            dWv += g["dW_UV_h"]
        res["dW_UK"][h] = dWk
        res["dW_UV"][h] = dWv
    return res


def _head_slice(p, x, heads):
    """The inputs one worker needs: its heads' q, dout and weight columns, and the
    shared latent and RoPE key."""
    cols_k = np.concatenate([np.arange(h * p.d_nope, (h + 1) * p.d_nope) for h in heads])
    cols_v = np.concatenate([np.arange(h * p.d_v, (h + 1) * p.d_v) for h in heads])
    return {"q": np.ascontiguousarray(x["q"][:, :, heads]), "dout": np.ascontiguousarray(x["dout"][:, :, heads]),
            "W_UK": np.ascontiguousarray(x["W_UK"][:, cols_k]), "W_UV": np.ascontiguousarray(x["W_UV"][:, cols_v]),
            "c_kv": x["c_kv"], "k_rope": x["k_rope"]}


def full_backward(p, x, scale=None, workers=None):
    """Every output of the block (out, lse, dq, dc_kv, dk_rope, dW_UK, dW_UV) from the
    per-head oracle, heads spread over `workers` spawned processes."""
    import oracle
    pos = oracle.query_positions(p.Sq, p.q_offset, p.q_split, p.q_offset2) if p.q_split > 0 else p.q_offset
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    n = workers or max(1, min(p.n_h, cores // 4))
    threads = max(1, cores // n)
    chunks = [list(range(p.n_h))[i::n] for i in range(n)]
    saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    for k in saved:
        os.environ[k] = str(threads)
    try:
        with mp.get_context("spawn").Pool(n) as pool:
            parts = pool.map(_worker, [(_head_slice(p, x, c), c, pos, p.causal, scale) for c in chunks])
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    out = np.zeros((p.B, p.Sq, p.n_h, p.d_v))
    lse = np.zeros((p.B, p.n_h, p.Sq))
    dq = np.zeros((p.B, p.Sq, p.n_h, p.d_qk))
    dc_kv = np.zeros((p.B, p.S, p.d_c))
    dk_rope = np.zeros((p.B, p.S, p.d_rope))
    dW_UK = np.zeros((p.d_c, p.n_h * p.d_nope))
    dW_UV = np.zeros((p.d_c, p.n_h * p.d_v))
    for r in parts:
        dc_kv += r["dc_kv"]
        dk_rope += r["dk_rope"]
        for (b, h), v in r["dq"].items():
            dq[b, :, h] = v
            out[b, :, h] = r["out"][(b, h)]
            lse[b, h] = r["lse"][(b, h)]
        for h, v in r["dW_UK"].items():
            dW_UK[:, h * p.d_nope:(h + 1) * p.d_nope] = v
            dW_UV[:, h * p.d_v:(h + 1) * p.d_v] = r["dW_UV"][h]
    return {"out": out, "lse": lse, "dq": dq, "dc_kv": dc_kv, "dk_rope": dk_rope, "dW_UK": dW_UK, "dW_UV": dW_UV}
