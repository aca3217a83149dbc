"""Pins for the fp64 oracle: checks against things other than the oracle itself.

The LAGA page ("A Training-Memory Regression in MLA Sequence Parallelism ...",
Abstract) prints no worked example, so the oracle is pinned by
  * brute-force attention written with scalar Python loops,
  * the absorbed MLA form the Abstract contrasts LAGA with (W_UK folded into
    the query, V recovered through W_UV after attending in latent space),
  * the Abstract's sequence-parallel claim: an SP shard's rows equal the SP=1
    rows, and shard gradients sum to the SP=1 gradients,
  * central finite differences of the loss <dout, out> for every input,
  * closed-form special cases, a hand-worked two-token example,
  * gradient identities (row-sum of ds is zero, homogeneity),
  * torch autograd in float64 on CPU as an independent derivative engine,
and a set of planted mistakes, each of which one of these pins must catch.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import oracle.laga_oracle as O
from mla_attention_sequence_gb300.configs import Problem
from mla_attention_sequence_gb300.synth import make_inputs


def small(B=2, Sq=5, S=9, n_h=2, d_c=6, d_nope=3, d_rope=2, d_v=4, q_offset=4, causal=True):
    return Problem(B=B, Sq=Sq, S=S, n_h=n_h, d_c=d_c, d_nope=d_nope, d_rope=d_rope, d_v=d_v,
                   q_offset=q_offset, causal=causal, dtype="f32")


def inputs64(p, seed=0):
    x = make_inputs(p, seed)
    return {k: v.astype(np.float64) for k, v in x.items()}


def run_fwd(p, x, scale=None):
    return oracle.mla_forward(x["q"], x["c_kv"], x["k_rope"], x["W_UK"], x["W_UV"],
                              p.q_offset, p.causal, scale)


def run_bwd(p, x, scale=None):
    return oracle.mla_backward(x["q"], x["c_kv"], x["k_rope"], x["W_UK"], x["W_UV"], x["dout"],
                               p.q_offset, p.causal, scale)


# --------------------------------------------------------------------------- brute force
def brute_force_forward(p, x, scale):
    """Scalar-loop attention: every product and exponential written out one by one."""
    out = np.zeros((p.B, p.Sq, p.n_h, p.d_v))
    lse = np.zeros((p.B, p.n_h, p.Sq))
    for b in range(p.B):
        for h in range(p.n_h):
            K = [[0.0] * p.d_qk for _ in range(p.S)]
            V = [[0.0] * p.d_v for _ in range(p.S)]
            for j in range(p.S):
                for d in range(p.d_nope):
                    K[j][d] = sum(x["c_kv"][b, j, c] * x["W_UK"][c, h * p.d_nope + d]
                                  for c in range(p.d_c))
                for d in range(p.d_rope):
                    K[j][p.d_nope + d] = x["k_rope"][b, j, d]
                for d in range(p.d_v):
                    V[j][d] = sum(x["c_kv"][b, j, c] * x["W_UV"][c, h * p.d_v + d]
                                  for c in range(p.d_c))
            for i in range(p.Sq):
                last = p.q_offset + i if p.causal else p.S - 1
                keys = range(0, last + 1)
                s = {j: scale * sum(x["q"][b, i, h, d] * K[j][d] for d in range(p.d_qk)) for j in keys}
                m = max(s.values())
                z = sum(math.exp(s[j] - m) for j in keys)
                lse[b, h, i] = m + math.log(z)
                for d in range(p.d_v):
                    out[b, i, h, d] = sum(math.exp(s[j] - m) / z * V[j][d] for j in keys)
    return out, lse


@pytest.mark.parametrize("causal,q_offset", [(True, 4), (True, 0), (False, 0)])
def test_brute_force_attention(causal, q_offset):
    p = small(causal=causal, q_offset=q_offset)
    x = inputs64(p, seed=1)
    scale = O.default_scale(p.d_nope, p.d_rope)
    out, lse = run_fwd(p, x)
    out_bf, lse_bf = brute_force_forward(p, x, scale)
    np.testing.assert_allclose(out, out_bf, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, lse_bf, rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------- absorbed form
def absorbed_forward(p, x, scale):
    """The absorbed MLA form: scores through q_nope W_UK^T against the latent, output
    attends over the latent and is mapped through W_UV afterwards."""
    out = np.zeros((p.B, p.Sq, p.n_h, p.d_v))
    lse = np.zeros((p.B, p.n_h, p.Sq))
    for b in range(p.B):
        c = x["c_kv"][b]
        for h in range(p.n_h):
            wk = x["W_UK"][:, h * p.d_nope:(h + 1) * p.d_nope]
            wv = x["W_UV"][:, h * p.d_v:(h + 1) * p.d_v]
            qn = x["q"][b, :, h, :p.d_nope]
            qr = x["q"][b, :, h, p.d_nope:]
            q_lat = qn @ wk.T  # [Sq, d_c]: the absorbed query
            s = scale * (q_lat @ c.T + qr @ x["k_rope"][b].T)
            if p.causal:
                s = np.where(np.arange(p.S)[None, :] <= p.q_offset + np.arange(p.Sq)[:, None], s, -np.inf)
            m = s.max(1, keepdims=True)
            e = np.exp(s - m)
            lse[b, h] = m[:, 0] + np.log(e.sum(1))
            ctx_lat = (e / e.sum(1, keepdims=True)) @ c  # attention in latent space
            out[b, :, h, :] = ctx_lat @ wv
    return out, lse


def test_oracle_absorbed_form_equals_explicit_and_the_test_restatement():
    """The oracle's absorbed form (used by the GPU absorbed path's parity tests)
    equals the explicit form and this file's own restatement of the absorbed form,
    on a causal shard and a non-causal problem; its intermediates have the widths
    the Abstract describes (n_h x d_c per query row)."""
    for causal, q_offset in [(True, 5), (False, 0)]:
        p = small(n_h=3, S=11, Sq=6, q_offset=q_offset, causal=causal)
        x = inputs64(p, seed=4)
        keep = {}
        out, lse = oracle.absorbed_forward(x["q"], x["c_kv"], x["k_rope"], x["W_UK"], x["W_UV"], p.q_offset,
                                           p.causal, keep=keep)
        ref_out, ref_lse = run_fwd(p, x)
        np.testing.assert_allclose(out, ref_out, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(lse, ref_lse, rtol=1e-11, atol=1e-12)
        if causal:
            o2, l2 = absorbed_forward(p, x, O.default_scale(p.d_nope, p.d_rope))
            np.testing.assert_allclose(out, o2, rtol=1e-11, atol=1e-12)
        assert keep["q_lat"].shape == (p.B, p.Sq, p.n_h, p.d_c) and keep["ctx"].shape == (p.B, p.Sq, p.n_h, p.d_c)


def test_oracle_absorbed_form_hand_worked():
    """The hand-worked two-token example of the default-scale test, through the
    absorbed form: q_lat_1 = q_nope_1 W_UK^T = (0, 2 ln 3) against c_kv = I gives the
    same scores (0, ln 3) at scale 1/2, so out = (2, 5) and lse = (1, ln 4)."""
    ln3 = math.log(3.0)
    x = {"q": np.array([[[[0.0, 0.0, 0.0, 2.0]], [[1.0, 0.0, 0.0, 0.0]]]]),
         "c_kv": np.array([[[1.0, 0.0], [0.0, 1.0]]]), "k_rope": np.array([[[0.0, 1.0], [0.0, 0.0]]]),
         "W_UK": np.array([[0.0, 0.0], [2.0 * ln3, 0.0]]), "W_UV": np.array([[2.0], [6.0]])}
    keep = {}
    out, lse = oracle.absorbed_forward(x["q"], x["c_kv"], x["k_rope"], x["W_UK"], x["W_UV"], 0, True, keep=keep)
    np.testing.assert_allclose(out[0, :, 0, 0], [2.0, 5.0], rtol=1e-14)
    np.testing.assert_allclose(lse[0, 0], [1.0, math.log(4.0)], rtol=1e-14)
    np.testing.assert_allclose(keep["q_lat"][0, 1, 0], [0.0, 2.0 * ln3], rtol=1e-14)
    np.testing.assert_allclose(keep["ctx"][0, 1, 0], [0.25, 0.75], rtol=1e-14)


@pytest.mark.parametrize("seed", [0, 7])
def test_absorbed_form_equals_explicit(seed):
    p = small(n_h=3, S=11, Sq=6, q_offset=5)
    x = inputs64(p, seed)
    scale = O.default_scale(p.d_nope, p.d_rope)
    out, lse = run_fwd(p, x)
    out_a, lse_a = absorbed_forward(p, x, scale)
    np.testing.assert_allclose(out, out_a, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(lse, lse_a, rtol=1e-11, atol=1e-12)


def test_absorbed_form_mid_heads_subset():
    """Absorbed vs explicit at the real latent width d_c=512, head dims 128/64."""
    p = Problem(B=1, Sq=24, S=40, n_h=2, d_c=512, d_nope=128, d_rope=64, d_v=128,
                q_offset=16, causal=True, dtype="bf16")
    x = inputs64(p, seed=3)
    scale = O.default_scale(p.d_nope, p.d_rope)
    out, lse = run_fwd(p, x)
    out_a, lse_a = absorbed_forward(p, x, scale)
    np.testing.assert_allclose(out, out_a, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse, lse_a, rtol=1e-11, atol=1e-12)


# --------------------------------------------------------------------------- SP shards
@pytest.mark.parametrize("sp", [2, 4])
def test_sequence_parallel_shards_match_sp1(sp):
    S = 16
    p1 = small(B=1, Sq=S, S=S, q_offset=0)
    x = inputs64(p1, seed=11)
    out1, lse1 = run_fwd(p1, x)
    g1 = run_bwd(p1, x)
    sh = S // sp
    sums = {k: np.zeros_like(g1[k]) for k in ("dc_kv", "dk_rope", "dW_UK", "dW_UV")}
    for r in range(sp):
        pr = p1.with_(Sq=sh, q_offset=r * sh)
        xr = dict(x)
        xr["q"] = x["q"][:, r * sh:(r + 1) * sh]
        xr["dout"] = x["dout"][:, r * sh:(r + 1) * sh]
        o, l = run_fwd(pr, xr)
        g = run_bwd(pr, xr)
        np.testing.assert_allclose(o, out1[:, r * sh:(r + 1) * sh], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(l, lse1[:, :, r * sh:(r + 1) * sh], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(g["dq"], g1["dq"][:, r * sh:(r + 1) * sh], rtol=1e-11, atol=1e-13)
        # latent rows beyond the shard's causal prefix get no gradient
        np.testing.assert_array_equal(g["dc_kv"][:, (r + 1) * sh:], 0.0)
        np.testing.assert_array_equal(g["dk_rope"][:, (r + 1) * sh:], 0.0)
        for k in sums:
            sums[k] += g[k]
    for k in sums:
        np.testing.assert_allclose(sums[k], g1[k], rtol=1e-11, atol=1e-12)


# --------------------------------------------------------------------------- zigzag shards
@pytest.mark.parametrize("sp", [2, 4])
def test_zigzag_shards_match_sp1(sp):
    """Zigzag sequence parallelism: the sequence cut into 2*sp chunks, rank r holding
    chunks r and 2*sp-1-r as one two-segment shard. Gathered, the ranks' outputs,
    LSEs and dq reproduce the SP=1 result row for row, and their latent and weight
    gradients sum to SP=1's."""
    S = 16
    c = S // (2 * sp)
    p1 = small(B=1, Sq=S, S=S, q_offset=0)
    x = inputs64(p1, seed=12)
    out1, lse1 = run_fwd(p1, x)
    g1 = run_bwd(p1, x)
    sums = {k: np.zeros_like(g1[k]) for k in ("dc_kv", "dk_rope", "dW_UK", "dW_UV")}
    for r in range(sp):
        a, b = c * r, c * (2 * sp - 1 - r)
        rows = np.r_[a:a + c, b:b + c]
        q, dout = x["q"][:, rows], x["dout"][:, rows]
        o, l = oracle.mla_forward(q, x["c_kv"], x["k_rope"], x["W_UK"], x["W_UV"], a, True, None, c, b)
        g = oracle.mla_backward(q, x["c_kv"], x["k_rope"], x["W_UK"], x["W_UV"], dout, a, True, None, c, b)
        np.testing.assert_allclose(o, out1[:, rows], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(l, lse1[:, :, rows], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(g["dq"], g1["dq"][:, rows], rtol=1e-11, atol=1e-13)
        for k in sums:
            sums[k] += g[k]
    for k in sums:
        np.testing.assert_allclose(sums[k], g1[k], rtol=1e-11, atol=1e-12)


def test_query_positions_of_a_two_segment_shard():
    np.testing.assert_array_equal(oracle.query_positions(6, 4), [4, 5, 6, 7, 8, 9])
    np.testing.assert_array_equal(oracle.query_positions(6, 4, 2, 20), [4, 5, 20, 21, 22, 23])


# --------------------------------------------------------------------------- finite differences
def loss(p, x):
    out, _ = run_fwd(p, x)
    return float((out * x["dout"]).sum())


@pytest.mark.parametrize("causal,q_offset", [(True, 3), (False, 0)])
def test_finite_differences_every_input(causal, q_offset):
    p = small(B=1, Sq=6, S=10, n_h=2, q_offset=q_offset, causal=causal)
    x = inputs64(p, seed=5)
    g = run_bwd(p, x)
    grads = {"q": g["dq"], "c_kv": g["dc_kv"], "k_rope": g["dk_rope"], "W_UK": g["dW_UK"],
             "W_UV": g["dW_UV"]}
    rng = np.random.default_rng(9)
    h = 1e-6
    for name, grad in grads.items():
        for trial in range(2):
            direction = rng.standard_normal(x[name].shape)
            xp, xm = dict(x), dict(x)
            xp[name] = x[name] + h * direction
            xm[name] = x[name] - h * direction
            fd = (loss(p, xp) - loss(p, xm)) / (2 * h)
            an = float((grad * direction).sum())
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, fd, an)
        # a few single entries, including one in the masked-out latent tail
        flat = grad.reshape(-1)
        for idx in [0, flat.size // 2, flat.size - 1]:
            xp, xm = dict(x), dict(x)
            xp[name] = x[name].copy().reshape(-1)
            xm[name] = x[name].copy().reshape(-1)
            xp[name][idx] += h
            xm[name][idx] -= h
            xp[name] = xp[name].reshape(x[name].shape)
            xm[name] = xm[name].reshape(x[name].shape)
            fd = (loss(p, xp) - loss(p, xm)) / (2 * h)
            assert abs(fd - flat[idx]) <= 1e-6 * max(1.0, abs(flat[idx])), (name, idx, fd, flat[idx])


def absorbed_loss(p, x, scale=None):
    out, _ = oracle.absorbed_forward(x["q"], x["c_kv"], x["k_rope"], x["W_UK"], x["W_UV"], p.q_offset, p.causal,
                                     scale)
    return float((out * x["dout"]).sum())


def run_absorbed_bwd(p, x, scale=None):
    return O.absorbed_backward(x["q"], x["c_kv"], x["k_rope"], x["W_UK"], x["W_UV"], x["dout"], p.q_offset,
                                    p.causal, scale)


@pytest.mark.parametrize("causal,q_offset", [(True, 3), (False, 0)])
def test_absorbed_backward_finite_differences(causal, q_offset):
    """The absorbed form's backward against central differences of its own forward
    (loss <dout, out> through q_lat and the latent-space context), in random
    directions of every input."""
    p = small(B=2, Sq=6, S=10, n_h=2, q_offset=q_offset, causal=causal)
    x = inputs64(p, seed=15)
    g = run_absorbed_bwd(p, x)
    grads = {"q": g["dq"], "c_kv": g["dc_kv"], "k_rope": g["dk_rope"], "W_UK": g["dW_UK"], "W_UV": g["dW_UV"]}
    rng = np.random.default_rng(19)
    h = 1e-6
    for name, grad in grads.items():
        for _ in range(3):
            direction = rng.standard_normal(x[name].shape)
            xp, xm = dict(x), dict(x)
            xp[name] = x[name] + h * direction
            xm[name] = x[name] - h * direction
            fd = (absorbed_loss(p, xp) - absorbed_loss(p, xm)) / (2 * h)
            an = float((grad * direction).sum())
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, fd, an)


def test_absorbed_backward_equals_explicit_backward():
    """Both forms compute one function, so their gradients agree (here also at an
    explicit scale and with the latent wider than a head)."""
    for scale in (None, 0.3):
        p = small(B=2, Sq=7, S=12, n_h=3, d_c=9, q_offset=5)
        x = inputs64(p, seed=23)
        a = run_absorbed_bwd(p, x, scale)
        e = run_bwd(p, x, scale)
        for k in e:
            np.testing.assert_allclose(a[k], e[k], rtol=1e-10, atol=1e-12, err_msg=k)


# --------------------------------------------------------------------------- autograd
def test_torch_autograd_float64():
    """torch's CPU autograd in float64 differentiates the explicit form independently."""
    p = small(B=2, Sq=7, S=12, n_h=3, q_offset=5)
    x = inputs64(p, seed=21)
    t = {k: torch.tensor(v, requires_grad=(k != "dout")) for k, v in x.items()}
    scale = O.default_scale(p.d_nope, p.d_rope)
    k_nope = (t["c_kv"] @ t["W_UK"]).view(p.B, p.S, p.n_h, p.d_nope)
    v = (t["c_kv"] @ t["W_UV"]).view(p.B, p.S, p.n_h, p.d_v)
    k = torch.cat([k_nope, t["k_rope"][:, :, None, :].expand(p.B, p.S, p.n_h, p.d_rope)], dim=-1)
    mask = torch.arange(p.S)[None, :] <= (p.q_offset + torch.arange(p.Sq))[:, None]
    s = torch.einsum("bihd,bjhd->bhij", t["q"], k) * scale
    s = s.masked_fill(~mask, float("-inf"))
    out = torch.einsum("bhij,bjhd->bihd", torch.softmax(s, dim=-1), v)
    lse = torch.logsumexp(s, dim=-1)
    (out * t["dout"]).sum().backward()
    o, l = run_fwd(p, x)
    g = run_bwd(p, x)
    np.testing.assert_allclose(o, out.detach().numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l, lse.detach().numpy(), rtol=1e-12, atol=1e-13)
    for name, key in [("q", "dq"), ("c_kv", "dc_kv"), ("k_rope", "dk_rope"),
                      ("W_UK", "dW_UK"), ("W_UV", "dW_UV")]:
        np.testing.assert_allclose(g[key], t[name].grad.numpy(), rtol=1e-10, atol=1e-12)


# --------------------------------------------------------------------------- closed forms
def test_single_query_sees_only_key_zero():
    p = small(B=1, Sq=1, S=7, q_offset=0)
    x = inputs64(p, seed=2)
    out, lse = run_fwd(p, x)
    k_nope, v = oracle.reconstruct(x["c_kv"], x["W_UK"], x["W_UV"], p.n_h)
    scale = O.default_scale(p.d_nope, p.d_rope)
    for h in range(p.n_h):
        np.testing.assert_allclose(out[0, 0, h], v[0, 0, h], rtol=1e-14)
        k0 = np.concatenate([k_nope[0, 0, h], x["k_rope"][0, 0]])
        np.testing.assert_allclose(lse[0, h, 0], scale * x["q"][0, 0, h] @ k0, rtol=1e-13)


def test_uniform_weights_give_prefix_mean():
    p = small(B=1, Sq=5, S=9, q_offset=4)
    x = inputs64(p, seed=4)
    x["W_UK"][:] = 0.0
    x["q"][..., p.d_nope:] = 0.0
    out, lse = run_fwd(p, x)
    _, v = oracle.reconstruct(x["c_kv"], x["W_UK"], x["W_UV"], p.n_h)
    for i in range(p.Sq):
        n = p.q_offset + i + 1
        np.testing.assert_allclose(out[0, i], v[0, :n].mean(axis=0), rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(lse[0, :, i], math.log(n), rtol=1e-14)


def test_noncausal_single_key():
    p = small(B=1, Sq=3, S=1, q_offset=0, causal=False)
    x = inputs64(p, seed=6)
    out, _ = run_fwd(p, x)
    _, v = oracle.reconstruct(x["c_kv"], x["W_UK"], x["W_UV"], p.n_h)
    for i in range(p.Sq):
        np.testing.assert_allclose(out[0, i], v[0, 0], rtol=1e-14)


def test_hand_worked_two_token_example():
    """Two tokens, one head, d_c=2, d_nope=d_rope=d_v=1, scale 1, worked by hand.

    c_kv = I, so K_nope = (0, ln 3) and V = (2, 6). Query 0 sees key 0 only:
    s_00 = q_0 . [0, 0.25] = 0.5. Query 1 sees both keys with scores (0, ln 3),
    weights (1/4, 3/4): out_1 = 2/4 + 18/4 = 5 and lse_1 = ln 4.
    Backward from dout = 1: dV = (5/4, 3/4); ds_1 = (1/4 (2-5), 3/4 (6-5)) = (-3/4, 3/4),
    ds_0 = 0; dq_1 = -3/4 K_0 + 3/4 K_1 = (3/4 ln 3, 3/4 - 3/16);
    dK_nope = (-3/4, 3/4) and dK_rope = 0; dW_UK = (-3/4, 3/4); dW_UV = (5/4, 3/4);
    dc_kv_0 = -3/4 (0, ln 3) + 5/4 (2, 6); dc_kv_1 = 3/4 (0, ln 3) + 3/4 (2, 6).
    """
    ln3 = math.log(3.0)
    x = {
        "q": np.array([[[[0.5, 2.0]], [[1.0, 0.0]]]]),
        "c_kv": np.array([[[1.0, 0.0], [0.0, 1.0]]]),
        "k_rope": np.array([[[0.25], [1.0]]]),
        "W_UK": np.array([[0.0], [ln3]]),
        "W_UV": np.array([[2.0], [6.0]]),
        "dout": np.ones((1, 2, 1, 1)),
    }
    out, lse = oracle.mla_forward(x["q"], x["c_kv"], x["k_rope"], x["W_UK"], x["W_UV"], 0, True, 1.0)
    np.testing.assert_allclose(out[0, :, 0, 0], [2.0, 5.0], rtol=1e-14)
    np.testing.assert_allclose(lse[0, 0], [0.5, math.log(4.0)], rtol=1e-14)
    g = oracle.mla_backward(x["q"], x["c_kv"], x["k_rope"], x["W_UK"], x["W_UV"], x["dout"], 0, True, 1.0)
    np.testing.assert_allclose(g["dq"][0, :, 0], [[0.0, 0.0], [0.75 * ln3, 0.5625]], atol=1e-14)
    np.testing.assert_allclose(g["dk_rope"][0, :, 0], [0.0, 0.0], atol=1e-14)
    np.testing.assert_allclose(g["dW_UK"][:, 0], [-0.75, 0.75], atol=1e-14)
    np.testing.assert_allclose(g["dW_UV"][:, 0], [1.25, 0.75], atol=1e-14)
    np.testing.assert_allclose(g["dc_kv"][0], [[2.5, 7.5 - 0.75 * ln3], [1.5, 4.5 + 0.75 * ln3]],
                               atol=1e-13)


def test_default_scale_is_one_over_root_of_query_key_width():
    """Reading of the pages' silence on the softmax scale: 1/sqrt(d_nope + d_rope),
    the width of the concatenated query/key (192 at the DeepSeek-V3 dims, 48 tiny)."""
    assert O.default_scale(128, 64) == pytest.approx(1.0 / 13.856406460551018, rel=1e-15)  # sqrt(192)
    assert O.default_scale(32, 16) == pytest.approx(1.0 / 6.928203230275509, rel=1e-15)  # sqrt(48)
    assert O.default_scale(2, 2) == 0.5


def test_hand_worked_example_at_the_default_scale():
    """Two tokens, one head, d_c = 2, d_nope = d_rope = 2 (so the default scale is
    1/sqrt(4) = 1/2), d_v = 1, worked by hand with no scale passed.

    c_kv = I, W_UK = [[0, 0], [2 ln 3, 0]]: K_nope = ((0, 0), (2 ln 3, 0)).
    k_rope = ((0, 1), (0, 0)); W_UV = (2, 6): V = (2, 6).
    Query 0 = (0, 0, 0, 2) sees key 0 only: s_00 = 1/2 * 2 = 1, out_0 = 2, lse_0 = 1.
    Query 1 = (1, 0, 0, 0) sees both: scores (0, 1/2 * 2 ln 3) = (0, ln 3), weights
    (1/4, 3/4): out_1 = 5, lse_1 = ln 4.
    Backward from dout = 1: ds_1 = (1/4 (2-5), 3/4 (6-5)) = (-3/4, 3/4), ds_0 = 0;
    dq_1 = 1/2 (-3/4 K_0 + 3/4 K_1) = (3/4 ln 3, 0, 0, -3/8);
    dK_0 = 1/2 (-3/4) q_1 = (-3/8, 0, 0, 0), dK_1 = (3/8, 0, 0, 0): dk_rope = 0;
    dW_UK = dK_nope = ((-3/8, 0), (3/8, 0)); dV = (1 + 1/4, 3/4): dW_UV = (5/4, 3/4);
    dc_kv_0 = (-3/8, 0) W_UK^T + 5/4 (2, 6) = (5/2, 15/2 - 3/4 ln 3),
    dc_kv_1 = (3/8, 0) W_UK^T + 3/4 (2, 6) = (3/2, 9/2 + 3/4 ln 3).
    A scale of 1/sqrt(d_nope) (or no scale) moves every one of these numbers."""
    ln3 = math.log(3.0)
    x = {
        "q": np.array([[[[0.0, 0.0, 0.0, 2.0]], [[1.0, 0.0, 0.0, 0.0]]]]),
        "c_kv": np.array([[[1.0, 0.0], [0.0, 1.0]]]),
        "k_rope": np.array([[[0.0, 1.0], [0.0, 0.0]]]),
        "W_UK": np.array([[0.0, 0.0], [2.0 * ln3, 0.0]]),
        "W_UV": np.array([[2.0], [6.0]]),
        "dout": np.ones((1, 2, 1, 1)),
    }
    out, lse = oracle.mla_forward(x["q"], x["c_kv"], x["k_rope"], x["W_UK"], x["W_UV"], 0, True)
    np.testing.assert_allclose(out[0, :, 0, 0], [2.0, 5.0], rtol=1e-14)
    np.testing.assert_allclose(lse[0, 0], [1.0, math.log(4.0)], rtol=1e-14)
    g = oracle.mla_backward(x["q"], x["c_kv"], x["k_rope"], x["W_UK"], x["W_UV"], x["dout"], 0, True)
    np.testing.assert_allclose(g["dq"][0, :, 0], [[0.0, 0.0, 0.0, 0.0], [0.75 * ln3, 0.0, 0.0, -0.375]],
                               atol=1e-14)
    np.testing.assert_allclose(g["dk_rope"][0], [[0.0, 0.0], [0.0, 0.0]], atol=1e-14)
    np.testing.assert_allclose(g["dW_UK"], [[-0.375, 0.0], [0.375, 0.0]], atol=1e-14)
    np.testing.assert_allclose(g["dW_UV"][:, 0], [1.25, 0.75], atol=1e-14)
    np.testing.assert_allclose(g["dc_kv"][0], [[2.5, 7.5 - 0.75 * ln3], [1.5, 4.5 + 0.75 * ln3]], atol=1e-13)


# --------------------------------------------------------------------------- identities
def inner(a, b):
    return float((np.asarray(a) * np.asarray(b)).sum())


def test_gradient_identities():
    """<dq,q> = <dK,K> (homogeneity of the scores); <dV,V> = <dout,out>;
    at the block level <dW_UK,W_UK> + <dk_rope,k_rope> = <dq,q>,
    <dW_UV,W_UV> = <dout,out>, <dc_kv,c_kv> = <dW_UK,W_UK> + <dW_UV,W_UV>."""
    p = small(B=2, Sq=8, S=13, n_h=3, q_offset=5)
    x = inputs64(p, seed=8)
    out, _ = run_fwd(p, x)
    g = run_bwd(p, x)
    lhs_q = inner(g["dq"], x["q"])
    np.testing.assert_allclose(inner(g["dW_UK"], x["W_UK"]) + inner(g["dk_rope"], x["k_rope"]), lhs_q,
                               rtol=1e-10)
    np.testing.assert_allclose(inner(g["dW_UV"], x["W_UV"]), inner(x["dout"], out), rtol=1e-10)
    np.testing.assert_allclose(inner(g["dc_kv"], x["c_kv"]),
                               inner(g["dW_UK"], x["W_UK"]) + inner(g["dW_UV"], x["W_UV"]), rtol=1e-10)


def test_key_shift_invariance_means_ds_rows_sum_to_zero():
    """Adding one vector to every visible key shifts each score row by a constant, so
    out is unchanged, and dq (= scale sum_j ds_ij K_j) is unchanged iff sum_j ds_ij = 0."""
    p = small(B=1, Sq=6, S=6, n_h=1, q_offset=0, causal=True)
    x = inputs64(p, seed=12)
    scale = O.default_scale(p.d_nope, p.d_rope)
    k_nope, v = O.reconstruct_head(x["c_kv"][0], x["W_UK"], x["W_UV"], 0, p.d_nope, p.d_v)
    K = O.head_key(k_nope, x["k_rope"][0])
    q_h = x["q"][0, :, 0, :]
    o, l = O.attention_head_forward(q_h, K, v, 0, True, scale)
    dq, _, _ = O.attention_head_backward(q_h, K, v, o, l, x["dout"][0, :, 0, :], 0, True, scale)
    shift = np.random.default_rng(1).standard_normal(p.d_qk)
    o2, l2 = O.attention_head_forward(q_h, K + shift, v, 0, True, scale)
    dq2, _, _ = O.attention_head_backward(q_h, K + shift, v, o2, l2, x["dout"][0, :, 0, :], 0, True, scale)
    np.testing.assert_allclose(o2, o, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dq2, dq, rtol=1e-9, atol=1e-12)


def test_probability_rows_sum_to_one():
    """With V = identity-like one-hot values the outputs are the probabilities themselves."""
    p = small(B=1, Sq=4, S=6, n_h=1, q_offset=2, d_v=6)
    x = inputs64(p, seed=13)
    scale = O.default_scale(p.d_nope, p.d_rope)
    k_nope, _ = O.reconstruct_head(x["c_kv"][0], x["W_UK"], x["W_UV"], 0, p.d_nope, p.d_v)
    K = O.head_key(k_nope, x["k_rope"][0])
    probs, _ = O.attention_head_forward(x["q"][0, :, 0, :], K, np.eye(p.S), p.q_offset, True, scale)
    np.testing.assert_allclose(probs.sum(axis=1), 1.0, rtol=1e-14)
    for i in range(p.Sq):
        assert np.all(probs[i, p.q_offset + i + 1:] == 0.0)
        assert np.all(probs[i, :p.q_offset + i + 1] > 0.0)


# --------------------------------------------------------------------------- planted mistakes
def _mask_off_by_one(rows, n_keys, q_offset, causal):
    rows = np.asarray(rows)
    if not causal:
        return np.ones((rows.shape[0], n_keys), dtype=bool)
    return np.arange(n_keys)[None, :] < (q_offset + rows)[:, None] + (rows[:, None] == 0)


def _reconstruct_head_swapped(c_kv_b, W_UK, W_UV, h, d_nope, d_v):
    c = np.asarray(c_kv_b, np.float64)
    hh = (h + 1) % (W_UK.shape[1] // d_nope)
    return c @ W_UK[:, hh * d_nope:(hh + 1) * d_nope], c @ W_UV[:, h * d_v:(h + 1) * d_v]


def _attention_backward_no_scale_dq(q_h, K_h, V_h, out_h, lse_h, dout_h, q_offset, causal, scale):
    dq, dK, dV = _ORIG_BWD(q_h, K_h, V_h, out_h, lse_h, dout_h, q_offset, causal, scale)
    return dq / scale, dK, dV


def _attention_backward_sign(q_h, K_h, V_h, out_h, lse_h, dout_h, q_offset, causal, scale):
    dq, dK, dV = _ORIG_BWD(q_h, K_h, V_h, out_h, lse_h, dout_h, q_offset, causal, scale)
    return dq, -dK, dV


def _head_key_transposed_rope(k_nope_h, k_rope_b):
    return np.concatenate([np.asarray(k_rope_b, np.float64), np.asarray(k_nope_h, np.float64)], axis=1)[
        :, :k_nope_h.shape[1] + k_rope_b.shape[1]]


def _default_scale_nope_only(d_nope, d_rope):
    return 1.0 / np.sqrt(d_nope)


def _absorbed_backward_rope_sign(q, c_kv, k_rope, W_UK, W_UV, dout, q_offset=0, causal=True, scale=None):
    # a sign error on the RoPE part of dq
    g = _ORIG_ABS_BWD(q, c_kv, k_rope, W_UK, W_UV, dout, q_offset, causal, scale)
    d_nope = W_UK.shape[1] // q.shape[2]
    g["dq"][..., d_nope:] *= -1.0
    return g


def _absorbed_backward_rope_key_unscaled(q, c_kv, k_rope, W_UK, W_UV, dout, q_offset=0, causal=True, scale=None):
    # forgets the softmax scale on the RoPE-key gradient
    g = _ORIG_ABS_BWD(q, c_kv, k_rope, W_UK, W_UV, dout, q_offset, causal, scale)
    s = scale if scale is not None else O.default_scale(W_UK.shape[1] // q.shape[2], q.shape[3] - W_UK.shape[1] // q.shape[2])
    g["dk_rope"] = g["dk_rope"] / s
    return g


_ORIG_ABS_BWD = O.absorbed_backward


_ORIG_BWD = O.attention_head_backward


def _pins_pass():
    """Run the quick pins; return False as soon as one fails."""
    checks = [
        lambda: test_brute_force_attention(True, 4),
        lambda: test_finite_differences_every_input(True, 3),
        lambda: test_torch_autograd_float64(),
        lambda: test_hand_worked_two_token_example(),
        lambda: test_hand_worked_example_at_the_default_scale(),
        lambda: test_absorbed_backward_finite_differences(True, 3),
    ]
    for c in checks:
        try:
            c()
        except AssertionError:
            return False
    return True


@pytest.mark.parametrize("target,mutant", [
    ("visible_mask", _mask_off_by_one),
    ("reconstruct_head", _reconstruct_head_swapped),
    ("attention_head_backward", _attention_backward_no_scale_dq),
    ("attention_head_backward", _attention_backward_sign),
    ("head_key", _head_key_transposed_rope),
    ("default_scale", _default_scale_nope_only),
    ("absorbed_backward", _absorbed_backward_rope_sign),
    ("absorbed_backward", _absorbed_backward_rope_key_unscaled),
])
def test_planted_mistakes_are_caught(monkeypatch, target, mutant):
    assert _pins_pass()
    monkeypatch.setattr(O, target, mutant)
    assert not _pins_pass(), f"no pin caught the planted mistake in {target}"


# --------------------------------------------------------------------------- multi-process helper
def test_head_parallel_oracle_helper_matches_the_oracle():
    """The helper the full-size GPU tests use (heads dealt to spawned workers, each
    calling the per-head oracle) returns the oracle's own results."""
    import oracle_heads
    p = small(B=2, Sq=6, S=11, n_h=5, q_offset=5)
    x = make_inputs(p, seed=31)
    got = oracle_heads.full_backward(p, x, workers=2)
    xs = inputs64(p, seed=31)
    out, lse = run_fwd(p, xs)
    ref = run_bwd(p, xs)
    ref.update(out=out, lse=lse)
    for k, r in ref.items():
        np.testing.assert_allclose(got[k], r, rtol=1e-12, atol=1e-14, err_msg=k)


# --------------------------------------------------------------------------- random tiny shapes
def draw_tiny(c):
    """Seeded random tiny problem c (fp64 inputs): batch, heads and every width drawn,
    d_rope = 0 included; causal or not; one or two query segments; the default or an
    explicit scale."""
    rng = np.random.default_rng(4000 + c)
    d_rope = int(rng.choice([0, 1, 3]))
    causal = bool(rng.random() < 0.7)
    S = int(rng.integers(2, 12))
    two = bool(rng.random() < 0.4) and S >= 3
    if two:
        n0, n1 = int(rng.integers(1, 4)), int(rng.integers(1, 4))
        Sq = n0 + n1
        off0 = int(rng.integers(0, S - n0 + 1)) if causal else 0
        off1 = int(rng.integers(0, S - n1 + 1)) if causal else 0
        seg = dict(q_split=n0, q_offset2=off1)
    else:
        Sq = int(rng.integers(1, S + 1)) if causal else int(rng.integers(1, 6))
        off0 = int(rng.integers(0, S - Sq + 1)) if causal else 0
        seg = {}
    p = Problem(B=int(rng.integers(1, 3)), Sq=Sq, S=S, n_h=int(rng.integers(1, 4)), d_c=int(rng.integers(1, 6)),
                d_nope=int(rng.integers(1, 5)), d_rope=d_rope, d_v=int(rng.integers(1, 5)), q_offset=off0,
                causal=causal, dtype="f32", **seg)
    scale = float(rng.uniform(0.2, 1.5)) if rng.random() < 0.5 else None
    return p, scale


def positions(p):
    """Absolute position of each local query row: rows [0, q_split) at q_offset + i,
    rows [q_split, Sq) at q_offset2 + (i - q_split)."""
    return [p.q_offset + i if (p.q_split == 0 or i < p.q_split) else p.q_offset2 + i - p.q_split
            for i in range(p.Sq)]


def brute_force_forward_at(p, x, scale, pos):
    """brute_force_forward with each query row at an explicit position."""
    out = np.zeros((p.B, p.Sq, p.n_h, p.d_v))
    lse = np.zeros((p.B, p.n_h, p.Sq))
    for b in range(p.B):
        for h in range(p.n_h):
            K = [[sum(x["c_kv"][b, j, c] * x["W_UK"][c, h * p.d_nope + d] for c in range(p.d_c))
                  for d in range(p.d_nope)] + [x["k_rope"][b, j, d] for d in range(p.d_rope)] for j in range(p.S)]
            V = [[sum(x["c_kv"][b, j, c] * x["W_UV"][c, h * p.d_v + d] for c in range(p.d_c)) for d in range(p.d_v)]
                 for j in range(p.S)]
            for i in range(p.Sq):
                keys = range(0, (pos[i] if p.causal else p.S - 1) + 1)
                s = {j: scale * sum(x["q"][b, i, h, d] * K[j][d] for d in range(p.d_qk)) for j in keys}
                m = max(s.values())
                z = sum(math.exp(s[j] - m) for j in keys)
                lse[b, h, i] = m + math.log(z)
                for d in range(p.d_v):
                    out[b, i, h, d] = sum(math.exp(s[j] - m) / z * V[j][d] for j in keys)
    return out, lse


@pytest.mark.parametrize("c", range(12))
def test_random_tiny_shapes_brute_force_and_finite_differences(c):
    """The oracle's forward against the scalar-loop brute force, and its backward
    against central differences of <dout, out> along random directions, on random
    tiny shapes (two-segment shards and d_rope = 0 among them)."""
    p, scale = draw_tiny(c)
    x = inputs64(p, seed=300 + c)
    sc = scale if scale is not None else 1.0 / math.sqrt(p.d_nope + p.d_rope)
    out, lse = oracle.mla_forward(x["q"], x["c_kv"], x["k_rope"], x["W_UK"], x["W_UV"], p.q_offset, p.causal, scale,
                                  p.q_split, p.q_offset2)
    out_bf, lse_bf = brute_force_forward_at(p, x, sc, positions(p))
    np.testing.assert_allclose(out, out_bf, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(lse, lse_bf, rtol=1e-11, atol=1e-12)

    def f(xx):
        o, _ = oracle.mla_forward(xx["q"], xx["c_kv"], xx["k_rope"], xx["W_UK"], xx["W_UV"], p.q_offset, p.causal,
                                  scale, p.q_split, p.q_offset2)
        return float((o * xx["dout"]).sum())

    g = oracle.mla_backward(x["q"], x["c_kv"], x["k_rope"], x["W_UK"], x["W_UV"], x["dout"], p.q_offset, p.causal,
                            scale, p.q_split, p.q_offset2)
    grads = {"q": g["dq"], "c_kv": g["dc_kv"], "k_rope": g["dk_rope"], "W_UK": g["dW_UK"], "W_UV": g["dW_UV"]}
    rng = np.random.default_rng(50 + c)
    h = 1e-6
    for name, grad in grads.items():
        assert grad.shape == x[name].shape, name
        if grad.size == 0:
            continue
        direction = rng.standard_normal(x[name].shape)
        xp, xm = dict(x), dict(x)
        xp[name] = x[name] + h * direction
        xm[name] = x[name] - h * direction
        fd = (f(xp) - f(xm)) / (2 * h)
        an = float((grad * direction).sum())
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (c, name, fd, an)
