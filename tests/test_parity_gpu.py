"""GPU path vs the fp64 oracle, through the C ABI, on the same seeded inputs.

Tolerances (per output tensor): max|gpu - oracle| <= 1e-4 * max|oracle| for fp32
problems and <= 2e-2 * max|oracle| for bf16 problems.
"""
import numpy as np
import pytest
import torch

import oracle
from mla_attention_sequence_gb300 import laga
from mla_attention_sequence_gb300.configs import DSV3_LAST_RANK, MID_BF16, TINY_F32, Problem
from mla_attention_sequence_gb300.synth import make_inputs

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}
# A gradient that is exactly zero in exact arithmetic (one visible key: p = 1, so
# ds = dp - D = 0) comes out at the rounding level; it is compared absolutely.
ZERO_FLOOR = 1e-5
KEYS = ("out", "lse", "dq", "dc_kv", "dk_rope", "dW_UK", "dW_UV")


@pytest.fixture(scope="module", autouse=True)
def built():
    from mla_attention_sequence_gb300 import build
    build.build()
    laga.lib()


def dev():
    return torch.device("cuda", 0)


def to_dev(x, p):
    dt = torch.float32 if p.dtype == "f32" else torch.bfloat16
    return {k: torch.from_numpy(v).to(dev()).to(dt).contiguous() for k, v in x.items()}


def np64(t):
    return t.float().cpu().numpy().astype(np.float64)


def run_gpu(p, x, variant="auto", backward=True, scale=None):
    t = to_dev(x, p)
    out, lse = laga.fwd(t["q"], t["c_kv"], t["k_rope"], t["W_UK"], t["W_UV"], p.q_offset, p.causal, scale, variant,
                        q_split=p.q_split, q_offset2=p.q_offset2)
    res = {"out": out, "lse": lse}
    if backward:
        res.update(laga.bwd(t["q"], t["c_kv"], t["k_rope"], t["W_UK"], t["W_UV"], out, lse, t["dout"], p.q_offset,
                            p.causal, scale, "auto" if variant == "fused_recon" else variant, q_split=p.q_split,
                            q_offset2=p.q_offset2))
    laga.check(dev())
    return res


def run_oracle(p, x, backward=True, scale=None):
    x64 = {k: v.astype(np.float64) for k, v in x.items()}
    out, lse = oracle.mla_forward(x64["q"], x64["c_kv"], x64["k_rope"], x64["W_UK"], x64["W_UV"], p.q_offset,
                                  p.causal, scale, p.q_split, p.q_offset2)
    ref = {"out": out, "lse": lse}
    if backward:
        ref.update(oracle.mla_backward(x64["q"], x64["c_kv"], x64["k_rope"], x64["W_UK"], x64["W_UV"], x64["dout"],
                                       p.q_offset, p.causal, scale, p.q_split, p.q_offset2))
    return ref


def assert_close(got, ref, tol, keys=None, tag=""):
    bad = []
    for k in keys or ref.keys():
        a = np64(got[k]) if torch.is_tensor(got[k]) else got[k]
        r = ref[k]
        assert a.shape == r.shape, (k, a.shape, r.shape)
        if r.size == 0:  # e.g. dk_rope without a RoPE part (d_rope = 0): the shape is all there is
            continue
        assert np.isfinite(a).all(), f"{tag} {k}: non-finite values"
        err = np.abs(a - r).max()
        bound = tol * np.abs(r).max() if np.abs(r).max() > 0 else ZERO_FLOOR
        if not err <= bound:
            bad.append(f"{k}: max|err|={err:.3e} > {bound:.3e}")
    assert not bad, f"{tag} " + "; ".join(bad)


def small(**kw):
    base = dict(B=1, Sq=256, S=256, n_h=2, d_c=512, d_nope=128, d_rope=64, d_v=128, q_offset=0, causal=True,
                dtype="bf16")
    base.update(kw)
    return Problem(**base)


# ------------------------------------------------------------------ CUDA-core path
def test_tiny_f32_forward_backward():
    p = TINY_F32
    x = make_inputs(p, seed=0)
    assert_close(run_gpu(p, x), run_oracle(p, x), TOL["f32"], tag="tiny f32")


@pytest.mark.parametrize("kw", [dict(q_offset=5, Sq=11, S=23, causal=True), dict(q_offset=0, Sq=9, S=14, causal=False)])
def test_simt_f32_ragged(kw):
    p = Problem(B=2, n_h=3, d_c=24, d_nope=8, d_rope=4, d_v=12, dtype="f32", **kw)
    x = make_inputs(p, seed=1)
    assert_close(run_gpu(p, x), run_oracle(p, x), TOL["f32"], tag="simt f32 ragged")


def test_simt_bf16_on_request():
    p = small(Sq=70, S=150, q_offset=80, n_h=2)
    x = make_inputs(p, seed=2)
    assert_close(run_gpu(p, x, "simt"), run_oracle(p, x), TOL["bf16"], tag="simt bf16")


# ------------------------------------------------------------------ tensor-core path
@pytest.mark.parametrize("n_h", [4, 3])
def test_reconstruct_tensor_cores(n_h):
    p = small(B=2, S=300, Sq=1, n_h=n_h)
    x = make_inputs(p, seed=3, with_dout=False)
    t = to_dev(x, p)
    kn, v = laga.reconstruct(t["c_kv"], t["W_UK"], t["W_UV"], p.n_h)
    laga.check(dev())
    rk, rv = oracle.reconstruct(x["c_kv"].astype(np.float64), x["W_UK"].astype(np.float64),
                                x["W_UV"].astype(np.float64), p.n_h)
    # K/V come out of one bf16 rounding of an fp32 accumulation: 2^-8 relative
    for a, r in ((kn, rk), (v, rv)):
        err = np.abs(np64(a) - r)
        assert (err <= 2.0 ** -8 * np.abs(r) + 1e-3 * np.abs(r).max()).all()


TC_CASES = {
    "aligned": small(),
    "ragged_offset": small(B=2, n_h=3, Sq=200, S=520, q_offset=300),
    "noncausal_ragged": small(n_h=2, Sq=77, S=333, causal=False),
    "single_query_first": small(Sq=1, S=1, q_offset=0),
    "single_query_last": small(Sq=1, S=701, q_offset=700),
    "multi_tile": small(B=1, n_h=2, Sq=384, S=1000, q_offset=600),
    # two-segment (zigzag) shards: rows from q_split on start at q_offset2
    "two_segments": small(B=1, n_h=2, Sq=256, S=1024, q_offset=128, q_split=128, q_offset2=768),
    "two_segments_ragged": small(B=2, n_h=3, Sq=300, S=900, q_offset=0, q_split=128, q_offset2=600),
    "two_segments_noncausal": small(n_h=2, Sq=256, S=500, causal=False, q_split=128, q_offset2=0),
}


@pytest.mark.parametrize("variant", ["materialize", "fused_recon"])
@pytest.mark.parametrize("name", list(TC_CASES))
def test_tensor_core_forward(name, variant):
    p = TC_CASES[name]
    x = make_inputs(p, seed=10)
    if p.q_split and variant == "fused_recon":  # two segments: materialize path only
        with pytest.raises(laga.LagaError) as err:
            run_gpu(p, x, variant, backward=False)
        assert err.value.status == 2
        return
    assert_close(run_gpu(p, x, variant, backward=False), run_oracle(p, x, backward=False), TOL["bf16"],
                 tag=f"{name} {variant}")


@pytest.mark.parametrize("name", list(TC_CASES))
def test_tensor_core_backward(name):
    p = TC_CASES[name]
    x = make_inputs(p, seed=11)
    assert_close(run_gpu(p, x, "materialize"), run_oracle(p, x), TOL["bf16"], tag=name)


# ------------------------------------------------------------------ explicit softmax scale
# Every other case takes the default scale (softmax_scale <= 0). These pass one
# explicitly: it feeds the exponent scale of all three attention kernels and the
# final dq / dK scaling, so a wrong or ignored value shows in every output.
SCALED_CASES = {
    "tc_ragged_causal": (small(B=2, n_h=3, Sq=200, S=520, q_offset=300), "materialize"),
    "tc_two_segments": (small(B=2, n_h=3, Sq=300, S=900, q_offset=0, q_split=128, q_offset2=600), "materialize"),
    "tc_noncausal": (small(n_h=2, Sq=77, S=333, causal=False), "materialize"),
    "simt_f32": (Problem(B=2, n_h=3, d_c=24, d_nope=8, d_rope=4, d_v=12, dtype="f32", q_offset=5, Sq=11, S=23,
                         causal=True), "simt"),
}


@pytest.mark.parametrize("scale", [0.05, 0.2])
@pytest.mark.parametrize("name", list(SCALED_CASES))
def test_explicit_softmax_scale(name, scale):
    p, variant = SCALED_CASES[name]
    x = make_inputs(p, seed=16)
    assert_close(run_gpu(p, x, variant, scale=scale), run_oracle(p, x, scale=scale), TOL[p.dtype],
                 tag=f"{name} scale={scale}")


def test_explicit_softmax_scale_fused_forward():
    p = small(B=2, n_h=3, Sq=200, S=520, q_offset=300)
    x = make_inputs(p, seed=17)
    assert_close(run_gpu(p, x, "fused_recon", backward=False, scale=0.2),
                 run_oracle(p, x, backward=False, scale=0.2), TOL["bf16"], tag="fused scale=0.2")


def test_explicit_scale_equal_to_default_is_bitwise_default():
    """softmax_scale = 1/sqrt(192) passed explicitly takes the same arithmetic as the default."""
    p = small(B=1, n_h=2, Sq=200, S=520, q_offset=300)
    x = make_inputs(p, seed=18)
    a = run_gpu(p, x)
    b = run_gpu(p, x, scale=float(np.float32(1.0) / np.sqrt(np.float32(192.0))))
    for k in KEYS:
        assert torch.equal(a[k], b[k]), k


# ------------------------------------------------------------------ all 128 heads, element by element
def test_full_head_count_shard_every_output():
    """n_h = 128, the DeepSeek-V3 head count, on a shard small enough for the whole
    oracle: every output element by element, including the two cross-head
    reductions (dc_kv's contraction over n_h * 256 = 32768 and dk_rope's sum over
    128 heads)."""
    p = small(B=1, n_h=128, Sq=512, S=2048, q_offset=1536)
    x = make_inputs(p, seed=19)
    assert_close(run_gpu(p, x), run_oracle(p, x), TOL["bf16"], tag="n_h=128 shard")


def test_dsv3_last_rank_full_oracle_every_output():
    """The DeepSeek-V3 SP=8 last-rank shard (the benchmark's launch configuration):
    all seven outputs element by element against the full 128-head fp64 oracle.
    The oracle's heads are split over worker processes; each worker runs the
    per-head oracle on its heads and adds up their dc_kv / dk_rope contributions."""
    import oracle_heads
    p = DSV3_LAST_RANK
    x = make_inputs(p, seed=2007)
    ref = oracle_heads.full_backward(p, x)
    got = run_gpu(p, x)
    assert_close(got, ref, TOL["bf16"], tag="dsv3 last rank, full oracle")


def test_mid_config_full_parity():
    p = MID_BF16
    x = make_inputs(p, seed=1000)
    assert_close(run_gpu(p, x), run_oracle(p, x), TOL["bf16"], tag="mid")


def test_lse_and_out_of_padded_rows_are_untouched():
    """Rows beyond Sq are never written; the tensors keep what the caller put there."""
    p = small(Sq=130, S=400, q_offset=200)
    x = make_inputs(p, seed=12)
    t = to_dev(x, p)
    out = torch.full((p.B, p.Sq + 1, p.n_h, p.d_v), 7.0, dtype=torch.bfloat16, device=dev())
    lse = torch.full((p.B, p.n_h, p.Sq), 7.0, device=dev())
    o, l = laga.fwd(t["q"], t["c_kv"], t["k_rope"], t["W_UK"], t["W_UV"], p.q_offset, True, out=out[:, :p.Sq],
                    lse=lse)
    torch.cuda.synchronize()
    assert (out[:, p.Sq:].float() == 7.0).all()


# ------------------------------------------------------------------ full size, sampled
def test_dsv3_last_rank_sampled_heads_and_identities():
    """The DeepSeek-V3 SP=8 last-rank shard at full size (the benchmark's launch
    configuration): selected heads against the per-head oracle, and the
    gradient identities that tie dc_kv and dk_rope to the other outputs."""
    p = DSV3_LAST_RANK
    x = make_inputs(p, seed=2007)
    t = to_dev(x, p)
    out, lse = laga.fwd(t["q"], t["c_kv"], t["k_rope"], t["W_UK"], t["W_UV"], p.q_offset, True)
    g = laga.bwd(t["q"], t["c_kv"], t["k_rope"], t["W_UK"], t["W_UV"], out, lse, t["dout"], p.q_offset, True)
    laga.check(dev())
    x64 = {k: v.astype(np.float64) for k, v in x.items()}
    for h in (0, 77, 127):
        ref = oracle.mla_backward_head(x64["q"], x64["c_kv"], x64["k_rope"], x64["W_UK"], x64["W_UV"], x64["dout"],
                                       0, h, p.q_offset, True)
        got = {"out": out[0, :, h], "lse": lse[0, h], "dq": g["dq"][0, :, h],
               "dW_UK": g["dW_UK"][:, h * 128:(h + 1) * 128], "dW_UV": g["dW_UV"][:, h * 128:(h + 1) * 128]}
        want = {"out": ref["out_h"], "lse": ref["lse_h"], "dq": ref["dq_h"], "dW_UK": ref["dW_UK_h"],
                "dW_UV": ref["dW_UV_h"]}
        assert_close(got, want, TOL["bf16"], tag=f"dsv3 head {h}")

    def inner(a, b):
        return float((np64(a) * (b if isinstance(b, np.ndarray) else np64(b))).sum())

    # <dW_UV, W_UV> = <dout, out>;  <dW_UK, W_UK> + <dk_rope, k_rope> = <dq, q>;
    # <dc_kv, c_kv> = <dW_UK, W_UK> + <dW_UV, W_UV>
    a_uv = inner(g["dW_UV"], x64["W_UV"])
    a_uk = inner(g["dW_UK"], x64["W_UK"])
    a_r = inner(g["dk_rope"], x64["k_rope"])
    a_q = inner(g["dq"], x64["q"])
    a_o = inner(t["dout"], out)
    a_c = inner(g["dc_kv"], x64["c_kv"])
    scale_ = max(abs(a_q), abs(a_o), 1.0)
    assert abs(a_uv - a_o) <= 2e-2 * scale_
    assert abs(a_uk + a_r - a_q) <= 2e-2 * scale_
    assert abs(a_c - (a_uk + a_uv)) <= 2e-2 * scale_


@pytest.mark.parametrize("r", range(8))
def test_dsv3_every_rank_shard_sampled(r):
    """Every SP=8 rank shard of the DeepSeek-V3 layer (q_offset = 2048 r), forward and
    backward at full size: one head per rank against the per-head oracle, plus
    the gradient identities over all heads."""
    from mla_attention_sequence_gb300.configs import dsv3_rank
    p = dsv3_rank(r)
    x = make_inputs(p, seed=3000 + r)
    t = to_dev(x, p)
    out, lse = laga.fwd(t["q"], t["c_kv"], t["k_rope"], t["W_UK"], t["W_UV"], p.q_offset, True)
    g = laga.bwd(t["q"], t["c_kv"], t["k_rope"], t["W_UK"], t["W_UV"], out, lse, t["dout"], p.q_offset, True)
    laga.check(dev())
    x64 = {k: v.astype(np.float64) for k, v in x.items()}
    h = (37 * r + 5) % p.n_h
    ref = oracle.mla_backward_head(x64["q"], x64["c_kv"], x64["k_rope"], x64["W_UK"], x64["W_UV"], x64["dout"],
                                   0, h, p.q_offset, True)
    got = {"out": out[0, :, h], "lse": lse[0, h], "dq": g["dq"][0, :, h],
           "dW_UK": g["dW_UK"][:, h * 128:(h + 1) * 128], "dW_UV": g["dW_UV"][:, h * 128:(h + 1) * 128]}
    want = {"out": ref["out_h"], "lse": ref["lse_h"], "dq": ref["dq_h"], "dW_UK": ref["dW_UK_h"],
            "dW_UV": ref["dW_UV_h"]}
    assert_close(got, want, TOL["bf16"], tag=f"rank {r} head {h}")
    # latent rows beyond the shard's causal prefix get no gradient
    tail = p.q_offset + p.Sq
    assert not g["dc_kv"][:, tail:].any() and not g["dk_rope"][:, tail:].any()

    def inner(a, b):
        return float((np64(a) * b).sum())
    a_q = inner(g["dq"], x64["q"])
    a_o = inner(out, x64["dout"])
    scale_ = max(abs(a_q), abs(a_o), 1.0)
    assert abs(inner(g["dW_UV"], x64["W_UV"]) - a_o) <= 2e-2 * scale_
    assert abs(inner(g["dW_UK"], x64["W_UK"]) + inner(g["dk_rope"], x64["k_rope"]) - a_q) <= 2e-2 * scale_


@pytest.mark.parametrize("r", [0, 7])
def test_dsv3_zigzag_shard_sampled(r):
    """Zigzag SP=8 shards of the DeepSeek-V3 layer (rank r holds sequence chunks r and
    15 - r of 1024 rows), forward and backward at full size: one head against the
    per-head oracle with the shard's two-segment positions, plus the gradient
    identities over all heads."""
    from mla_attention_sequence_gb300.configs import dsv3_zigzag_rank
    p = dsv3_zigzag_rank(r)
    x = make_inputs(p, seed=4000 + r)
    t = to_dev(x, p)
    out, lse = laga.fwd(t["q"], t["c_kv"], t["k_rope"], t["W_UK"], t["W_UV"], p.q_offset, True,
                        q_split=p.q_split, q_offset2=p.q_offset2)
    g = laga.bwd(t["q"], t["c_kv"], t["k_rope"], t["W_UK"], t["W_UV"], out, lse, t["dout"], p.q_offset, True,
                 q_split=p.q_split, q_offset2=p.q_offset2)
    laga.check(dev())
    x64 = {k: v.astype(np.float64) for k, v in x.items()}
    h = (29 * r + 3) % p.n_h
    pos = oracle.query_positions(p.Sq, p.q_offset, p.q_split, p.q_offset2)
    ref = oracle.mla_backward_head(x64["q"], x64["c_kv"], x64["k_rope"], x64["W_UK"], x64["W_UV"], x64["dout"],
                                   0, h, pos, True)
    got = {"out": out[0, :, h], "lse": lse[0, h], "dq": g["dq"][0, :, h],
           "dW_UK": g["dW_UK"][:, h * 128:(h + 1) * 128], "dW_UV": g["dW_UV"][:, h * 128:(h + 1) * 128]}
    want = {"out": ref["out_h"], "lse": ref["lse_h"], "dq": ref["dq_h"], "dW_UK": ref["dW_UK_h"],
            "dW_UV": ref["dW_UV_h"]}
    assert_close(got, want, TOL["bf16"], tag=f"zigzag rank {r} head {h}")
    tail = p.skv_eff  # latent rows beyond every query's position get no gradient
    assert not g["dc_kv"][:, tail:].any() and not g["dk_rope"][:, tail:].any()

    def inner(a, b):
        return float((np64(a) * b).sum())
    a_q = inner(g["dq"], x64["q"])
    a_o = inner(out, x64["dout"])
    scale_ = max(abs(a_q), abs(a_o), 1.0)
    assert abs(inner(g["dW_UV"], x64["W_UV"]) - a_o) <= 2e-2 * scale_
    assert abs(inner(g["dW_UK"], x64["W_UK"]) + inner(g["dk_rope"], x64["k_rope"]) - a_q) <= 2e-2 * scale_


@pytest.mark.parametrize("seq,n_h", [(4096, 32), (32768, 32), (8192, 128)])
def test_sweep_shapes_sampled(seq, n_h):
    """Last-rank SP=8 shards of the sweep (sequence length x heads), both forward
    variants and the backward, one head against the per-head oracle."""
    from mla_attention_sequence_gb300.configs import dsv3_rank
    p = dsv3_rank(7, seq=seq, n_h=n_h)
    x = make_inputs(p, seed=seq + n_h)
    t = to_dev(x, p)
    outs = {v: laga.fwd(t["q"], t["c_kv"], t["k_rope"], t["W_UK"], t["W_UV"], p.q_offset, True, None, v)
            for v in ("materialize", "fused_recon")}
    out, lse = outs["materialize"]
    g = laga.bwd(t["q"], t["c_kv"], t["k_rope"], t["W_UK"], t["W_UV"], out, lse, t["dout"], p.q_offset, True)
    laga.check(dev())
    x64 = {k: v.astype(np.float64) for k, v in x.items()}
    h = n_h - 1
    ref = oracle.mla_backward_head(x64["q"], x64["c_kv"], x64["k_rope"], x64["W_UK"], x64["W_UV"], x64["dout"],
                                   0, h, p.q_offset, True)
    for v, (o, l) in outs.items():
        assert_close({"out": o[0, :, h], "lse": l[0, h]}, {"out": ref["out_h"], "lse": ref["lse_h"]}, TOL["bf16"],
                     tag=f"sweep S={seq} n_h={n_h} {v}")
    assert_close({"dq": g["dq"][0, :, h], "dW_UK": g["dW_UK"][:, h * 128:(h + 1) * 128],
                  "dW_UV": g["dW_UV"][:, h * 128:(h + 1) * 128]},
                 {"dq": ref["dq_h"], "dW_UK": ref["dW_UK_h"], "dW_UV": ref["dW_UV_h"]}, TOL["bf16"],
                 tag=f"sweep S={seq} n_h={n_h} backward")


# ------------------------------------------------------------------ SP shards, determinism
def test_sequence_parallel_shards_on_gpu():
    S, sp = 1024, 4
    p1 = small(B=1, n_h=2, Sq=S, S=S, q_offset=0)
    x = make_inputs(p1, seed=13)
    full = run_gpu(p1, x)
    sh = S // sp
    sums = {k: 0.0 for k in ("dc_kv", "dk_rope", "dW_UK", "dW_UV")}
    for r in range(sp):
        pr = p1.with_(Sq=sh, q_offset=r * sh)
        xr = dict(x)
        xr["q"] = np.ascontiguousarray(x["q"][:, r * sh:(r + 1) * sh])
        xr["dout"] = np.ascontiguousarray(x["dout"][:, r * sh:(r + 1) * sh])
        g = run_gpu(pr, xr)
        # same tiles, same order: forward rows are bitwise those of SP=1
        assert torch.equal(g["out"], full["out"][:, r * sh:(r + 1) * sh])
        assert torch.equal(g["lse"], full["lse"][:, :, r * sh:(r + 1) * sh])
        # dq rows come from the same query tiles walking the same key tiles
        assert torch.equal(g["dq"], full["dq"][:, r * sh:(r + 1) * sh])
        for k in sums:
            sums[k] = sums[k] + np64(g[k])
    for k in sums:
        ref = np64(full[k])
        assert np.abs(sums[k] - ref).max() <= 2e-2 * np.abs(ref).max(), k


@pytest.mark.parametrize("variant", ["auto", "simt"])
def test_backward_reusing_forward_kv_matches(variant):
    """LAGA_FLAG_REUSE_KV: a backward that reads the forward's K_nope/V from the
    shared workspace gives bitwise the same gradients as one that rebuilds them."""
    p = small(B=2, n_h=3, Sq=200, S=520, q_offset=300)
    x = make_inputs(p, seed=15)
    t = to_dev(x, p)
    nb = max(laga.fwd_workspace_bytes(p, variant), laga.bwd_workspace_bytes(p, variant))
    ws = torch.empty(nb, dtype=torch.uint8, device=dev())
    out, lse = laga.fwd(t["q"], t["c_kv"], t["k_rope"], t["W_UK"], t["W_UV"], p.q_offset, True, None, variant, ws)
    g1 = laga.bwd(t["q"], t["c_kv"], t["k_rope"], t["W_UK"], t["W_UV"], out, lse, t["dout"], p.q_offset, True,
                  None, variant, ws, reuse_kv=True)
    g1 = {k: v.clone() for k, v in g1.items()}
    g2 = laga.bwd(t["q"], t["c_kv"], t["k_rope"], t["W_UK"], t["W_UV"], out, lse, t["dout"], p.q_offset, True,
                  None, variant)
    laga.check(dev())
    for k in g1:
        assert torch.equal(g1[k], g2[k]), k


def test_fused_reconstruction_matches_materialized_at_full_size():
    """Both forward variants on the DSV3 last-rank shard: same outputs within the
    bf16 tolerance (they round K/V to bf16 at the same point)."""
    p = DSV3_LAST_RANK
    x = make_inputs(p, seed=2008, with_dout=False)
    t = to_dev(x, p)
    oa, la = laga.fwd(t["q"], t["c_kv"], t["k_rope"], t["W_UK"], t["W_UV"], p.q_offset, True, None, "materialize")
    ob, lb = laga.fwd(t["q"], t["c_kv"], t["k_rope"], t["W_UK"], t["W_UV"], p.q_offset, True, None, "fused_recon")
    laga.check(dev())
    assert_close({"out": ob, "lse": lb}, {"out": np64(oa), "lse": np64(la)}, TOL["bf16"], tag="fused vs materialized")


def test_determinism():
    p = small(B=1, n_h=4, Sq=512, S=1024, q_offset=512)
    x = make_inputs(p, seed=14)
    a = run_gpu(p, x)
    b = run_gpu(p, x)
    # no atomics anywhere: every output is produced in a fixed order
    for k in ("out", "lse", "dq", "dc_kv", "dk_rope", "dW_UK", "dW_UV"):
        assert torch.equal(a[k], b[k]), k


# ------------------------------------------------------------------ the absorbed form (comparison path)
ABSORBED_CASES = {
    "aligned": small(n_h=2, Sq=256, S=256),
    "ragged_offset": small(B=2, n_h=3, Sq=200, S=520, q_offset=300),
    "noncausal_ragged": small(n_h=2, Sq=77, S=333, causal=False),
    "single_query_last": small(Sq=1, S=701, q_offset=700),
    "multi_tile": small(B=1, n_h=2, Sq=384, S=1000, q_offset=600),
}


@pytest.mark.parametrize("name", list(ABSORBED_CASES))
def test_absorbed_forward(name):
    """laga_mla_absorbed_fwd (q_lat GEMM, latent-space attention, output GEMM) against
    the oracle's absorbed form, and its out / lse against the explicit form's."""
    p = ABSORBED_CASES[name]
    x = make_inputs(p, seed=20)
    t = to_dev(x, p)
    out, lse = laga.absorbed_fwd(t["q"], t["c_kv"], t["k_rope"], t["W_UK"], t["W_UV"], p.q_offset, p.causal)
    laga.check(dev())
    x64 = {k: v.astype(np.float64) for k, v in x.items()}
    ref_out, ref_lse = oracle.absorbed_forward(x64["q"], x64["c_kv"], x64["k_rope"], x64["W_UK"], x64["W_UV"],
                                               p.q_offset, p.causal)
    assert_close({"out": out, "lse": lse}, {"out": ref_out, "lse": ref_lse}, TOL["bf16"], tag=f"absorbed {name}")


def test_absorbed_forward_dsv3_sampled_heads():
    """The absorbed form on the DeepSeek-V3 SP=8 last-rank shard: sampled heads against
    the per-head oracle (out and lse are the explicit form's)."""
    p = DSV3_LAST_RANK
    x = make_inputs(p, seed=2009, with_dout=False)
    t = to_dev(x, p)
    out, lse = laga.absorbed_fwd(t["q"], t["c_kv"], t["k_rope"], t["W_UK"], t["W_UV"], p.q_offset, True)
    laga.check(dev())
    x64 = {k: v.astype(np.float64) for k, v in x.items()}
    for h in (0, 127):
        ro, rl = oracle.mla_forward_head(x64["q"], x64["c_kv"], x64["k_rope"], x64["W_UK"], x64["W_UV"], 0, h,
                                         p.q_offset, True)
        assert_close({"out": out[0, :, h], "lse": lse[0, h]}, {"out": ro, "lse": rl}, TOL["bf16"],
                     tag=f"absorbed dsv3 head {h}")


def test_absorbed_forward_rejects_two_segments():
    p = TC_CASES["two_segments"]
    assert laga.absorbed_workspace_bytes(p) == 0
    d = laga.make_desc(p)
    L = laga.lib()
    import ctypes
    fake = ctypes.c_void_p(4096)
    assert L.laga_mla_absorbed_fwd(ctypes.byref(d), *([fake] * 8), 1 << 30, None) == 2
