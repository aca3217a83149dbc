"""Seeded random shapes through the tensor-core path, each against the fp64 oracle
at the bf16 tolerance (2e-2 * max|oracle| per output tensor).

The draw covers what the hand-picked cases cover one at a time, in combination:
batch 1 or 2; 1 to 9 heads (the dK/dV kernel's groups of 1, 2 and 4 heads
per CTA, and several groups of 4); ragged query and latent lengths (partial 64-
and 128-row tiles); causal shards at random offsets, non-causal calls, and
two-segment shards; the default softmax scale and explicit ones. The shapes come from a fixed seed, so every run
checks the same cases, and the inputs of case c are drawn with seed 500 + c."""
import numpy as np
import pytest

from mla_attention_sequence_gb300.synth import make_inputs
from test_parity_gpu import TOL, assert_close, run_gpu, run_oracle, small

N_CASES = 48


def draw_case(c: int):
    """Case c of the fixed draw: (problem, softmax scale or None)."""
    rng = np.random.default_rng(9000 + c)
    B = int(rng.integers(1, 3))
    n_h = int(rng.integers(1, 10))
    causal = bool(rng.random() < 0.75)
    scale = float(rng.uniform(0.04, 0.12)) if rng.random() < 0.25 else None
    if rng.random() < 0.3:
        # two segments: rows [0, q_split) at q_offset, the rest at q_offset2
        q_split = 128 * int(rng.integers(1, 3))
        n1 = int(rng.integers(1, 200))
        S = int(rng.integers(q_split + n1, 1000))
        if causal:
            q_offset = int(rng.integers(0, S - q_split + 1))
            q_offset2 = int(rng.integers(0, S - n1 + 1))
        else:
            q_offset, q_offset2 = 0, 0
        return small(B=B, n_h=n_h, Sq=q_split + n1, S=S, q_offset=q_offset, causal=causal, q_split=q_split,
                     q_offset2=q_offset2), scale
    S = int(rng.integers(1, 900))
    if causal:
        Sq = int(rng.integers(1, S + 1))
        q_offset = int(rng.integers(0, S - Sq + 1))
    else:
        Sq = int(rng.integers(1, 400))
        q_offset = 0
    return small(B=B, n_h=n_h, Sq=Sq, S=S, q_offset=q_offset, causal=causal), scale


def test_draw_spans_the_cases_it_claims():
    """The fixed draw holds every head-group size, both batch sizes, causal and
    non-causal calls, two-segment shards, explicit scales and ragged tiles."""
    cases = [draw_case(c) for c in range(N_CASES)]
    ps = [p for p, _ in cases]
    assert {p.n_h % 4 == 0 for p in ps} == {True, False} and any(p.n_h == 8 for p in ps)
    assert {p.n_h % 2 for p in ps} == {0, 1}
    assert {p.B for p in ps} == {1, 2}
    assert {p.causal for p in ps} == {True, False}
    assert any(p.q_split > 0 for p in ps)
    assert any(s is not None for _, s in cases)
    assert any(p.Sq % 64 for p in ps) and any(p.S % 128 for p in ps)


@pytest.fixture(scope="module")
def built():
    from mla_attention_sequence_gb300 import build, laga
    build.build()
    laga.lib()


@pytest.mark.gpu
@pytest.mark.parametrize("c", range(N_CASES))
def test_random_shape_matches_oracle(built, c):
    p, scale = draw_case(c)
    x = make_inputs(p, seed=500 + c)
    assert_close(run_gpu(p, x, scale=scale), run_oracle(p, x, scale=scale), TOL["bf16"], tag=f"case {c}: {p}")


N_SIMT = 16


def draw_simt_case(c: int):
    """Case c of the fp32 draw for the CUDA-core path (any widths): random head
    widths, d_rope = 0 included, at the fp32 tolerance (1e-4 * max|oracle|)."""
    from mla_attention_sequence_gb300.configs import Problem
    rng = np.random.default_rng(7000 + c)
    d_c = int(rng.choice([16, 24, 64]))
    d_nope = int(rng.choice([8, 16, 32]))
    d_rope = int(rng.choice([0, 4, 16]))
    d_v = int(rng.choice([8, 12, 32]))
    B, n_h = int(rng.integers(1, 3)), int(rng.integers(1, 5))
    causal = bool(rng.random() < 0.75)
    S = int(rng.integers(1, 60))
    Sq = int(rng.integers(1, S + 1)) if causal else int(rng.integers(1, 40))
    q_offset = int(rng.integers(0, S - Sq + 1)) if causal else 0
    return Problem(B=B, Sq=Sq, S=S, n_h=n_h, d_c=d_c, d_nope=d_nope, d_rope=d_rope, d_v=d_v, q_offset=q_offset,
                   causal=causal, dtype="f32")


def test_simt_draw_spans_zero_rope_and_both_masks():
    ps = [draw_simt_case(c) for c in range(N_SIMT)]
    assert any(p.d_rope == 0 for p in ps) and any(p.d_rope > 0 for p in ps)
    assert {p.causal for p in ps} == {True, False}


@pytest.mark.gpu
@pytest.mark.parametrize("c", range(N_SIMT))
def test_random_simt_shape_matches_oracle(built, c):
    p = draw_simt_case(c)
    x = make_inputs(p, seed=800 + c)
    assert_close(run_gpu(p, x), run_oracle(p, x), TOL["f32"], tag=f"simt case {c}: {p}")


# ------------------------------------------------------------------ other entry points, same draw
N_ABSORBED = 12


@pytest.mark.gpu
@pytest.mark.parametrize("c", range(N_ABSORBED))
def test_random_absorbed_forward_matches_oracle(built, c):
    """laga_mla_absorbed_fwd on the draw's single-segment shapes against the oracle's
    absorbed form (which equals the explicit form, I2)."""
    import oracle
    from mla_attention_sequence_gb300 import laga
    from test_parity_gpu import dev, to_dev
    p, scale = draw_case(c)
    if p.q_split:
        p = p.with_(q_split=0, q_offset2=0, Sq=min(p.Sq, p.S - p.q_offset) if p.causal else p.Sq)
    x = make_inputs(p, seed=600 + c, with_dout=False)
    t = to_dev(x, p)
    out, lse = laga.absorbed_fwd(t["q"], t["c_kv"], t["k_rope"], t["W_UK"], t["W_UV"], p.q_offset, p.causal, scale)
    laga.check(dev())
    x64 = {k: v.astype(np.float64) for k, v in x.items()}
    ro, rl = oracle.absorbed_forward(x64["q"], x64["c_kv"], x64["k_rope"], x64["W_UK"], x64["W_UV"], p.q_offset,
                                     p.causal, scale)
    assert_close({"out": out, "lse": lse}, {"out": ro, "lse": rl}, TOL["bf16"], tag=f"absorbed case {c}: {p}")


N_REUSE = 8


def visible_rows(p) -> int:
    """Latent rows some query of the shard sees, rounded up to the 128-row tile."""
    if not p.causal:
        last = p.S
    else:
        last = max(off + n for _, n, off in p.segments())
    return -(-last // 128) * 128


@pytest.mark.gpu
@pytest.mark.parametrize("c", range(N_REUSE))
def test_random_reuse_and_prebuilt_paths_are_bitwise(built, c):
    """On the draw's shapes: the backward reading the forward's K/V from the shared
    workspace (LAGA_FLAG_REUSE_KV) equals the backward that rebuilds them, and a
    forward over K/V rebuilt by laga_mla_reconstruct_rows in random 128-row ranges,
    in random order, the last one possibly past the visible prefix
    (LAGA_FLAG_KV_PREBUILT), equals the plain forward, bit for bit."""
    import torch
    from mla_attention_sequence_gb300 import laga
    from test_parity_gpu import dev, to_dev
    p, scale = draw_case(c)
    x = make_inputs(p, seed=700 + c)
    t = to_dev(x, p)
    args = (t["q"], t["c_kv"], t["k_rope"], t["W_UK"], t["W_UV"])
    seg = dict(q_split=p.q_split, q_offset2=p.q_offset2)
    ws = torch.empty(max(laga.fwd_workspace_bytes(p), laga.bwd_workspace_bytes(p)), dtype=torch.uint8, device=dev())
    out, lse = laga.fwd(*args, p.q_offset, p.causal, scale, workspace=ws, **seg)
    g_reuse = laga.bwd(*args, out, lse, t["dout"], p.q_offset, p.causal, scale, workspace=ws, reuse_kv=True, **seg)
    g_plain = laga.bwd(*args, out, lse, t["dout"], p.q_offset, p.causal, scale, **seg)
    # K/V rebuilt range by range into a fresh workspace, then the prebuilt forward
    rng = np.random.default_rng(100 + c)
    n_tiles = visible_rows(p) // 128
    cuts = sorted(set(int(v) for v in rng.integers(1, n_tiles, size=min(3, max(0, n_tiles - 1))))) if n_tiles > 1 else []
    bounds = [0] + cuts + [n_tiles]
    ranges = [(128 * a, 128 * (b - a)) for a, b in zip(bounds[:-1], bounds[1:])]
    if rng.random() < 0.5:  # the last range may run past the visible prefix
        ranges[-1] = (ranges[-1][0], ranges[-1][1] + int(rng.integers(1, 300)))
    order = rng.permutation(len(ranges))
    ws2 = torch.zeros(laga.fwd_workspace_bytes(p), dtype=torch.uint8, device=dev())
    for i in order:
        laga.reconstruct_rows(*args, ranges[i][0], ranges[i][1], ws2, p.q_offset, p.causal, **seg)
    out2, lse2 = laga.fwd(*args, p.q_offset, p.causal, scale, workspace=ws2, kv_prebuilt=True, **seg)
    laga.check(dev())
    for k in g_plain:
        assert torch.equal(g_reuse[k], g_plain[k]), f"case {c}: {k} differs with REUSE_KV"
    assert torch.equal(out2, out) and torch.equal(lse2, lse), f"case {c}: prebuilt forward differs ({ranges})"


N_SIMT_BF16 = 8


@pytest.mark.gpu
@pytest.mark.parametrize("c", range(N_SIMT_BF16))
def test_random_simt_bf16_shape_matches_oracle(built, c):
    """The CUDA-core path with bf16 storage (any widths) at the bf16 tolerance."""
    p = draw_simt_case(100 + c).with_(dtype="bf16")
    x = make_inputs(p, seed=900 + c)
    assert_close(run_gpu(p, x), run_oracle(p, x), TOL["bf16"], tag=f"simt bf16 case {c}: {p}")
