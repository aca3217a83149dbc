"""Host-side checks of the workload shapes (no GPU): the SP=8 shards of the
DeepSeek-V3 layer, contiguous and zigzag, cover every query position of the
sequence exactly once; zigzag shards see equal numbers of (query, key) pairs; the
pair counts match a brute-force count of the causal mask."""
import numpy as np
import pytest

from mla_attention_sequence_gb300.configs import GROUPS, Problem, dsv3_rank, dsv3_zigzag_rank


def positions(p):
    return np.concatenate([np.arange(off, off + n) for _, n, off in p.segments()])


@pytest.mark.parametrize("group", sorted(GROUPS))
def test_shards_cover_the_sequence_once(group):
    shards = GROUPS[group]
    pos = np.sort(np.concatenate([positions(p) for p in shards]))
    np.testing.assert_array_equal(pos, np.arange(shards[0].S))


def test_zigzag_ranks_see_equal_work():
    pairs = {dsv3_zigzag_rank(r).pairs for r in range(8)}
    assert len(pairs) == 1
    assert sum(dsv3_zigzag_rank(r).pairs for r in range(8)) == sum(dsv3_rank(r).pairs for r in range(8))


@pytest.mark.parametrize("p", [
    Problem(B=2, Sq=12, S=40, n_h=1, d_c=1, d_nope=1, d_rope=0, d_v=1, q_offset=7),
    Problem(B=1, Sq=12, S=40, n_h=1, d_c=1, d_nope=1, d_rope=0, d_v=1, q_offset=3, q_split=5, q_offset2=30),
    Problem(B=1, Sq=12, S=40, n_h=1, d_c=1, d_nope=1, d_rope=0, d_v=1, q_offset=3, q_split=5, q_offset2=30,
            causal=False),
])
def test_pair_count_matches_the_mask(p):
    pos = positions(p)
    keys = np.arange(p.S)
    vis = (keys[None, :] <= pos[:, None]) if p.causal else np.ones((p.Sq, p.S), dtype=bool)
    assert p.pairs == p.B * int(vis.sum())
    if p.causal:
        assert p.skv_eff == int(pos.max()) + 1
