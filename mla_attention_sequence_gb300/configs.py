"""Problem shapes for the LAGA MLA attention block.

A ``Problem`` fixes every size of one call: batch ``B``, local query shard
length ``Sq``, gathered latent length ``S`` (= Skv), heads ``n_h``, latent
width ``d_c``, the no-RoPE and RoPE query/key widths ``d_nope`` / ``d_rope``,
value width ``d_v``, the shard's first absolute query position ``q_offset``,
the causal flag and the element type.

The named shapes follow the workloads of "A Training-Memory Regression in MLA
Sequence Parallelism ... LAGA" (weekinpapers page, Abstract): DeepSeek-V3
attention dimensions (n_h=128, seq=16384) with sequence parallelism SP=8,
where each rank holds a contiguous query shard and the full gathered latent.
This module holds data only: no arithmetic of the method.
"""
from __future__ import annotations

from dataclasses import dataclass, replace


@dataclass(frozen=True)
class Problem:
    B: int
    Sq: int
    S: int
    n_h: int
    d_c: int
    d_nope: int
    d_rope: int
    d_v: int
    q_offset: int = 0
    causal: bool = True
    dtype: str = "bf16"  # "bf16" or "f32"
    name: str = ""
    # Two-segment (zigzag) shard: q_split > 0 puts rows [q_split, Sq) at
    # positions q_offset2, q_offset2 + 1, ...; rows [0, q_split) stay at q_offset + i.
    q_split: int = 0
    q_offset2: int = 0

    def segments(self):
        """(first local row, rows, first absolute position) of each query segment."""
        if self.q_split <= 0:
            return [(0, self.Sq, self.q_offset)]
        return [(0, self.q_split, self.q_offset), (self.q_split, self.Sq - self.q_split, self.q_offset2)]

    @property
    def d_qk(self) -> int:
        return self.d_nope + self.d_rope

    @property
    def skv_eff(self) -> int:
        """Latent rows any query of the shard can see."""
        return max(off + n for _, n, off in self.segments()) if self.causal else self.S

    @property
    def pairs(self) -> int:
        """Visible (query, key) pairs summed over the batch."""
        if self.causal:
            return self.B * sum(n * off + n * (n + 1) // 2 for _, n, off in self.segments())
        return self.B * self.Sq * self.S

    def flops_fwd(self) -> int:
        """Algorithmic forward flops: attention (QK^T and PV) plus the K/V
        reconstruction contraction over the visible latent prefix."""
        attn = 2 * self.pairs * self.n_h * (self.d_qk + self.d_v)
        recon = 2 * self.B * self.skv_eff * self.d_c * self.n_h * (self.d_nope + self.d_v)
        return attn + recon

    def flops_bwd(self) -> int:
        """Algorithmic backward flops: twice the forward (no recompute)."""
        return 2 * self.flops_fwd()

    def flops_step(self) -> int:
        return self.flops_fwd() + self.flops_bwd()

    def flops_step_fa(self) -> int:
        """The step under the FlashAttention convention: the algorithmic flops plus
        the backward's recomputation of the scores, 2 * pairs * n_h * d_qk."""
        return self.flops_step() + 2 * self.pairs * self.n_h * self.d_qk

    def with_(self, **kw) -> "Problem":
        return replace(self, **kw)


TINY_F32 = Problem(B=1, Sq=256, S=256, n_h=4, d_c=64, d_nope=32, d_rope=16, d_v=32,
                   q_offset=0, causal=True, dtype="f32", name="tiny_f32")

MID_BF16 = Problem(B=2, Sq=4096, S=4096, n_h=16, d_c=512, d_nope=128, d_rope=64, d_v=128,
                   q_offset=0, causal=True, dtype="bf16", name="mid_bf16")


def dsv3_rank(r: int, sp: int = 8, seq: int = 16384, n_h: int = 128) -> Problem:
    """One contiguous SP shard of a DeepSeek-V3-dimension MLA layer."""
    sq = seq // sp
    return Problem(B=1, Sq=sq, S=seq, n_h=n_h, d_c=512, d_nope=128, d_rope=64, d_v=128,
                   q_offset=sq * r, causal=True, dtype="bf16",
                   name=f"dsv3_sp{sp}_rank{r}_S{seq}_h{n_h}")


DSV3_LAST_RANK = dsv3_rank(7)


def dsv3_zigzag_rank(r: int, sp: int = 8, seq: int = 16384, n_h: int = 128) -> Problem:
    """One zigzag SP shard: the sequence cut into 2*sp chunks, rank r holding
    chunks r and 2*sp-1-r, so every rank sees the same number of (query, key) pairs."""
    c = seq // (2 * sp)
    return Problem(B=1, Sq=2 * c, S=seq, n_h=n_h, d_c=512, d_nope=128, d_rope=64, d_v=128,
                   q_offset=c * r, causal=True, dtype="bf16", q_split=c, q_offset2=c * (2 * sp - 1 - r),
                   name=f"dsv3_sp{sp}_zigzag_rank{r}_S{seq}_h{n_h}")


def sweep_points():
    """Last-rank SP=8 shards over sequence length and head count."""
    for seq in (4096, 8192, 16384, 32768):
        for n_h in (32, 64, 128):
            yield dsv3_rank(7, sp=8, seq=seq, n_h=n_h)


NAMED = {p.name: p for p in [TINY_F32, MID_BF16] + [dsv3_rank(r) for r in range(8)]
         + [dsv3_zigzag_rank(r) for r in range(8)] + list(sweep_points())}

# Workloads made of several shards run back to back in one step: every SP=8
# rank of the DeepSeek-V3 layer in turn (q_offset = 2048 r), i.e. the whole
# 16384-token sequence's attention block as eight rank-local calls.
GROUPS = {"dsv3_sp8_all_ranks_S16384_h128": [dsv3_rank(r) for r in range(8)],
          "dsv3_sp8_zigzag_all_ranks_S16384_h128": [dsv3_zigzag_rank(r) for r in range(8)]}
