"""Sequence-parallel LAGA across ranks: the steps either side of the local op.

"A Training-Memory Regression in MLA Sequence Parallelism ... LAGA" (weekinpapers
page, Abstract): each sequence-parallel (SP) rank keeps only its shard of the
compressed latent; the ranks gather the latent (as the absorbed form does, which
is what makes the communication small) and every rank then rebuilds all heads'
K and V from the gathered latent locally. This module is that exchange around
the library's local op:

  forward   pack this rank's latent rows [B, S/SP, d_c] and RoPE-key rows
            [B, S/SP, d_rope] into one [B, S/SP, d_c + d_rope] tensor, all-gather
            it over the SP group, unpack the full-sequence c_kv and k_rope, and run
            the local forward for this rank's query rows at their positions;
  backward  run the local backward, which returns this rank's contribution to
            dc_kv and dk_rope for every latent row (its queries see all of them)
            and to dW_UK / dW_UV; reduce-scatter the packed [dc_kv | dk_rope] over
            the group, so each rank receives the full gradient of its own latent
            rows, and all-reduce dW_UK and dW_UV.

Shard layouts: "contiguous" (rank r holds rows [r S/SP, (r+1) S/SP)) and
"zigzag" (the sequence cut into 2 SP chunks; rank r holds chunks r and
2 SP - 1 - r, a two-segment query shard). A rank's latent rows and query rows
are the same sequence positions.

The collectives are torch.distributed calls (NCCL between GPUs, gloo on CPU);
the local op is a parameter, by default the library's C-ABI forward and
backward (laga.fwd / laga.bwd), so the exchange logic can be exercised on CPU
with any op of the same signature. Remote latent rows always land in this
rank's memory through the collective before any kernel reads them.

Overlapped forward (overlap=True): the gather runs as one broadcast per source
rank, all issued asynchronously in one global order; this rank rebuilds K_nope
and V for its own rows at once (laga.reconstruct_rows into the forward's
workspace), then for each remote chunk waits for its broadcast and rebuilds
its rows while the later broadcasts are still in flight; the attention then
runs on the prebuilt K/V (laga.fwd with kv_prebuilt) and the backward reuses
them (reuse_kv). The local steps come from an ops object (LibraryOps by
default) so that the chunk logic also runs on CPU ranks.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Callable

import torch
import torch.distributed as dist


@dataclass(frozen=True)
class Layout:
    """Which sequence rows each of `sp` ranks holds, for a sequence of `seq` rows."""
    seq: int
    sp: int
    kind: str = "contiguous"  # or "zigzag"

    def __post_init__(self):
        parts = self.sp if self.kind == "contiguous" else 2 * self.sp
        if self.kind not in ("contiguous", "zigzag"):
            raise ValueError("layout is 'contiguous' or 'zigzag'")
        if self.seq % parts:
            raise ValueError(f"sequence length {self.seq} is not a multiple of {parts}")

    @property
    def rows_per_rank(self) -> int:
        return self.seq // self.sp

    def segments(self, rank: int) -> list[tuple[int, int]]:
        """(first sequence row, rows) of each contiguous piece rank `rank` holds, in order."""
        if self.kind == "contiguous":
            n = self.seq // self.sp
            return [(rank * n, n)]
        c = self.seq // (2 * self.sp)
        return [(rank * c, c), ((2 * self.sp - 1 - rank) * c, c)]

    def rows(self, rank: int) -> torch.Tensor:
        """Sequence positions of rank `rank`'s rows, in its local order."""
        return torch.cat([torch.arange(a, a + n) for a, n in self.segments(rank)])

    def query_args(self, rank: int) -> dict:
        """The local op's position arguments for this rank's query rows."""
        seg = self.segments(rank)
        if len(seg) == 1:
            return {"q_offset": seg[0][0], "q_split": 0, "q_offset2": 0}
        return {"q_offset": seg[0][0], "q_split": seg[0][1], "q_offset2": seg[1][0]}

    def gather_order(self) -> torch.Tensor:
        """Index that puts the rank-major concatenation of all ranks' rows into
        sequence order (applied to the gathered rows)."""
        owner = torch.cat([self.rows(r) for r in range(self.sp)])
        return torch.argsort(owner)


class LibraryOps:
    """The overlapped path's local steps through the library's C ABI."""

    def prepare(self, q, c_kv, k_rope, W_UK, W_UV, pos, causal):
        from . import laga
        p = laga.problem_of(q, c_kv, k_rope, W_UK, W_UV, pos["q_offset"], causal, pos["q_split"], pos["q_offset2"])
        return torch.empty(laga.bwd_workspace_bytes(p), dtype=torch.uint8, device=q.device)

    def rebuild(self, q, c_kv, k_rope, W_UK, W_UV, pos, causal, row0, rows, ws):
        from . import laga
        laga.reconstruct_rows(q, c_kv, k_rope, W_UK, W_UV, row0, rows, ws, pos["q_offset"], causal, pos["q_split"],
                              pos["q_offset2"])

    def fwd_prebuilt(self, q, c_kv, k_rope, W_UK, W_UV, pos, causal, ws):
        from . import laga
        return laga.fwd(q, c_kv, k_rope, W_UK, W_UV, pos["q_offset"], causal, workspace=ws, q_split=pos["q_split"],
                        q_offset2=pos["q_offset2"], kv_prebuilt=True)

    def bwd_reuse(self, q, c_kv, k_rope, W_UK, W_UV, out, lse, dout, pos, causal, ws):
        from . import laga
        return laga.bwd(q, c_kv, k_rope, W_UK, W_UV, out, lse, dout, pos["q_offset"], causal, workspace=ws,
                        reuse_kv=True, q_split=pos["q_split"], q_offset2=pos["q_offset2"])


def _local_fwd_default(q, c_kv, k_rope, W_UK, W_UV, q_offset, causal, q_split, q_offset2):
    from . import laga
    return laga.fwd(q, c_kv, k_rope, W_UK, W_UV, q_offset, causal, q_split=q_split, q_offset2=q_offset2)


def _local_bwd_default(q, c_kv, k_rope, W_UK, W_UV, out, lse, dout, q_offset, causal, q_split, q_offset2):
    from . import laga
    return laga.bwd(q, c_kv, k_rope, W_UK, W_UV, out, lse, dout, q_offset, causal, q_split=q_split,
                    q_offset2=q_offset2)


class SPAttention:
    """One LAGA attention block's forward and backward over an SP process group.

    Every rank calls forward / backward with its own shard (layout.rows(rank) of
    the sequence): q, dout [B, S/SP, n_h, .]; c_kv_shard [B, S/SP, d_c];
    k_rope_shard [B, S/SP, d_rope]; and the full W_UK, W_UV (replicated)."""

    def __init__(self, layout: Layout, group=None, causal: bool = True,
                 local_fwd: Callable | None = None, local_bwd: Callable | None = None,
                 overlap: bool = False, ops=None):
        self.layout = layout
        self.group = group
        self.causal = causal
        self.local_fwd = local_fwd or _local_fwd_default
        self.local_bwd = local_bwd or _local_bwd_default
        self.overlap = overlap
        self.ops = ops or LibraryOps()
        self._ws = None
        self.rank = dist.get_rank(group)
        if dist.get_world_size(group) != layout.sp:
            raise ValueError("the process group's size must equal the layout's SP degree")
        self._order = layout.gather_order()
        self._saved = None

    # ---------------------------------------------------------------- collectives
    def gather_latent(self, c_kv_shard: torch.Tensor, k_rope_shard: torch.Tensor):
        """All-gather of the packed latent: returns the full-sequence c_kv [B, S, d_c]
        and k_rope [B, S, d_rope] in sequence order."""
        d_c = c_kv_shard.shape[2]
        packed = torch.cat([c_kv_shard, k_rope_shard], dim=2).contiguous()  # [B, S/SP, d_c + d_rope]
        parts = [torch.empty_like(packed) for _ in range(self.layout.sp)]
        dist.all_gather(parts, packed, group=self.group)
        full = torch.cat(parts, dim=1)  # rank-major rows
        full = full.index_select(1, self._order.to(full.device))  # sequence order
        return full[:, :, :d_c].contiguous(), full[:, :, d_c:].contiguous()

    def scatter_latent_grad(self, dc_kv: torch.Tensor, dk_rope: torch.Tensor):
        """Reduce-scatter of the packed latent gradient: every rank contributes its
        partial [dc_kv | dk_rope] for all S rows and receives the sum over ranks for
        its own rows (in its local order)."""
        d_c = dc_kv.shape[2]
        packed = torch.cat([dc_kv, dk_rope], dim=2)
        owner = torch.cat([self.layout.rows(r) for r in range(self.layout.sp)]).to(packed.device)
        rank_major = packed.index_select(1, owner)  # rank r's rows r-th
        n = self.layout.rows_per_rank
        inputs = [rank_major[:, r * n:(r + 1) * n].contiguous() for r in range(self.layout.sp)]
        out = torch.empty_like(inputs[0])
        dist.reduce_scatter(out, inputs, op=dist.ReduceOp.SUM, group=self.group)
        return out[:, :, :d_c].contiguous(), out[:, :, d_c:].contiguous()

    def reduce_weight_grads(self, dW_UK: torch.Tensor, dW_UV: torch.Tensor):
        """All-reduce (sum) of the weight gradients every rank computed from its queries."""
        dist.all_reduce(dW_UK, op=dist.ReduceOp.SUM, group=self.group)
        dist.all_reduce(dW_UV, op=dist.ReduceOp.SUM, group=self.group)
        return dW_UK, dW_UV

    def _global_rank(self, group_rank: int) -> int:
        return group_rank if self.group is None else dist.get_global_rank(self.group, group_rank)

    def gather_and_rebuild(self, q, c_kv_shard, k_rope_shard, W_UK, W_UV, pos):
        """The overlapped gather: returns the full c_kv, k_rope and the workspace
        holding K_nope / V rebuilt for every row, chunk by chunk as chunks arrive."""
        B, n, d_c = c_kv_shard.shape
        S, sp = self.layout.seq, self.layout.sp
        packed = torch.cat([c_kv_shard, k_rope_shard], dim=2).contiguous()
        bufs, works = [], []
        for src in range(sp):  # one global order on every rank
            buf = packed if src == self.rank else torch.empty_like(packed)
            works.append(dist.broadcast(buf, src=self._global_rank(src), group=self.group, async_op=True))
            bufs.append(buf)
        c_full = torch.empty((B, S, d_c), dtype=packed.dtype, device=packed.device)
        r_full = torch.empty((B, S, packed.shape[2] - d_c), dtype=packed.dtype, device=packed.device)
        ws = self.ops.prepare(q, c_full, r_full, W_UK, W_UV, pos, self.causal)
        order = [self.rank] + [r for r in range(sp) if r != self.rank]  # own rows first: no wait
        for src in order:
            if src != self.rank:
                works[src].wait()
            off = 0
            for a, length in self.layout.segments(src):  # (first row, rows)
                b = a + length
                c_full[:, a:b] = bufs[src][:, off:off + length, :d_c]
                r_full[:, a:b] = bufs[src][:, off:off + length, d_c:]
                off += length
                # the chunk that ends the sequence also covers the padded rows past it
                self.ops.rebuild(q, c_full, r_full, W_UK, W_UV, pos, self.causal, a, (b - a) + (127 if b == S else 0),
                                 ws)
        works[self.rank].wait()
        return c_full, r_full, ws

    # ---------------------------------------------------------------- the block
    def forward(self, q, c_kv_shard, k_rope_shard, W_UK, W_UV):
        """Returns this rank's out [B, S/SP, n_h, d_v] and lse [B, n_h, S/SP]."""
        pos = self.layout.query_args(self.rank)
        if self.overlap:
            c_kv, k_rope, ws = self.gather_and_rebuild(q, c_kv_shard, k_rope_shard, W_UK, W_UV, pos)
            out, lse = self.ops.fwd_prebuilt(q, c_kv, k_rope, W_UK, W_UV, pos, self.causal, ws)
            self._ws = ws
            self._saved = (q, c_kv, k_rope, W_UK, W_UV, out, lse)
            return out, lse
        c_kv, k_rope = self.gather_latent(c_kv_shard, k_rope_shard)
        out, lse = self.local_fwd(q, c_kv, k_rope, W_UK, W_UV, pos["q_offset"], self.causal, pos["q_split"],
                                  pos["q_offset2"])
        self._saved = (q, c_kv, k_rope, W_UK, W_UV, out, lse)
        return out, lse

    def backward(self, dout):
        """Returns dq (this rank's rows), dc_kv and dk_rope (this rank's latent rows,
        summed over all ranks' queries) and dW_UK, dW_UV (summed over the group)."""
        if self._saved is None:
            raise RuntimeError("backward before forward")
        q, c_kv, k_rope, W_UK, W_UV, out, lse = self._saved
        pos = self.layout.query_args(self.rank)
        if self._ws is not None:  # overlapped forward: its workspace still holds K_nope / V
            g = self.ops.bwd_reuse(q, c_kv, k_rope, W_UK, W_UV, out, lse, dout, pos, self.causal, self._ws)
            self._ws = None
        else:
            g = self.local_bwd(q, c_kv, k_rope, W_UK, W_UV, out, lse, dout, pos["q_offset"], self.causal,
                               pos["q_split"], pos["q_offset2"])
        dc, dr = self.scatter_latent_grad(g["dc_kv"], g["dk_rope"])
        dWk, dWv = self.reduce_weight_grads(g["dW_UK"], g["dW_UV"])
        self._saved = None
        return {"dq": g["dq"], "dc_kv": dc, "dk_rope": dr, "dW_UK": dWk, "dW_UV": dWv}

    def bytes_per_step(self, B: int, d_c: int, d_rope: int, n_h: int, d_nope: int, d_v: int,
                       elem: int = 2) -> dict:
        """Bytes each rank sends in one forward + backward: the latent all-gather and
        the latent-gradient reduce-scatter move (SP-1)/SP of the packed latent, the
        weight all-reduce (ring) 2 (SP-1)/SP of the weights."""
        sp, S = self.layout.sp, self.layout.seq
        latent = B * S * (d_c + d_rope) * elem
        weights = d_c * n_h * (d_nope + d_v) * elem
        f = (sp - 1) / sp
        return {"all_gather": latent * f, "reduce_scatter": latent * f, "all_reduce": 2 * weights * f}
