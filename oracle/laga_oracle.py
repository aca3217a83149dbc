"""Plain fp64 CPU oracle of the LAGA MLA attention block (forward and backward).

TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this module. The library's compute path never
calls it and shares no code with it.

What it computes
----------------
"A Training-Memory Regression in MLA Sequence Parallelism ... LAGA"
(weekinpapers page, Abstract) describes LAGA as keeping the absorbed form's
gather of the compressed latent while rejecting the absorb reformulation:
every sequence-parallel rank rebuilds the per-head K and V from the gathered
latent and then runs ordinary attention. The same Abstract states LAGA is
bit-identical to Megatron-Core's explicit form at SP=1, so the oracle is the
explicit form written out directly:

  1. reconstruct   K_nope[b,j,h,:] = c_kv[b,j,:] @ W_UK[:, h*d_nope:(h+1)*d_nope]
                   V[b,j,h,:]      = c_kv[b,j,:] @ W_UV[:, h*d_v:(h+1)*d_v]
  2. RoPE concat   K_h[j] = [K_nope[b,j,h,:] | k_rope[b,j,:]]  (one RoPE key for all heads)
  3. attention     s_ij = scale * q_i . K_j, key j visible to local query i iff
                   j <= q_offset + i (causal), lse_i = log sum_j exp(s_ij),
                   out_i = sum_j exp(s_ij - lse_i) V_j
  4. attention backward (closed-form softmax gradient)
  5. reconstruction backward  dW_UK = c_kv^T dK_nope, dW_UV = c_kv^T dV,
                   dc_kv = dK_nope W_UK^T + dV W_UV^T, dk_rope = sum over heads.

Readings where the page is silent (each listed in the design notes): the
softmax scale defaults to 1/sqrt(d_nope + d_rope); q is laid out as
[q_nope | q_rope]; lse is the natural log of the scaled scores; the causal
diagonal is inclusive in absolute positions; batch elements are independent
and dW sums over them.

Everything is float64; inputs are upcast exactly. Row chunks only bound
memory, they do not change the arithmetic.

absorbed_forward writes out the absorbed MLA form the Abstract contrasts LAGA
with (W_UK folded into the query, attention in the latent space); it reaches
the same out and lse by a different factorisation of the same scores.
absorbed_backward takes that form's gradients through its own steps.

Every function here has a pin in the CPU test suite (brute-force attention,
the absorbed form against the explicit one, sequence-parallel shard
consistency, finite differences, closed-form special cases, hand-worked
examples and gradient identities).
"""
from __future__ import annotations

import numpy as np

ROW_CHUNK = 1024


def default_scale(d_nope: int, d_rope: int) -> float:
    """Softmax scale when the caller gives none: 1/sqrt(query-key width)."""
    return 1.0 / np.sqrt(d_nope + d_rope)


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def reconstruct_head(c_kv_b, W_UK, W_UV, h, d_nope, d_v):
    """Step 1 for one batch element and head: K_nope_h = c_kv W_UK_h, V_h = c_kv W_UV_h.

    LAGA Abstract: per-head K/V are rebuilt locally from the gathered latent.
    """
    c = _f64(c_kv_b)
    k = c @ _f64(W_UK[:, h * d_nope:(h + 1) * d_nope])
    v = c @ _f64(W_UV[:, h * d_v:(h + 1) * d_v])
    return k, v


def head_key(k_nope_h, k_rope_b):
    """Step 2: the head's full key is its no-RoPE key followed by the shared RoPE key."""
    return np.concatenate([_f64(k_nope_h), _f64(k_rope_b)], axis=1)


def query_positions(sq, q_offset, q_split=0, q_offset2=0):
    """Absolute position of every local query row. One segment: q_offset + i. A
    two-segment (zigzag) shard, q_split > 0: rows i < q_split at q_offset + i,
    rows i >= q_split at q_offset2 + (i - q_split)."""
    i = np.arange(sq)
    if q_split <= 0:
        return q_offset + i
    return np.where(i < q_split, q_offset + i, q_offset2 + (i - q_split))


def visible_mask(rows, n_keys, q_offset, causal):
    """Which keys each local query row sees: j <= position of row i when causal, else
    all. q_offset is the first row's position (an int) or every row's position."""
    rows = np.asarray(rows)
    if not causal:
        return np.ones((rows.shape[0], n_keys), dtype=bool)
    pos = q_offset + rows if np.isscalar(q_offset) else np.asarray(q_offset)[rows]
    return np.arange(n_keys)[None, :] <= pos[:, None]


def attention_head_forward(q_h, K_h, V_h, q_offset, causal, scale, rows=None):
    """Step 3 for one head: masked scaled scores, natural-log LSE, softmax-weighted V.

    Returns (out [len(rows), d_v], lse [len(rows)]).
    """
    q_h = _f64(q_h)
    rows = np.arange(q_h.shape[0]) if rows is None else np.asarray(rows)
    n_keys = K_h.shape[0]
    outs, lses = [], []
    for c0 in range(0, rows.shape[0], ROW_CHUNK):
        r = rows[c0:c0 + ROW_CHUNK]
        s = scale * (q_h[r] @ K_h.T)
        s = np.where(visible_mask(r, n_keys, q_offset, causal), s, -np.inf)
        m = s.max(axis=1, keepdims=True)
        e = np.exp(s - m)
        l = e.sum(axis=1, keepdims=True)
        outs.append((e / l) @ V_h)
        lses.append(m[:, 0] + np.log(l[:, 0]))
    return np.concatenate(outs, axis=0), np.concatenate(lses, axis=0)


def attention_head_backward(q_h, K_h, V_h, out_h, lse_h, dout_h, q_offset, causal, scale):
    """Step 4 for one head, from the closed-form softmax gradient.

    p_ij = exp(s_ij - lse_i); D_i = dout_i . out_i; dV_j = sum_i p_ij dout_i;
    dp_ij = dout_i . V_j; ds_ij = p_ij (dp_ij - D_i);
    dq_i = scale sum_j ds_ij K_j; dK_j = scale sum_i ds_ij q_i.
    Returns (dq_h [Sq,d_qk], dK_h [n_keys,d_qk], dV_h [n_keys,d_v]).
    """
    q_h, out_h, dout_h = _f64(q_h), _f64(out_h), _f64(dout_h)
    lse_h = _f64(lse_h)
    sq, n_keys = q_h.shape[0], K_h.shape[0]
    dq = np.zeros_like(q_h)
    dK = np.zeros((n_keys, K_h.shape[1]))
    dV = np.zeros((n_keys, V_h.shape[1]))
    D = (dout_h * out_h).sum(axis=1)
    for c0 in range(0, sq, ROW_CHUNK):
        r = np.arange(c0, min(sq, c0 + ROW_CHUNK))
        s = scale * (q_h[r] @ K_h.T)
        vis = visible_mask(r, n_keys, q_offset, causal)
        p = np.where(vis, np.exp(np.where(vis, s, 0.0) - lse_h[r][:, None]), 0.0)
        dV += p.T @ dout_h[r]
        dp = dout_h[r] @ V_h.T
        ds = p * (dp - D[r][:, None])
        dq[r] = scale * (ds @ K_h)
        dK += scale * (ds.T @ q_h[r])
    return dq, dK, dV


def mla_forward_head(q, c_kv, k_rope, W_UK, W_UV, b, h, q_offset, causal, scale=None, rows=None):
    """Steps 1-3 for one (batch, head); rows selects local query rows (default all)."""
    d_qk = q.shape[3]
    n_h = q.shape[2]
    d_nope = W_UK.shape[1] // n_h
    d_v = W_UV.shape[1] // n_h
    d_rope = d_qk - d_nope
    if scale is None:
        scale = default_scale(d_nope, d_rope)
    k_nope, v = reconstruct_head(c_kv[b], W_UK, W_UV, h, d_nope, d_v)
    K_h = head_key(k_nope, k_rope[b])
    return attention_head_forward(q[b, :, h, :], K_h, v, q_offset, causal, scale, rows)


def mla_forward(q, c_kv, k_rope, W_UK, W_UV, q_offset=0, causal=True, scale=None, q_split=0, q_offset2=0):
    """Forward of the attention block: returns out [B,Sq,n_h,d_v] and lse [B,n_h,Sq] (fp64).
    q_split > 0: a two-segment shard (rows from q_split on start at position q_offset2)."""
    B, Sq, n_h, _ = q.shape
    if q_split > 0:
        q_offset = query_positions(Sq, q_offset, q_split, q_offset2)
    d_v = W_UV.shape[1] // n_h
    out = np.zeros((B, Sq, n_h, d_v))
    lse = np.zeros((B, n_h, Sq))
    for b in range(B):
        for h in range(n_h):
            o, l = mla_forward_head(q, c_kv, k_rope, W_UK, W_UV, b, h, q_offset, causal, scale)
            out[b, :, h, :] = o
            lse[b, h, :] = l
    return out, lse


def mla_backward_head(q, c_kv, k_rope, W_UK, W_UV, dout, b, h, q_offset, causal, scale=None):
    """Steps 1-5 for one (batch, head), each gradient as this head's contribution.

    Returns a dict with dq_h [Sq,d_qk], dK_nope_h, dV_h, dK_rope_h (this head's
    RoPE-key gradient, before the sum over heads), dW_UK_h [d_c,d_nope],
    dW_UV_h [d_c,d_v] (this batch element only) and dc_kv_h [S,d_c].
    """
    d_qk = q.shape[3]
    n_h = q.shape[2]
    d_nope = W_UK.shape[1] // n_h
    d_v = W_UV.shape[1] // n_h
    d_rope = d_qk - d_nope
    if scale is None:
        scale = default_scale(d_nope, d_rope)
    k_nope, v = reconstruct_head(c_kv[b], W_UK, W_UV, h, d_nope, d_v)
    K_h = head_key(k_nope, k_rope[b])
    q_h = q[b, :, h, :]
    out_h, lse_h = attention_head_forward(q_h, K_h, v, q_offset, causal, scale)
    dq, dK, dV = attention_head_backward(q_h, K_h, v, out_h, lse_h, dout[b, :, h, :],
                                         q_offset, causal, scale)
    dK_nope, dK_rope = dK[:, :d_nope], dK[:, d_nope:]
    c = _f64(c_kv[b])
    wk = _f64(W_UK[:, h * d_nope:(h + 1) * d_nope])
    wv = _f64(W_UV[:, h * d_v:(h + 1) * d_v])
    return {
        "dq_h": dq, "dK_nope_h": dK_nope, "dV_h": dV, "dK_rope_h": dK_rope,
        "dW_UK_h": c.T @ dK_nope, "dW_UV_h": c.T @ dV,
        "dc_kv_h": dK_nope @ wk.T + dV @ wv.T,
        "out_h": out_h, "lse_h": lse_h,
    }


def mla_backward(q, c_kv, k_rope, W_UK, W_UV, dout, q_offset=0, causal=True, scale=None, q_split=0, q_offset2=0):
    """Backward of the attention block for the loss <dout, out>.

    Returns dq [B,Sq,n_h,d_qk], dc_kv [B,S,d_c], dk_rope [B,S,d_rope],
    dW_UK [d_c,n_h*d_nope], dW_UV [d_c,n_h*d_v] (all fp64). Latent rows that no
    query of the shard can see get zero gradient, since they enter nothing.
    q_split > 0: a two-segment shard, as in mla_forward.
    """
    B, Sq, n_h, d_qk = q.shape
    if q_split > 0:
        q_offset = query_positions(Sq, q_offset, q_split, q_offset2)
    S, d_c = c_kv.shape[1], c_kv.shape[2]
    d_nope = W_UK.shape[1] // n_h
    d_v = W_UV.shape[1] // n_h
    dq = np.zeros((B, Sq, n_h, d_qk))
    dc_kv = np.zeros((B, S, d_c))
    dk_rope = np.zeros((B, S, d_qk - d_nope))
    dW_UK = np.zeros((d_c, n_h * d_nope))
    dW_UV = np.zeros((d_c, n_h * d_v))
    for b in range(B):
        for h in range(n_h):
            g = mla_backward_head(q, c_kv, k_rope, W_UK, W_UV, dout, b, h, q_offset, causal, scale)
            dq[b, :, h, :] = g["dq_h"]
            dk_rope[b] += g["dK_rope_h"]
            dc_kv[b] += g["dc_kv_h"]
            dW_UK[:, h * d_nope:(h + 1) * d_nope] += g["dW_UK_h"]
            dW_UV[:, h * d_v:(h + 1) * d_v] += g["dW_UV_h"]
    return {"dq": dq, "dc_kv": dc_kv, "dk_rope": dk_rope, "dW_UK": dW_UK, "dW_UV": dW_UV}


def absorbed_forward(q, c_kv, k_rope, W_UK, W_UV, q_offset=0, causal=True, scale=None, keep=None):
    """The absorbed MLA form (the variant the LAGA Abstract contrasts with: W_UK is
    folded into the query and attention runs over the compressed latent):

      q_lat_h = q_nope_h W_UK_h^T,  s = scale ([q_lat_h | q_rope_h] [c_kv | k_rope]^T),
      ctx_h = softmax(s) c_kv,      out_h = ctx_h W_UV_h.

    Returns out [B,Sq,n_h,d_v] and lse [B,n_h,Sq] (fp64). If `keep` is a dict, the
    intermediates q_lat and ctx ([B,Sq,n_h,d_c]) are stored in it."""
    B, Sq, n_h, d_qk = q.shape
    S, d_c = c_kv.shape[1], c_kv.shape[2]
    d_nope = W_UK.shape[1] // n_h
    d_v = W_UV.shape[1] // n_h
    if scale is None:
        scale = default_scale(d_nope, d_qk - d_nope)
    out = np.zeros((B, Sq, n_h, d_v))
    lse = np.zeros((B, n_h, Sq))
    q_lat_all = np.zeros((B, Sq, n_h, d_c))
    ctx_all = np.zeros((B, Sq, n_h, d_c))
    for b in range(B):
        key = np.concatenate([_f64(c_kv[b]), _f64(k_rope[b])], axis=1)  # one key for every head
        for h in range(n_h):
            q_lat = _f64(q[b, :, h, :d_nope]) @ _f64(W_UK[:, h * d_nope:(h + 1) * d_nope]).T
            q_abs = np.concatenate([q_lat, _f64(q[b, :, h, d_nope:])], axis=1)
            s = scale * (q_abs @ key.T)
            s = np.where(visible_mask(np.arange(Sq), S, q_offset, causal), s, -np.inf)
            m = s.max(axis=1, keepdims=True)
            e = np.exp(s - m)
            l = e.sum(axis=1, keepdims=True)
            ctx = (e / l) @ _f64(c_kv[b])  # attention in the latent space
            out[b, :, h, :] = ctx @ _f64(W_UV[:, h * d_v:(h + 1) * d_v])
            lse[b, h, :] = m[:, 0] + np.log(l[:, 0])
            q_lat_all[b, :, h] = q_lat
            ctx_all[b, :, h] = ctx
    if keep is not None:
        keep["q_lat"] = q_lat_all
        keep["ctx"] = ctx_all
    return out, lse



def absorbed_backward(q, c_kv, k_rope, W_UK, W_UV, dout, q_offset=0, causal=True, scale=None):
    """Gradients of <dout, out> for the absorbed form, taken through its own steps
    (the latent-space context and the absorbed query), per (batch, head):

      dctx = dout W_UV_h^T,           dW_UV_h = ctx^T dout,
      dP = dctx c_kv^T,               dS = P o (dP - rowsum(dP o P)),
      dq_lat = scale dS c_kv,         dq_rope = scale dS k_rope,
      dc_kv += scale dS^T q_lat + P^T dctx,   dk_rope += scale dS^T q_rope,
      dq_nope = dq_lat W_UK_h,        dW_UK_h = dq_lat^T q_nope_h.

    The absorbed form is the explicit form's function written another way, so these
    equal mla_backward's gradients up to rounding. Returns the same dict
    (dq, dc_kv, dk_rope, dW_UK, dW_UV), fp64."""
    B, Sq, n_h, d_qk = q.shape
    S, d_c = c_kv.shape[1], c_kv.shape[2]
    d_nope = W_UK.shape[1] // n_h
    d_v = W_UV.shape[1] // n_h
    if scale is None:
        scale = default_scale(d_nope, d_qk - d_nope)
    dq = np.zeros((B, Sq, n_h, d_qk))
    dc_kv = np.zeros((B, S, d_c))
    dk_rope = np.zeros((B, S, d_qk - d_nope))
    dW_UK = np.zeros((d_c, n_h * d_nope))
    dW_UV = np.zeros((d_c, n_h * d_v))
    for b in range(B):
        c = _f64(c_kv[b])
        r = _f64(k_rope[b])
        key = np.concatenate([c, r], axis=1)
        for h in range(n_h):
            wk = _f64(W_UK[:, h * d_nope:(h + 1) * d_nope])
            wv = _f64(W_UV[:, h * d_v:(h + 1) * d_v])
            q_nope = _f64(q[b, :, h, :d_nope])
            q_rope = _f64(q[b, :, h, d_nope:])
            q_lat = q_nope @ wk.T
            s = scale * (np.concatenate([q_lat, q_rope], axis=1) @ key.T)
            s = np.where(visible_mask(np.arange(Sq), S, q_offset, causal), s, -np.inf)
            e = np.exp(s - s.max(axis=1, keepdims=True))
            P = e / e.sum(axis=1, keepdims=True)
            ctx = P @ c
            g = _f64(dout[b, :, h, :])
            dctx = g @ wv.T
            dW_UV[:, h * d_v:(h + 1) * d_v] += ctx.T @ g
            dP = dctx @ c.T
            dS = P * (dP - (dP * P).sum(axis=1, keepdims=True))
            dq_lat = scale * (dS @ c)
            dq[b, :, h, d_nope:] = scale * (dS @ r)
            dc_kv[b] += scale * (dS.T @ q_lat) + P.T @ dctx
            dk_rope[b] += scale * (dS.T @ q_rope)
            dq[b, :, h, :d_nope] = dq_lat @ wk
            dW_UK[:, h * d_nope:(h + 1) * d_nope] += dq_lat.T @ q_nope
    return {"dq": dq, "dc_kv": dc_kv, "dk_rope": dk_rope, "dW_UK": dW_UK, "dW_UV": dW_UV}

def reconstruct(c_kv, W_UK, W_UV, n_h):
    """Step 1 for the whole batch: K_nope [B,S,n_h,d_nope] and V [B,S,n_h,d_v]."""
    B, S, d_c = c_kv.shape
    c = _f64(c_kv).reshape(B * S, d_c)
    k = (c @ _f64(W_UK)).reshape(B, S, n_h, -1)
    v = (c @ _f64(W_UV)).reshape(B, S, n_h, -1)
    return k, v
