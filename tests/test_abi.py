"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every entry point the header declares, and rejects bad arguments before any
launch."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from mla_attention_sequence_gb300 import build, laga
    build.build()
    return laga.lib()


def header_functions():
    text = open(os.path.join(ROOT, "include", "laga_mla.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(laga_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = header_functions()
    for n in ("laga_mla_fwd", "laga_mla_bwd", "laga_mla_fwd_workspace_size", "laga_mla_bwd_workspace_size",
              "laga_mla_check", "laga_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(L):
    for n in header_functions():
        assert hasattr(L, n), n
    from mla_attention_sequence_gb300 import laga
    assert set(laga.EXPORTS) <= set(header_functions())


def test_version_and_status_strings(L):
    assert L.laga_mla_version() >= 100
    for code, name in [(0, b"LAGA_OK"), (1, b"LAGA_ERR_INVALID_ARG"), (2, b"LAGA_ERR_UNSUPPORTED"),
                       (3, b"LAGA_ERR_WORKSPACE"), (4, b"LAGA_ERR_CUDA"), (5, b"LAGA_ERR_TIMEOUT")]:
        assert L.laga_status_string(code) == name


def desc(**kw):
    from mla_attention_sequence_gb300 import laga
    from mla_attention_sequence_gb300.configs import DSV3_LAST_RANK
    p = DSV3_LAST_RANK.with_(**{k: v for k, v in kw.items() if k in DSV3_LAST_RANK.__dataclass_fields__})
    return laga.make_desc(p, None, kw.get("variant", "auto"))


FAKE = ctypes.c_void_p(4096)  # aligned, never dereferenced: validation fails first


def call_fwd(L, d, **ptrs):
    args = {k: FAKE for k in ("q", "c", "r", "wk", "wv", "o", "l", "ws")}
    args.update(ptrs)
    return L.laga_mla_fwd(ctypes.byref(d), args["q"], args["c"], args["r"], args["wk"], args["wv"], args["o"],
                          args["l"], args["ws"], ctypes.c_size_t(1 << 40), None)


def test_invalid_arguments_are_rejected_before_launch(L):
    assert L.laga_mla_fwd(None, *([FAKE] * 8), ctypes.c_size_t(0), None) == 1
    # causal shard beyond the latent
    assert call_fwd(L, desc(q_offset=15000)) == 1
    assert b"q_offset" in L.laga_mla_last_error()
    # null / misaligned pointers
    assert call_fwd(L, desc(), q=None) == 1
    assert call_fwd(L, desc(), o=ctypes.c_void_p(4097)) == 1
    # non-positive sizes
    assert call_fwd(L, desc(n_h=0)) == 1
    assert call_fwd(L, desc(Sq=0)) == 1


def test_two_segment_shards_are_checked_before_launch(L):
    def two(q_split, q_offset2, **kw):
        d = desc(**kw)
        d.q_split, d.q_offset2 = q_split, q_offset2
        return d
    # q_split must be a multiple of 128 inside (0, sq)
    assert call_fwd(L, two(100, 0)) == 1
    assert b"q_split" in L.laga_mla_last_error()
    assert call_fwd(L, two(-128, 0)) == 1
    assert call_fwd(L, two(desc().sq, 0)) == 1
    # the second segment must end inside the latent for a causal shard
    assert call_fwd(L, two(128, desc().skv)) == 1
    assert b"q_offset2" in L.laga_mla_last_error()
    # only the tensor-core materialize path takes two segments
    assert call_fwd(L, two(128, 0, variant="simt")) == 2
    assert call_fwd(L, two(128, 0, variant="fused_recon")) == 2
    assert b"two query segments" in L.laga_mla_last_error()
    # a valid zigzag shard passes the checks and asks for a workspace
    d = two(128, 0)
    assert L.laga_mla_fwd_workspace_size(ctypes.byref(d)) > 0


def test_unknown_flag_bits_rejected(L):
    d = desc()
    d.flags = 4  # bits 0 (REUSE_KV) and 1 (KV_PREBUILT) are defined
    assert call_fwd(L, d) == 1
    assert b"flags" in L.laga_mla_last_error()


def test_reconstruct_rows_argument_checks(L):
    """laga_mla_reconstruct_rows rejects bad row ranges and unsupported paths before
    any launch (no device memory is touched: the checks precede the workspace)."""
    from mla_attention_sequence_gb300 import laga
    fn = L.laga_mla_reconstruct_rows
    fn.argtypes = [ctypes.POINTER(laga.LagaDesc), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                   ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    p16 = ctypes.c_void_p(256)  # aligned, never dereferenced: every call below fails a check first
    d = desc(variant="materialize")
    for row0, rows in ((64, 128), (-128, 128), (0, 0), (0, 100)):
        assert fn(ctypes.byref(d), p16, p16, p16, row0, rows, None, 0, None) == 1, (row0, rows)
    assert fn(ctypes.byref(d), p16, p16, p16, 0, 128, None, 0, None) == 3  # workspace missing
    f32 = desc(dtype="f32")
    assert fn(ctypes.byref(f32), p16, p16, p16, 0, 128, None, 0, None) == 2  # CUDA-core path: unsupported


def test_unsupported_tensor_core_dims(L):
    d = desc(d_c=256, variant="materialize")
    assert call_fwd(L, d) == 2
    d = desc(dtype="f32", variant="materialize")
    assert call_fwd(L, d) == 2


def test_workspace_errors(L):
    d = desc()
    n = L.laga_mla_fwd_workspace_size(ctypes.byref(d))
    assert n > 0
    r = L.laga_mla_fwd(ctypes.byref(d), *([FAKE] * 7), None, ctypes.c_size_t(n), None)
    assert r == 3
    r = L.laga_mla_fwd(ctypes.byref(d), *([FAKE] * 7), FAKE, ctypes.c_size_t(n - 1), None)
    assert r == 3


def test_workspace_sizes_match_layout(L):
    from mla_attention_sequence_gb300 import laga
    from mla_attention_sequence_gb300.configs import DSV3_LAST_RANK, MID_BF16, TINY_F32
    p = DSV3_LAST_RANK
    # forward: materialised K_nope and V for the visible prefix, bf16
    assert laga.fwd_workspace_bytes(p) == 2 * p.B * 16384 * p.n_h * 128 * 2
    nb = laga.bwd_workspace_bytes(p)
    # backward: K_nope, V, dK_nope, dV (bf16), the RoPE-key gradient partials of the
    # dK/dV kernel's head groups (4 heads per CTA at n_h = 128; fp32), lse and D rows
    kv = p.B * 16384 * p.n_h * 128 * 2
    dkr = p.B * 16384 * (p.n_h // 4) * 64 * 4
    rows = p.B * p.n_h * 2048 * 4
    assert nb == 4 * kv + dkr + 2 * rows
    assert laga.fwd_workspace_bytes(MID_BF16) > 0
    assert laga.fwd_workspace_bytes(TINY_F32) > 0
    assert laga.fwd_workspace_bytes(p, "fused_recon") == 0
    assert laga.bwd_workspace_bytes(p, "fused_recon") == 0  # forward-only variant


def test_binding_refuses_cpu_tensors():
    import torch
    from mla_attention_sequence_gb300 import laga
    q = torch.zeros(1, 4, 2, 48)
    c = torch.zeros(1, 4, 64)
    r = torch.zeros(1, 4, 16)
    wk = torch.zeros(64, 64)
    wv = torch.zeros(64, 64)
    with pytest.raises(RuntimeError, match="CUDA"):
        laga.fwd(q, c, r, wk, wv)
