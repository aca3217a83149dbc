"""laga_mla_fwd_noalloc: the forward for callers that cannot allocate device memory.

Such callers (a plug-in whose host framework owns all device memory, a runtime
with a fixed memory budget, a C caller without an allocator) cannot pass a
workspace, so this entry point keeps the forward's scratch in a static device
array of the library. The test calls it through the C ABI twice in a row, on
two different problems, the larger one second (so that a region the second
call failed to write would still hold the first call's data or zeros, not the
right values), and checks each result against laga_mla_fwd (the entry point
with a caller workspace). Both run the same kernels in the same order on the
same inputs, and the library's kernels are bitwise reproducible, so the results
must be bitwise equal; that is a stricter check than the bf16 tolerance the
parity tests use (max|diff| <= 2e-2 * max|reference|), which therefore holds
too. This file is collected last.
"""
import ctypes

import pytest
import torch

from mla_attention_sequence_gb300 import laga
from mla_attention_sequence_gb300.configs import DSV3_LAST_RANK, Problem
from mla_attention_sequence_gb300.synth import make_inputs

pytestmark = pytest.mark.gpu



def _lib():
    from mla_attention_sequence_gb300 import build
    build.build()
    L = laga.lib()
    f = L.laga_mla_fwd_noalloc
    vp = ctypes.c_void_p
    f.argtypes = [ctypes.POINTER(laga.LagaDesc), vp, vp, vp, vp, vp, vp, vp, vp]
    f.restype = ctypes.c_int
    return L


def _noalloc_forward(L, p, t):
    dev = t["q"].device
    out = torch.empty((p.B, p.Sq, p.n_h, p.d_v), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((p.B, p.n_h, p.Sq), dtype=torch.float32, device=dev)
    d = laga.make_desc(p)
    st = L.laga_mla_fwd_noalloc(ctypes.byref(d), t["q"].data_ptr(), t["c_kv"].data_ptr(), t["k_rope"].data_ptr(),
                                t["W_UK"].data_ptr(), t["W_UV"].data_ptr(), out.data_ptr(), lse.data_ptr(),
                                torch.cuda.current_stream(dev).cuda_stream)
    assert st == 0, L.laga_mla_last_error()
    assert L.laga_mla_check(torch.cuda.current_stream(dev).cuda_stream) == 0
    return out, lse


def test_noalloc_forward_matches_workspace_forward_twice():
    L = _lib()
    dev = torch.device("cuda", 0)
    problems = [
        Problem(B=2, Sq=200, S=520, n_h=3, d_c=512, d_nope=128, d_rope=64, d_v=128, q_offset=300, causal=True,
                dtype="bf16"),
        # larger second: 32 MiB of the 64 MiB array
        Problem(B=1, Sq=1000, S=4096, n_h=16, d_c=512, d_nope=128, d_rope=64, d_v=128, q_offset=3000, causal=True,
                dtype="bf16"),
    ]
    for i, p in enumerate(problems):
        x = make_inputs(p, seed=40 + i, with_dout=False)
        t = {k: torch.from_numpy(v).to(dev).to(torch.bfloat16).contiguous() for k, v in x.items()}
        ref_out, ref_lse = laga.fwd(t["q"], t["c_kv"], t["k_rope"], t["W_UK"], t["W_UV"], p.q_offset, p.causal)
        out, lse = _noalloc_forward(L, p, t)
        torch.cuda.synchronize()
        assert laga.fwd_workspace_bytes(p) <= 64 * 1024 * 1024
        assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
        assert torch.equal(out, ref_out), f"call {i}: out differs"
        assert torch.equal(lse, ref_lse), f"call {i}: lse differs"


def test_noalloc_rejects_problems_beyond_the_static_array():
    L = _lib()
    d = laga.make_desc(DSV3_LAST_RANK)
    need = L.laga_mla_fwd_workspace_size(ctypes.byref(d))
    assert need > 64 * 1024 * 1024
    fake = ctypes.c_void_p(4096)  # never dereferenced: the size check comes first
    st = L.laga_mla_fwd_noalloc(ctypes.byref(d), *([fake] * 7), None)
    assert st == 3  # LAGA_ERR_WORKSPACE
    assert b"static array" in L.laga_mla_last_error()
