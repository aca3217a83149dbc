"""Python binding of liblaga_mla.so (the C ABI in include/laga_mla.h).

Argument marshalling only: tensors are checked, outputs and workspace are
allocated with torch on the inputs' device, and every step of the computation
runs in the library's CUDA kernels on torch's current stream. There is no CPU
path: calling with CPU tensors, or without the built library, raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

from .configs import Problem

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build", "liblaga_mla.so")

LAGA_OK = 0
STATUS_NAMES = {0: "LAGA_OK", 1: "LAGA_ERR_INVALID_ARG", 2: "LAGA_ERR_UNSUPPORTED", 3: "LAGA_ERR_WORKSPACE",
                4: "LAGA_ERR_CUDA", 5: "LAGA_ERR_TIMEOUT"}
DTYPES = {"f32": 0, "bf16": 1}
VARIANTS = {"auto": 0, "materialize": 1, "fused_recon": 2, "simt": 3}
FLAG_REUSE_KV = 1
FLAG_KV_PREBUILT = 2

EXPORTS = ("laga_mla_fwd_workspace_size", "laga_mla_bwd_workspace_size", "laga_mla_fwd", "laga_mla_bwd",
           "laga_mla_reconstruct", "laga_mla_check", "laga_status_string", "laga_mla_last_error",
           "laga_mla_version", "laga_mla_selftest_timeout", "laga_mla_absorbed_fwd",
           "laga_mla_absorbed_fwd_workspace_size", "laga_mla_reconstruct_rows")


class LagaDesc(ctypes.Structure):
    """Mirror of laga_mla_desc."""
    _fields_ = [("batch", ctypes.c_int64), ("sq", ctypes.c_int64), ("skv", ctypes.c_int64),
                ("n_h", ctypes.c_int64), ("d_c", ctypes.c_int64), ("d_nope", ctypes.c_int64),
                ("d_rope", ctypes.c_int64), ("d_v", ctypes.c_int64), ("q_offset", ctypes.c_int64),
                ("causal", ctypes.c_int32), ("softmax_scale", ctypes.c_float), ("dtype", ctypes.c_int32),
                ("variant", ctypes.c_int32), ("flags", ctypes.c_int32), ("q_split", ctypes.c_int64),
                ("q_offset2", ctypes.c_int64)]


class LagaError(RuntimeError):
    def __init__(self, status: int, detail: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {detail}")
        self.status = status


_lib = None


def lib() -> ctypes.CDLL:
    """Load the library (built in-tree by the package's build step)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with mla_attention_sequence_gb300.build.build()")
    L = ctypes.CDLL(LIB_PATH)
    vp, sz, st = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
    pd = ctypes.POINTER(LagaDesc)
    L.laga_mla_fwd_workspace_size.argtypes = [pd]
    L.laga_mla_fwd_workspace_size.restype = sz
    L.laga_mla_bwd_workspace_size.argtypes = [pd]
    L.laga_mla_bwd_workspace_size.restype = sz
    L.laga_mla_fwd.argtypes = [pd, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.laga_mla_fwd.restype = st
    L.laga_mla_bwd.argtypes = [pd, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.laga_mla_bwd.restype = st
    L.laga_mla_absorbed_fwd_workspace_size.argtypes = [pd]
    L.laga_mla_absorbed_fwd_workspace_size.restype = sz
    L.laga_mla_absorbed_fwd.argtypes = [pd, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.laga_mla_absorbed_fwd.restype = st
    L.laga_mla_reconstruct.argtypes = [pd, vp, vp, vp, vp, vp, vp]
    L.laga_mla_reconstruct.restype = st
    L.laga_mla_reconstruct_rows.argtypes = [pd, vp, vp, vp, ctypes.c_int64, ctypes.c_int64, vp, sz, vp]
    L.laga_mla_reconstruct_rows.restype = st
    L.laga_mla_check.argtypes = [vp]
    L.laga_mla_check.restype = st
    L.laga_mla_selftest_timeout.argtypes = [vp]
    L.laga_mla_selftest_timeout.restype = st
    L.laga_status_string.argtypes = [st]
    L.laga_status_string.restype = ctypes.c_char_p
    L.laga_mla_last_error.argtypes = []
    L.laga_mla_last_error.restype = ctypes.c_char_p
    L.laga_mla_version.argtypes = []
    L.laga_mla_version.restype = ctypes.c_int
    _lib = L
    return L


def _raise_if(status: int):
    if status != LAGA_OK:
        raise LagaError(status, lib().laga_mla_last_error().decode(errors="replace"))


def make_desc(p: Problem, softmax_scale: float | None = None, variant: str = "auto", flags: int = 0) -> LagaDesc:
    return LagaDesc(p.B, p.Sq, p.S, p.n_h, p.d_c, p.d_nope, p.d_rope, p.d_v, p.q_offset, 1 if p.causal else 0,
                    float(softmax_scale) if softmax_scale else 0.0, DTYPES[p.dtype], VARIANTS[variant], flags,
                    p.q_split, p.q_offset2)


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def problem_of(q, c_kv, k_rope, W_UK, W_UV, q_offset: int, causal: bool, q_split: int = 0,
               q_offset2: int = 0) -> Problem:
    """Infer and check the problem sizes from the input tensors. q_split > 0 makes
    rows [q_split, Sq) a second query segment starting at position q_offset2."""
    if q.dim() != 4 or c_kv.dim() != 3 or k_rope.dim() != 3 or W_UK.dim() != 2 or W_UV.dim() != 2:
        raise ValueError("expected q [B,Sq,n_h,d_qk], c_kv [B,S,d_c], k_rope [B,S,d_rope], W [d_c, n_h*d]")
    B, Sq, n_h, d_qk = q.shape
    _, S, d_c = c_kv.shape
    d_rope = k_rope.shape[2]
    if c_kv.shape[0] != B or k_rope.shape[:2] != (B, S) or W_UK.shape[0] != d_c or W_UV.shape[0] != d_c:
        raise ValueError("inconsistent batch / latent shapes")
    if W_UK.shape[1] % n_h or W_UV.shape[1] % n_h:
        raise ValueError("W_UK / W_UV columns must be n_h * head width")
    d_nope, d_v = W_UK.shape[1] // n_h, W_UV.shape[1] // n_h
    if d_nope + d_rope != d_qk:
        raise ValueError("q's last dim must be d_nope + d_rope")
    dt = {torch.float32: "f32", torch.bfloat16: "bf16"}.get(q.dtype)
    if dt is None:
        raise TypeError("tensors must be float32 or bfloat16")
    for t in (q, c_kv, k_rope, W_UK, W_UV):
        if t.dtype != q.dtype:
            raise TypeError("all inputs must share one dtype")
        if not t.is_cuda:
            raise RuntimeError("LAGA MLA runs on CUDA tensors only")
        if not t.is_contiguous():
            raise ValueError("inputs must be contiguous")
    return Problem(B=B, Sq=Sq, S=S, n_h=n_h, d_c=d_c, d_nope=d_nope, d_rope=d_rope, d_v=d_v,
                   q_offset=int(q_offset), causal=bool(causal), dtype=dt, q_split=int(q_split),
                   q_offset2=int(q_offset2))


def fwd_workspace_bytes(p: Problem, variant: str = "auto") -> int:
    d = make_desc(p, None, variant)
    return int(lib().laga_mla_fwd_workspace_size(ctypes.byref(d)))


def bwd_workspace_bytes(p: Problem, variant: str = "auto") -> int:
    d = make_desc(p, None, variant)
    return int(lib().laga_mla_bwd_workspace_size(ctypes.byref(d)))


def _workspace(nbytes: int, device, given: torch.Tensor | None) -> torch.Tensor | None:
    if nbytes == 0:
        return None
    if given is not None:
        if given.numel() * given.element_size() < nbytes:
            raise ValueError("workspace too small")
        return given
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def fwd(q, c_kv, k_rope, W_UK, W_UV, q_offset: int = 0, causal: bool = True, softmax_scale: float | None = None,
        variant: str = "auto", workspace: torch.Tensor | None = None, out=None, lse=None, q_split: int = 0,
        q_offset2: int = 0, kv_prebuilt: bool = False):
    """laga_mla_fwd: returns (out [B,Sq,n_h,d_v], lse [B,n_h,Sq] fp32).

    kv_prebuilt=True (LAGA_FLAG_KV_PREBUILT): `workspace` already holds K_nope / V
    for every row the forward reads, from reconstruct_rows calls with the same
    arguments; the call runs the attention alone."""
    p = problem_of(q, c_kv, k_rope, W_UK, W_UV, q_offset, causal, q_split, q_offset2)
    if kv_prebuilt and workspace is None:
        raise ValueError("kv_prebuilt needs the workspace the rows were rebuilt into")
    d = make_desc(p, softmax_scale, variant, FLAG_KV_PREBUILT if kv_prebuilt else 0)
    L = lib()
    dev = q.device
    if out is None:
        out = torch.empty((p.B, p.Sq, p.n_h, p.d_v), dtype=q.dtype, device=dev)
    if lse is None:
        lse = torch.empty((p.B, p.n_h, p.Sq), dtype=torch.float32, device=dev)
    nbytes = int(L.laga_mla_fwd_workspace_size(ctypes.byref(d)))
    ws = _workspace(nbytes, dev, workspace)
    _raise_if(L.laga_mla_fwd(ctypes.byref(d), _ptr(q), _ptr(c_kv), _ptr(k_rope), _ptr(W_UK), _ptr(W_UV),
                             _ptr(out), _ptr(lse), _ptr(ws), nbytes, _stream(dev)))
    return out, lse


def bwd(q, c_kv, k_rope, W_UK, W_UV, out, lse, dout, q_offset: int = 0, causal: bool = True,
        softmax_scale: float | None = None, variant: str = "auto", workspace: torch.Tensor | None = None,
        grads: dict | None = None, reuse_kv: bool = False, q_split: int = 0, q_offset2: int = 0):
    """laga_mla_bwd: returns dict dq, dc_kv, dk_rope, dW_UK, dW_UV.

    reuse_kv=True (LAGA_FLAG_REUSE_KV): `workspace` is the buffer the forward
    ran with, still holding the K_nope/V it rebuilt; the backward reads them
    instead of rebuilding them."""
    p = problem_of(q, c_kv, k_rope, W_UK, W_UV, q_offset, causal, q_split, q_offset2)
    for t in (out, lse, dout):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("out, lse and dout must be contiguous CUDA tensors")
    if reuse_kv and workspace is None:
        raise ValueError("reuse_kv needs the workspace the forward ran with")
    d = make_desc(p, softmax_scale, variant, FLAG_REUSE_KV if reuse_kv else 0)
    L = lib()
    dev = q.device
    g = grads if grads is not None else {
        "dq": torch.empty_like(q), "dc_kv": torch.empty_like(c_kv), "dk_rope": torch.empty_like(k_rope),
        "dW_UK": torch.empty_like(W_UK), "dW_UV": torch.empty_like(W_UV)}
    nbytes = int(L.laga_mla_bwd_workspace_size(ctypes.byref(d)))
    ws = _workspace(nbytes, dev, workspace)
    _raise_if(L.laga_mla_bwd(ctypes.byref(d), _ptr(q), _ptr(c_kv), _ptr(k_rope), _ptr(W_UK), _ptr(W_UV),
                             _ptr(out), _ptr(lse), _ptr(dout), _ptr(g["dq"]), _ptr(g["dc_kv"]), _ptr(g["dk_rope"]),
                             _ptr(g["dW_UK"]), _ptr(g["dW_UV"]), _ptr(ws), nbytes, _stream(dev)))
    return g


def reconstruct_rows(q, c_kv, k_rope, W_UK, W_UV, row0: int, rows: int, workspace: torch.Tensor,
                     q_offset: int = 0, causal: bool = True, q_split: int = 0, q_offset2: int = 0,
                     variant: str = "auto"):
    """laga_mla_reconstruct_rows: the forward's K/V rebuild for latent rows
    [row0, row0 + rows) into `workspace` (of at least fwd_workspace_bytes), for a
    later fwd(..., workspace=workspace, kv_prebuilt=True) with the same arguments.
    row0 a multiple of 128; row0 + rows a multiple of 128 or past the last row any
    query sees."""
    p = problem_of(q, c_kv, k_rope, W_UK, W_UV, q_offset, causal, q_split, q_offset2)
    d = make_desc(p, None, variant)
    nbytes = workspace.numel() * workspace.element_size()
    _raise_if(lib().laga_mla_reconstruct_rows(ctypes.byref(d), _ptr(c_kv), _ptr(W_UK), _ptr(W_UV), int(row0),
                                              int(rows), _ptr(workspace), nbytes, _stream(q.device)))


def absorbed_fwd(q, c_kv, k_rope, W_UK, W_UV, q_offset: int = 0, causal: bool = True,
                 softmax_scale: float | None = None, workspace: torch.Tensor | None = None, out=None, lse=None):
    """laga_mla_absorbed_fwd (the absorbed MLA form, for comparison): returns
    (out [B,Sq,n_h,d_v], lse [B,n_h,Sq] fp32). The workspace holds the form's
    intermediates q_lat and ctx ([B,Sq,n_h,d_c] each)."""
    p = problem_of(q, c_kv, k_rope, W_UK, W_UV, q_offset, causal)
    d = make_desc(p, softmax_scale)
    L = lib()
    dev = q.device
    if out is None:
        out = torch.empty((p.B, p.Sq, p.n_h, p.d_v), dtype=q.dtype, device=dev)
    if lse is None:
        lse = torch.empty((p.B, p.n_h, p.Sq), dtype=torch.float32, device=dev)
    nbytes = int(L.laga_mla_absorbed_fwd_workspace_size(ctypes.byref(d)))
    if nbytes == 0:
        _raise_if(L.laga_mla_absorbed_fwd(ctypes.byref(d), None, None, None, None, None, None, None, None, 0,
                                          _stream(dev)))
    ws = _workspace(nbytes, dev, workspace)
    _raise_if(L.laga_mla_absorbed_fwd(ctypes.byref(d), _ptr(q), _ptr(c_kv), _ptr(k_rope), _ptr(W_UK), _ptr(W_UV),
                                      _ptr(out), _ptr(lse), _ptr(ws), nbytes, _stream(dev)))
    return out, lse


def absorbed_workspace_bytes(p: Problem) -> int:
    d = make_desc(p)
    return int(lib().laga_mla_absorbed_fwd_workspace_size(ctypes.byref(d)))


def reconstruct(c_kv, W_UK, W_UV, n_h: int, variant: str = "auto"):
    """laga_mla_reconstruct: per-head K_nope [B,S,n_h,d_nope] and V [B,S,n_h,d_v]."""
    B, S, d_c = c_kv.shape
    d_nope, d_v = W_UK.shape[1] // n_h, W_UV.shape[1] // n_h
    dt = {torch.float32: "f32", torch.bfloat16: "bf16"}[c_kv.dtype]
    p = Problem(B=B, Sq=1, S=S, n_h=n_h, d_c=d_c, d_nope=d_nope, d_rope=64 if dt == "bf16" else 0, d_v=d_v,
                q_offset=0, causal=False, dtype=dt)
    d = make_desc(p, None, variant)
    kn = torch.empty((B, S, n_h, d_nope), dtype=c_kv.dtype, device=c_kv.device)
    v = torch.empty((B, S, n_h, d_v), dtype=c_kv.dtype, device=c_kv.device)
    _raise_if(lib().laga_mla_reconstruct(ctypes.byref(d), _ptr(c_kv), _ptr(W_UK), _ptr(W_UV), _ptr(kn), _ptr(v),
                                         _stream(c_kv.device)))
    return kn, v


def check(device=None) -> None:
    """laga_mla_check on the current stream: raise on a device-side timeout or CUDA error."""
    dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
    _raise_if(lib().laga_mla_check(_stream(dev)))


def selftest_timeout(device=None) -> None:
    """laga_mla_selftest_timeout on the current stream: enqueue a kernel whose
    bounded wait expires (about 2 s); the next check() raises LAGA_ERR_TIMEOUT."""
    dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
    _raise_if(lib().laga_mla_selftest_timeout(_stream(dev)))


@dataclass
class StepBuffers:
    """Preallocated device buffers for repeated forward+backward steps of one
    problem. One workspace serves both calls: the backward reuses the K_nope/V
    the forward left in it."""
    p: Problem
    inputs: dict
    out: torch.Tensor
    lse: torch.Tensor
    grads: dict
    ws: torch.Tensor | None


def alloc_step(p: Problem, inputs: dict, variant: str = "auto") -> StepBuffers:
    dev = inputs["q"].device
    dt = inputs["q"].dtype
    out = torch.empty((p.B, p.Sq, p.n_h, p.d_v), dtype=dt, device=dev)
    lse = torch.empty((p.B, p.n_h, p.Sq), dtype=torch.float32, device=dev)
    grads = {"dq": torch.empty_like(inputs["q"]), "dc_kv": torch.empty_like(inputs["c_kv"]),
             "dk_rope": torch.empty_like(inputs["k_rope"]), "dW_UK": torch.empty_like(inputs["W_UK"]),
             "dW_UV": torch.empty_like(inputs["W_UV"])}
    nb = max(fwd_workspace_bytes(p, variant), bwd_workspace_bytes(p, variant))
    ws = torch.empty(nb, dtype=torch.uint8, device=dev) if nb else None
    return StepBuffers(p, inputs, out, lse, grads, ws)


def step(buf: StepBuffers, variant: str = "auto"):
    """One forward + backward pass of the attention block into preallocated buffers."""
    x, p = buf.inputs, buf.p
    fwd(x["q"], x["c_kv"], x["k_rope"], x["W_UK"], x["W_UV"], p.q_offset, p.causal, None, variant,
        buf.ws, buf.out, buf.lse, p.q_split, p.q_offset2)
    bwd(x["q"], x["c_kv"], x["k_rope"], x["W_UK"], x["W_UV"], buf.out, buf.lse, x["dout"], p.q_offset, p.causal,
        None, variant, buf.ws, buf.grads, reuse_kv=buf.ws is not None, q_split=p.q_split, q_offset2=p.q_offset2)
    return buf.out, buf.lse, buf.grads
