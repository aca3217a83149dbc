"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

This module only draws random numbers and rounds them to the storage type; it
holds none of the method's arithmetic, and neither the oracle nor the CUDA
path is imported here.

Recipe (the configurations' stated distributions): q, c_kv, k_rope and dout
are N(0, 1); W_UK and W_UV are N(0, 1/d_c) (variance 1/d_c, std 1/sqrt(d_c)).
Values are drawn in fp32 from NumPy's PCG64 in the fixed order q, c_kv, k_rope,
W_UK, W_UV, dout, then rounded to bf16 (round to nearest even) when the
problem's storage type is bf16. Arrays are returned as float32 holding exactly
representable values, so the fp64 upcast the oracle makes is exact.
"""
from __future__ import annotations

import numpy as np

from .configs import Problem


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); returns float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16) << 16
    return r.astype(np.uint32).view(np.float32)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """The upper 16 bits of float32 values that are already bf16-representable."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)


def make_inputs(p: Problem, seed: int, with_dout: bool = True) -> dict:
    """Draw one problem's inputs. Shapes follow the library's dense row-major layouts:

    q [B,Sq,n_h,d_nope+d_rope] (no-RoPE part first), c_kv [B,S,d_c],
    k_rope [B,S,d_rope], W_UK [d_c,n_h*d_nope], W_UV [d_c,n_h*d_v],
    dout [B,Sq,n_h,d_v].
    """
    g = np.random.Generator(np.random.PCG64(seed))
    f32 = np.float32

    def normal(shape, std=1.0):
        a = g.standard_normal(size=shape, dtype=f32)
        if std != 1.0:
            a *= f32(std)
        return a

    w_std = 1.0 / np.sqrt(p.d_c)
    out = {
        "q": normal((p.B, p.Sq, p.n_h, p.d_qk)),
        "c_kv": normal((p.B, p.S, p.d_c)),
        "k_rope": normal((p.B, p.S, p.d_rope)),
        "W_UK": normal((p.d_c, p.n_h * p.d_nope), w_std),
        "W_UV": normal((p.d_c, p.n_h * p.d_v), w_std),
    }
    if with_dout:
        out["dout"] = normal((p.B, p.Sq, p.n_h, p.d_v))
    if p.dtype == "bf16":
        out = {k: round_to_bf16(v) for k, v in out.items()}
    return out


def seed_for(config_index: int, rank: int = 0) -> int:
    """Seed convention: configuration index x 1000 + SP rank."""
    return config_index * 1000 + rank
