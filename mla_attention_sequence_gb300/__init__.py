"""LAGA (Latent All-Gather Attention) MLA attention block for one GB300 GPU.

The compute runs in liblaga_mla.so (C ABI, include/laga_mla.h): tcgen05/TMEM/TMA
kernels for the bf16 DeepSeek-V3 dimensions and fp32 CUDA-core kernels for any
other widths. `laga` is the thin torch binding; `configs` and `synth` hold the
problem shapes and the seeded synthetic inputs.
"""
from .configs import Problem  # noqa: F401

__all__ = ["Problem", "laga", "configs", "synth", "build"]
