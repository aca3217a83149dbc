"""fp64 CPU oracle of the LAGA MLA attention block: test infrastructure only.

Only the tests, the smoke check and the benchmark's CPU-baseline leg use it;
the library's compute path never imports it.
"""
from .laga_oracle import (  # noqa: F401
    default_scale, reconstruct, reconstruct_head, head_key, query_positions, visible_mask,
    attention_head_forward, attention_head_backward, mla_forward_head, mla_forward,
    mla_backward_head, mla_backward, absorbed_forward, absorbed_backward,
)
