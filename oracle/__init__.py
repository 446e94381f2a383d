"""CPU oracle for the USP attention step -- TEST INFRASTRUCTURE ONLY.

Plain fp64 numpy statement of the method (see ``usp_oracle``) plus a spawn
process pool for checking sampled rows of large workloads (``pool``).  Only
``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and
reference legs may import it; the library under
``diffusion_transformer_sequence_gb300`` never does.
"""
from .usp_oracle import (  # noqa: F401
    attention,
    attention_bwd,
    attention_bwd_sampled,
    attention_rows,
    e4m3_round,
    head2tok,
    lse_merge,
    quantize_e4m3_heads,
    ring_chunk,
    tok2head,
    usp_cross_attention,
    usp_forward,
    usp_forward_fp8,
    usp_forward_joint,
)
