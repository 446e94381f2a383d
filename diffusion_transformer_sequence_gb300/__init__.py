"""GB300-native USP (Ulysses x Ring) attention: C-ABI library + thin binding.

The compute path lives in ``libusp.so`` (``csrc/``, declared in
``include/usp.h``); this package only loads it and marshals torch tensors.
"""
from .api import (  # noqa: F401
    attention_bwd,
    attention_fwd,
    attention_fwd_fp8,
    attention_fwd_joint,
    attn_chunk_fwd,
    cross_attention_fwd,
    device_status,
    joint_workspace_bytes,
    lse_merge,
    quantize_e4m3,
    relayout_head2tok,
    relayout_tok2head,
    set_spin_limit,
    workspace_bytes,
)
from ._lib import UspError, lib  # noqa: F401
