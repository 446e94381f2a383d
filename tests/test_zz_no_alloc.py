"""The allocation-free forward entry point (usp_attention_fwd_noalloc).

Some hosts cannot hand this library a workspace: code under a framework whose
caching allocator owns the device memory, and latency-critical request paths
that must not call cudaMalloc/cudaFree.  For them the library keeps a fixed
64 MiB scratch array of its own.  This test calls the entry point through the
C ABI twice in a row on different inputs and checks each result against the
ordinary usp_attention_fwd (materialised, caller-provided workspace) within the
bf16 tolerances the other parity tests use.  It sits in a file of its own that
pytest collects last, and must pass both alone and after the other tests.
"""
import math

import numpy as np
import pytest
import torch

from diffusion_transformer_sequence_gb300 import workloads as wl
from tests.helpers import BF16_LSE_RTOL, BF16_O_ATOL, ensure_built, f64

pytestmark = pytest.mark.gpu


def _inputs(seed):
    w = wl.custom("noalloc", "bf16", 1, 4, 1024, 128, 2, 2, seed=seed)
    inp = wl.make_inputs(w)
    return w, [wl.to_token_stack(inp[n], w.ulysses, w.ring).cuda() for n in ("q", "k", "v")]


def test_noalloc_matches_workspace_entry_point_twice():
    ensure_built()
    import diffusion_transformer_sequence_gb300 as usp
    from diffusion_transformer_sequence_gb300 import _lib
    L = usp.lib()
    stream = torch.cuda.current_stream().cuda_stream
    for seed in (21, 22):                      # two calls in a row, different data
        w, (q, k, v) = _inputs(seed)
        out = torch.empty_like(q)
        lse = torch.empty(w.lse_stack_shape, dtype=torch.float32, device="cuda")
        st = L.usp_attention_fwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                         w.B, w.H, w.N, w.D, w.ulysses, w.ring, w.scale, _lib.USP_BF16, stream)
        assert st == _lib.USP_OK, L.usp_status_string(st)
        assert usp.device_status() == 0
        ref_o, ref_l = usp.attention_fwd(q, k, v, w.ulysses, w.ring, w.scale, mode="materialised")
        torch.cuda.synchronize()
        assert np.abs(f64(out) - f64(ref_o)).max() <= BF16_O_ATOL
        assert (np.abs(f64(lse) - f64(ref_l)) / np.abs(f64(ref_l))).max() <= BF16_LSE_RTOL


def test_noalloc_rejects_problems_beyond_its_scratch():
    ensure_built()
    import diffusion_transformer_sequence_gb300 as usp
    from diffusion_transformer_sequence_gb300 import _lib
    L = usp.lib()
    # Qwen-Image 2048^2 (u4) needs ~404 MB of workspace: more than the 64 MiB array.
    st = L.usp_attention_fwd_noalloc(0x10000, 0x10000, 0x10000, 0x10000, 0x10000, 1, 24, 16384, 128, 4, 1,
                                     1 / math.sqrt(128), _lib.USP_BF16, None)
    assert st == _lib.USP_ERR_WORKSPACE
