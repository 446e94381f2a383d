"""The allocation-free forward entry point (usp_attention_fwd_noalloc).

Some hosts cannot hand this library a workspace: code under a framework whose
caching allocator owns the device memory, and latency-critical request paths
that must not call cudaMalloc/cudaFree.  For them the library keeps a fixed
64 MiB scratch array of its own.  These tests call the entry point through the
C ABI, each case twice in a row on different inputs, and check every result
against the ordinary usp_attention_fwd (materialised, caller-provided
workspace): both run the same deterministic kernels, so the results must be
identical bit for bit.  The fp32 case (the handbook's four-card demo shape,
Ulysses 4, no ring merge) is also checked against the CPU oracle at the demo's
1e-5 bound, and one bf16 case is sized so its workspace reaches almost to the
end of the array.  The file sits where pytest collects it last and must pass
both alone and after the other tests.
"""
import math

import numpy as np
import pytest
import torch

from diffusion_transformer_sequence_gb300 import workloads as wl
from tests.helpers import F32_ATOL, ensure_built, f64

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 64 << 20


def _stacks(w):
    inp = wl.make_inputs(w, with_dout=False)
    return [wl.to_token_stack(inp[n], w.ulysses, w.ring).cuda() for n in ("q", "k", "v")]


def _noalloc(L, _lib, w, q, k, v):
    out = torch.full_like(q, float("nan"))
    lse = torch.full(w.lse_stack_shape, float("nan"), dtype=torch.float32, device="cuda")
    dt = _lib.USP_BF16 if w.dtype == "bf16" else _lib.USP_F32
    st = L.usp_attention_fwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                     w.B, w.H, w.N, w.D, w.ulysses, w.ring, w.scale, dt,
                                     torch.cuda.current_stream().cuda_stream)
    assert st == _lib.USP_OK, L.usp_status_string(st)
    return out, lse


def _largest_fitting_bf16_n(L, _lib, H=8, u=2, r=2):
    """The largest N (a multiple of u*r) whose materialised workspace still fits the array
    (found by bisection over the library's own workspace query)."""
    sp = u * r
    need = lambda n: L.usp_attention_workspace_bytes(1, H, n * sp, 128, u, r, _lib.USP_BF16,
                                                     _lib.USP_MATERIALISED, 0)
    lo, hi = 1, 2
    assert 0 < need(lo) <= SCRATCH_BYTES
    while need(hi) <= SCRATCH_BYTES:
        lo, hi = hi, 2 * hi
    while hi - lo > 1:                       # need(lo) fits, need(hi) does not
        mid = (lo + hi) // 2
        lo, hi = (mid, hi) if need(mid) <= SCRATCH_BYTES else (lo, mid)
    return lo * sp, need(lo)


def _cases(L, _lib):
    n_big, _ = _largest_fitting_bf16_n(L, _lib)
    return [
        ("bf16 u2 r2", lambda s: wl.custom("noalloc", "bf16", 1, 4, 1024, 128, 2, 2, seed=s)),
        ("fp32 demo u4 r1", lambda s: wl.custom("noalloc32", "f32", 1, 8, 256, 32, 4, 1, seed=s)),
        (f"bf16 u2 r2 N{n_big} (array almost full)",
         lambda s: wl.custom("noalloc_big", "bf16", 1, 8, n_big, 128, 2, 2, seed=s)),
    ]


def test_noalloc_bitwise_equal_to_workspace_entry_point_twice():
    ensure_built()
    import oracle
    import diffusion_transformer_sequence_gb300 as usp
    from diffusion_transformer_sequence_gb300 import _lib
    L = usp.lib()
    for what, make in _cases(L, _lib):
        for seed in (21, 22):                  # two calls in a row, different data
            w = make(seed)
            q, k, v = _stacks(w)
            out, lse = _noalloc(L, _lib, w, q, k, v)
            assert usp.device_status() == 0
            ref_o, ref_l = usp.attention_fwd(q, k, v, w.ulysses, w.ring, w.scale, mode="materialised")
            torch.cuda.synchronize()
            assert torch.equal(out, ref_o), f"{what}, seed {seed}: out differs from the workspace call"
            assert torch.equal(lse, ref_l), f"{what}, seed {seed}: lse differs from the workspace call"
            if w.dtype == "f32":
                ro, rl = oracle.usp_forward(*(f64(t) for t in (q, k, v)), w.ulysses, w.ring, w.scale)
                assert np.abs(f64(out) - ro).max() <= F32_ATOL, what
                assert np.abs(f64(lse) - rl).max() <= F32_ATOL, what


def test_noalloc_largest_case_reaches_the_end_of_the_array():
    ensure_built()
    import diffusion_transformer_sequence_gb300 as usp
    from diffusion_transformer_sequence_gb300 import _lib
    L = usp.lib()
    n, need = _largest_fitting_bf16_n(L, _lib)
    assert need > SCRATCH_BYTES - (2 << 20), f"workspace {need} is not close to the 64 MiB end"
    n2 = n + 4
    assert L.usp_attention_workspace_bytes(1, 8, n2, 128, 2, 2, _lib.USP_BF16, _lib.USP_MATERIALISED, 0) \
        > SCRATCH_BYTES


def test_noalloc_rejects_problems_beyond_its_scratch():
    ensure_built()
    import diffusion_transformer_sequence_gb300 as usp
    from diffusion_transformer_sequence_gb300 import _lib
    L = usp.lib()
    s = 1 / math.sqrt(128)
    # Qwen-Image 2048^2 (u4) needs ~404 MB of workspace: more than the 64 MiB array.
    st = L.usp_attention_fwd_noalloc(0x10000, 0x10000, 0x10000, 0x10000, 0x10000, 1, 24, 16384, 128, 4, 1,
                                     s, _lib.USP_BF16, None)
    assert st == _lib.USP_ERR_WORKSPACE
    # an invalid argument is reported as the workspace call reports it, before the size check
    st = L.usp_attention_fwd_noalloc(0x10000, 0x10000, 0x10000, 0x10000, 0x10000, 1, 24, 16384, 128, 5, 1,
                                     s, _lib.USP_BF16, None)
    assert st == _lib.USP_ERR_DIVISIBILITY
    st = L.usp_attention_fwd_noalloc(0x10000, 0x10000, 0x10000, 0x10001, 0x10000, 1, 24, 16384, 128, 4, 1,
                                     s, _lib.USP_BF16, None)
    assert st == _lib.USP_ERR_INVALID_ARG
    st = L.usp_attention_fwd_noalloc(0x10000, 0x10000, 0x10000, 0x10000, 0x10000, 1, 65536, 16384, 128, 1, 1,
                                     s, _lib.USP_BF16, None)
    assert st == _lib.USP_ERR_UNSUPPORTED
