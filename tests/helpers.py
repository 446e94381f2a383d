"""Shared test helpers: building the library, widening inputs for the oracle,
tolerance checks and guard canaries.  No method arithmetic lives here."""
from __future__ import annotations

import numpy as np
import torch

# Tolerances against the fp64 oracle (bf16 bounds are the stated ones; the
# fp32 bound is the handbook demo's allclose atol).
F32_ATOL = 1e-5
BF16_O_ATOL = 2e-2
BF16_LSE_RTOL = 1e-3
# Gradients (no stated bound): relative to the largest reference magnitude.
BF16_GRAD_REL = 2e-2
F32_GRAD_ATOL = 1e-5


def ensure_built():
    from diffusion_transformer_sequence_gb300 import build
    return build.build()


def f64(t: torch.Tensor) -> np.ndarray:
    """Exact widening of a CPU/GPU tensor to a float64 numpy array."""
    return t.detach().to("cpu").to(torch.float64).numpy()


def bits(t: torch.Tensor) -> np.ndarray:
    """The raw bit pattern (for bit-exact comparisons of re-layouts)."""
    t = t.detach().to("cpu").contiguous()
    view = {2: torch.int16, 4: torch.int32, 1: torch.uint8, 8: torch.int64}[t.element_size()]
    return t.view(view).numpy()


def check_out(got_o, got_l, ref_o, ref_l, dtype: str, what: str = ""):
    """Assert GPU (out, lse) agree with the fp64 oracle within the stated bounds."""
    go, gl = f64(got_o), f64(got_l)
    assert np.isfinite(go).all() and np.isfinite(gl).all(), f"{what}: non-finite output"
    eo = np.abs(go - ref_o).max() if go.size else 0.0
    if dtype == "f32":
        el = np.abs(gl - ref_l).max() if gl.size else 0.0
        assert eo <= F32_ATOL, f"{what}: max |dO| {eo:.3e} > {F32_ATOL}"
        assert el <= F32_ATOL, f"{what}: max |dLSE| {el:.3e} > {F32_ATOL}"
    else:
        el = (np.abs(gl - ref_l) / np.maximum(np.abs(ref_l), 1e-30)).max() if gl.size else 0.0
        assert eo <= BF16_O_ATOL, f"{what}: max |dO| {eo:.3e} > {BF16_O_ATOL}"
        assert el <= BF16_LSE_RTOL, f"{what}: max rel dLSE {el:.3e} > {BF16_LSE_RTOL}"
    return eo, el


class Canary:
    """A device buffer with poisoned guard regions on both sides of the view
    handed to a kernel; :meth:`check` asserts the guards are untouched."""

    PAD = 4096  # bytes on each side

    def __init__(self, shape, dtype, device="cuda"):
        n = int(np.prod(shape)) if len(shape) else 1
        esz = torch.tensor([], dtype=dtype).element_size()
        pad = self.PAD // esz
        self.raw = torch.empty(n + 2 * pad, dtype=dtype, device=device)
        self.raw.view(torch.uint8 if esz == 1 else {2: torch.int16, 4: torch.int32}[esz]).fill_(0x5A5A5A5A if esz == 4 else 0x5A5A if esz == 2 else 0x5A)
        self.pad = pad
        self.n = n
        self.view = self.raw[pad:pad + n].view(shape)
        self._guard = self.raw[:pad].clone(), self.raw[pad + n:].clone()

    def check(self):
        a, b = self._guard
        assert torch.equal(self.raw[:self.pad].view(torch.uint8), a.view(torch.uint8)), "guard before buffer overwritten"
        assert torch.equal(self.raw[self.pad + self.n:].view(torch.uint8), b.view(torch.uint8)), "guard after buffer overwritten"
