"""Seeded synthetic workloads for the USP attention step.

This module holds the five workload shapes, the seeded input generators and
the sampled-row selection.  It contains none of the method's arithmetic: it
only draws iid N(0,1) values and places them in the token-sharded layout that
the boundary defines, so both the CUDA path and the CPU oracle can be fed
from it without sharing any computation.

Shapes follow the workloads the pages measure or name:

* ``demo``   -- "Multi-GPU parallelism: spreading one step over several
  cards", section "Sequence parallelism: Ulysses and Ring": the four-card
  Ulysses simulation with B=1, H=8, N=256, D=32, P=4, fp32, drawn with
  ``torch.manual_seed(0)`` and three ``randn`` calls in the order q, k, v.
* ``qwen1024`` -- Qwen-Image 1024x1024 (vllm-omni parallelism guide,
  "Hybrid Ulysses + Ring" benchmark), hybrid Ulysses 2 x Ring 2.
* ``qwen2048`` -- Qwen-Image 2048x2048 (vllm-omni guide, "Ulysses-SP"
  benchmark), Ulysses 4.
* ``wan_s32k`` -- the "Wan shapes" B1 H40 S32768 D128 of the USP PR page,
  Design, "Ring kernel selection"; Ulysses 8 x Ring 4, forward + backward.
* ``wan720p``  -- Wan 720p 81-frame latent (21x45x80 tokens after (1,2,2)
  patchify) from the handbook's communication table, Ulysses 8 x Ring 2.

Token-sharded stack layout (the boundary's input layout): a tensor of global
shape [B, H, N, D] is stored as [ring, ulysses, B, H, Ns, D] with
Ns = N / (ulysses * ring); virtual rank (g, j) has sp_rank = g * ulysses + j
and holds tokens [sp_rank * Ns, (sp_rank + 1) * Ns) of every head (Ulysses
ranks contiguous, ring ranks strided, as in the USP PR page, Design,
"Coordinates").
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    dtype: str          # "f32" or "bf16": the dtype the inputs are stored in
    B: int
    H: int
    N: int
    D: int
    ulysses: int
    ring: int
    backward: bool
    seed: int
    row_seed: int
    description: str
    Nt: int = 0         # replicated text tokens of joint attention (0: image only)

    @property
    def sp(self) -> int:
        return self.ulysses * self.ring

    @property
    def Ns(self) -> int:
        return self.N // self.sp

    @property
    def Nr(self) -> int:
        return self.N // self.ring

    @property
    def Hu(self) -> int:
        return self.H // self.ulysses

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def elt(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def stack_shape(self) -> tuple:
        return (self.ring, self.ulysses, self.B, self.H, self.Ns, self.D)

    @property
    def lse_stack_shape(self) -> tuple:
        return (self.ring, self.ulysses, self.B, self.H, self.Ns)

    @property
    def t_bytes(self) -> int:
        return self.B * self.H * self.N * self.D * self.elt

    @property
    def fwd_flop(self) -> float:
        """Algorithmic forward FLOP of non-causal attention: 4*B*H*N^2*D."""
        return 4.0 * self.B * self.H * self.N * self.N * self.D

    def joint_flop(self, text_queries: bool = True) -> float:
        """Algorithmic FLOP of joint attention: every image (and text) query
        against all N + Nt keys, 4 FLOP per query-key-dim."""
        nq = self.N + (self.Nt if text_queries else 0)
        return 4.0 * self.B * self.H * nq * (self.N + self.Nt) * self.D

    @property
    def bwd_flop(self) -> float:
        """Algorithmic backward FLOP: 10*B*H*N^2*D (five N x N x D GEMMs)."""
        return 10.0 * self.B * self.H * self.N * self.N * self.D


WORKLOADS = {
    "demo": Workload("demo", "f32", 1, 8, 256, 32, 4, 1, False, 0, 2000,
                     "fp32 B1 H8 N256 D32 Ulysses P=4 (handbook four-card simulation)"),
    "qwen1024": Workload("qwen1024", "bf16", 1, 24, 4096, 128, 2, 2, False, 1001, 2001,
                         "bf16 B1 H24 N4096 D128 ulysses2 x ring2 (Qwen-Image 1024^2)"),
    "qwen2048": Workload("qwen2048", "bf16", 1, 24, 16384, 128, 4, 1, False, 1002, 2002,
                         "bf16 B1 H24 N16384 D128 ulysses4 (Qwen-Image 2048^2)"),
    "wan_s32k": Workload("wan_s32k", "bf16", 1, 40, 32768, 128, 8, 4, True, 1003, 2003,
                         "bf16 B1 H40 N32768 D128 ulysses8 x ring4, fwd+bwd (Wan shapes)"),
    "wan720p": Workload("wan720p", "bf16", 1, 40, 75600, 128, 8, 2, False, 1004, 2004,
                        "bf16 B1 H40 N75600 D128 ulysses8 x ring2 (Wan 720p 81 frames)"),
    # Joint text + image attention: the handbook's per-layer communication
    # table counts FLUX 1024^2 as 4608 tokens and Wan 720p 81 frames as 76112,
    # i.e. the image tokens plus 512 text tokens, which the vllm-omni guide
    # ("How to parallelize a new model") keeps replicated on every SP rank.
    "qwen1024_joint": Workload("qwen1024_joint", "bf16", 1, 24, 4096, 128, 2, 2, False, 1005, 2005,
                               "bf16 B1 H24 N4096+512 text D128 ulysses2 x ring2 (joint, 4608 tokens)", 512),
    "wan720p_joint": Workload("wan720p_joint", "bf16", 1, 40, 75600, 128, 8, 2, False, 1006, 2006,
                              "bf16 B1 H40 N75600+512 text D128 ulysses8 x ring2 (joint, 76112 tokens)", 512),
}

ORDER = ["demo", "qwen1024", "qwen2048", "wan_s32k", "wan720p"]
JOINT = ["qwen1024_joint", "wan720p_joint"]


def custom(name, dtype, B, H, N, D, ulysses, ring, seed=7, backward=False, Nt=0) -> Workload:
    """A workload of arbitrary shape (used by tests for ragged and edge cases)."""
    return Workload(name, dtype, B, H, N, D, ulysses, ring, backward, seed, seed + 1000,
                    f"{dtype} B{B} H{H} N{N} D{D} u{ulysses} r{ring}" + (f" Nt{Nt}" if Nt else ""), Nt)


def to_token_stack(x: torch.Tensor, ulysses: int, ring: int) -> torch.Tensor:
    """Place a global [B,H,N,D] (or [B,H,N]) tensor in the token-sharded stack.

    Virtual rank sp_rank takes the contiguous token slice
    [sp_rank*Ns, (sp_rank+1)*Ns) of every head, the same token split as the
    handbook's four-card simulation (card r takes the r-th of P equal token
    segments).  This is data
    placement of the inputs, not a step of the method.
    """
    sp = ulysses * ring
    B, H, N = x.shape[:3]
    Ns = N // sp
    tail = tuple(x.shape[3:])
    y = x.reshape(B, H, sp, Ns, *tail).movedim(2, 0).contiguous()
    return y.reshape(ring, ulysses, B, H, Ns, *tail)


def from_token_stack(t: torch.Tensor) -> torch.Tensor:
    """Inverse of :func:`to_token_stack`: stack [r,u,B,H,Ns,...] -> [B,H,N,...]."""
    r, u, B, H, Ns = t.shape[:5]
    tail = tuple(t.shape[5:])
    y = t.reshape(r * u, B, H, Ns, *tail).movedim(0, 2).contiguous()
    return y.reshape(B, H, r * u * Ns, *tail)


def make_inputs(w: Workload, with_dout: bool | None = None):
    """Draw q, k, v (and dO when the workload has a backward) for ``w``.

    Returns a dict of CPU tensors in ``w.torch_dtype`` holding the GLOBAL
    [B,H,N,D] tensors.  Values are iid N(0,1) from a CPU generator seeded
    with ``w.seed``, drawn in fp32 in the order q, k, v, dO and then cast
    (a bf16 cast rounds to nearest even; the oracle reads the cast values).
    For the handbook demo this reproduces ``torch.manual_seed(0)`` followed
    by three ``torch.randn(1, 8, 256, 32)`` calls.
    """
    if with_dout is None:
        with_dout = w.backward
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    names = ["q", "k", "v"] + (["dout"] if with_dout else [])
    out = {}
    for n in names:
        x = torch.randn(w.B, w.H, w.N, w.D, generator=g, dtype=torch.float32)
        out[n] = x.to(w.torch_dtype)
    return out


def sample_rows(w: Workload, count: int = 4096) -> torch.Tensor:
    """Seeded global query (or key) rows to check on large workloads.

    Always includes row 0, row N-1, every shard boundary +-1 (multiples of
    Ns and of Nr), the 128-row tile edges 127/128 inside each shard, and
    random rows from a generator seeded with ``w.row_seed`` up to ``count``.
    Returns a sorted int64 tensor of unique rows in [0, N).
    """
    N = w.N
    special = {0, N - 1}
    for step in (w.Ns, w.Nr):
        for b in range(0, N + 1, step):
            for d in (-1, 0, 1):
                if 0 <= b + d < N:
                    special.add(b + d)
    for s0 in range(0, N, w.Ns):
        for d in (127, 128, w.Ns - 1 - 127, w.Ns - 128):
            if 0 <= d < w.Ns:
                special.add(s0 + d)
    rows = set(special)
    if count >= N:
        return torch.arange(N, dtype=torch.int64)
    g = torch.Generator(device="cpu")
    g.manual_seed(w.row_seed)
    perm = torch.randperm(N, generator=g)
    i = 0
    while len(rows) < count and i < N:
        rows.add(int(perm[i]))
        i += 1
    return torch.tensor(sorted(rows), dtype=torch.int64)


def make_text_inputs(w: Workload):
    """Draw the replicated text tensors q_txt, k_txt, v_txt [B, H, Nt, D].

    iid N(0,1) from a CPU generator seeded with ``w.seed + 7919`` (drawn in
    fp32 in the order q_txt, k_txt, v_txt, then cast), independent of the
    image draws of :func:`make_inputs`.
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed + 7919)
    out = {}
    for n in ("q_txt", "k_txt", "v_txt"):
        x = torch.randn(w.B, w.H, w.Nt, w.D, generator=g, dtype=torch.float32)
        out[n] = x.to(w.torch_dtype)
    return out
