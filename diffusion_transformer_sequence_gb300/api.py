"""Python binding of libusp: argument marshalling only.

Every function takes torch tensors, checks shapes on the host, and calls the
C ABI entry point of the same name on the current CUDA stream.  All compute
runs in libusp's kernels; torch only provides device memory and the stream.
:func:`attention_fwd` and :func:`attention_bwd` also accept CPU tensors: the
inputs are copied to the device (through pinned memory) and the results
copied back, which is the end-to-end path a host caller uses.
"""
from __future__ import annotations

import math

import torch

from . import _lib
from ._lib import check

_DT = {torch.float32: _lib.USP_F32, torch.bfloat16: _lib.USP_BF16}
_MODES = {"materialised": _lib.USP_MATERIALISED, "fused": _lib.USP_FUSED}


def _dt(t: torch.Tensor) -> int:
    if t.dtype not in _DT:
        raise TypeError(f"unsupported dtype {t.dtype}; use float32 or bfloat16")
    return _DT[t.dtype]


def _dev(*ts):
    for t in ts:
        if not t.is_cuda:
            raise ValueError("tensor must be on a CUDA device")
        if not t.is_contiguous():
            raise ValueError("tensor must be contiguous")


def _stream():
    return ctypes_stream(torch.cuda.current_stream())


def ctypes_stream(s) -> int:
    return int(s.cuda_stream)


def _p(t):
    return None if t is None else t.data_ptr()


def relayout_tok2head(src: torch.Tensor, ulysses: int, ring: int, out: torch.Tensor | None = None):
    """Token-sharded [r,u,B,H,Ns(,D)] -> head-sharded [r,u,B,H/u,Nr(,D)]."""
    r, u, B, H, Ns = src.shape[:5]
    D = src.shape[5] if src.dim() == 6 else 1
    if (r, u) != (ring, ulysses):
        raise ValueError("stack shape does not match (ring, ulysses)")
    if H % ulysses:
        raise ValueError("H must be divisible by ulysses")
    shape = (r, u, B, H // u, u * Ns) + tuple(src.shape[5:])
    out = torch.empty(shape, dtype=src.dtype, device=src.device) if out is None else out
    _dev(src, out)
    check("usp_relayout_tok2head", _lib.lib().usp_relayout_tok2head(
        _p(src), _p(out), B, H, u * r * Ns, D, ulysses, ring, _dt(src), _stream()))
    return out


def relayout_head2tok(src: torch.Tensor, ulysses: int, ring: int, out: torch.Tensor | None = None):
    """Head-sharded [r,u,B,Hu,Nr(,D)] -> token-sharded [r,u,B,H,Ns(,D)]."""
    r, u, B, Hu, Nr = src.shape[:5]
    D = src.shape[5] if src.dim() == 6 else 1
    if (r, u) != (ring, ulysses):
        raise ValueError("stack shape does not match (ring, ulysses)")
    if Nr % ulysses:
        raise ValueError("Nr must be divisible by ulysses")
    shape = (r, u, B, Hu * u, Nr // u) + tuple(src.shape[5:])
    out = torch.empty(shape, dtype=src.dtype, device=src.device) if out is None else out
    _dev(src, out)
    check("usp_relayout_head2tok", _lib.lib().usp_relayout_head2tok(
        _p(src), _p(out), B, Hu * u, r * Nr, D, ulysses, ring, _dt(src), _stream()))
    return out


def attn_chunk_fwd(q, k, v, scale: float | None = None, out=None, lse=None):
    """(out, lse) of attention of q [B,H,Nq,D] against k, v [B,H,Nk,D]."""
    B, H, Nq, D = q.shape
    Nk = k.shape[2]
    if k.shape != (B, H, Nk, D) or v.shape != k.shape:
        raise ValueError("k and v must be [B,H,Nk,D] matching q")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device) if lse is None else lse
    _dev(q, k, v, out, lse)
    check("usp_attn_chunk_fwd", _lib.lib().usp_attn_chunk_fwd(
        _p(q), _p(k), _p(v), _p(out), _p(lse), B, H, Nq, Nk, D, scale, _dt(q), _stream()))
    return out, lse


def lse_merge(outs, lses, out=None, lse=None):
    """Merge R partials: outs [R,B,H,Nq,D], lses [R,B,H,Nq] -> (out, lse)."""
    R, B, H, Nq, D = outs.shape
    if lses.shape != (R, B, H, Nq) or lses.dtype != torch.float32:
        raise ValueError("lses must be fp32 [R,B,H,Nq]")
    out = torch.empty(outs.shape[1:], dtype=outs.dtype, device=outs.device) if out is None else out
    lse = torch.empty(lses.shape[1:], dtype=torch.float32, device=outs.device) if lse is None else lse
    _dev(outs, lses, out, lse)
    check("usp_lse_merge", _lib.lib().usp_lse_merge(
        _p(outs), _p(lses), R, _p(out), _p(lse), B, H, Nq, D, _dt(outs), _stream()))
    return out, lse


def workspace_bytes(B, H, N, D, ulysses, ring, dtype=torch.bfloat16, mode="fused", backward=False) -> int:
    return int(_lib.lib().usp_attention_workspace_bytes(B, H, N, D, ulysses, ring, _DT[dtype], _MODES[mode],
                                                        1 if backward else 0))


def _stack_dims(q, ulysses, ring):
    r, u, B, H, Ns, D = q.shape
    if (r, u) != (ring, ulysses):
        raise ValueError("q must be the token-sharded stack [ring, ulysses, B, H, Ns, D]")
    return B, H, r * u * Ns, D


def _to_device(ts, device):
    return [t.to(device, non_blocking=True).contiguous() for t in ts]


def _to_host(t: torch.Tensor) -> torch.Tensor:
    h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
    h.copy_(t, non_blocking=True)
    return h


def attention_fwd(q, k, v, ulysses: int, ring: int, scale: float | None = None, mode: str = "fused",
                  out=None, lse=None, workspace=None):
    """USP attention forward over token-sharded stacks [ring, ulysses, B, H, Ns, D].

    Returns (out, lse) with out in the stack layout and lse [ring, ulysses, B,
    H, Ns] fp32.  CPU inputs are copied to the current CUDA device and the
    results copied back to pinned host memory (synchronised before return).
    """
    host = not q.is_cuda
    if host:
        q, k, v = _to_device((q, k, v), torch.device("cuda", torch.cuda.current_device()))
    B, H, N, D = _stack_dims(q, ulysses, ring)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty(q.shape[:5], dtype=torch.float32, device=q.device) if lse is None else lse
    _dev(q, k, v, out, lse)
    need = workspace_bytes(B, H, N, D, ulysses, ring, q.dtype, mode)
    if need and (workspace is None or workspace.numel() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    check("usp_attention_fwd", _lib.lib().usp_attention_fwd(
        _p(q), _p(k), _p(v), _p(out), _p(lse), B, H, N, D, ulysses, ring, scale, _dt(q), _MODES[mode],
        _p(workspace) if need else None, need, _stream()))
    if host:
        out, lse = _to_host(out), _to_host(lse)
        torch.cuda.current_stream().synchronize()
    return out, lse


def joint_workspace_bytes(B, H, N, Nt, D, ulysses, ring, dtype=torch.bfloat16, mode="fused",
                          text_queries=True) -> int:
    return int(_lib.lib().usp_attention_joint_workspace_bytes(B, H, N, Nt, D, ulysses, ring, _DT[dtype],
                                                              _MODES[mode], 1 if text_queries else 0))


def attention_fwd_joint(q, k, v, k_txt, v_txt, ulysses: int, ring: int, scale: float | None = None,
                        q_txt=None, mode: str = "fused", workspace=None):
    """Joint text + image USP attention forward.

    q, k, v: token-sharded image stacks [ring, ulysses, B, H, Ns, D];
    k_txt, v_txt (and q_txt): replicated text tensors [B, H, Nt, D].
    Returns (out, lse) in the stack layout and, when q_txt is given,
    (out_txt [B, H, Nt, D], lse_txt [B, H, Nt]).  CPU inputs take the host
    path of :func:`attention_fwd`.
    """
    host = not q.is_cuda
    if host:
        dev = torch.device("cuda", torch.cuda.current_device())
        q, k, v, k_txt, v_txt = _to_device((q, k, v, k_txt, v_txt), dev)
        if q_txt is not None:
            (q_txt,) = _to_device((q_txt,), dev)
    B, H, N, D = _stack_dims(q, ulysses, ring)
    Nt = k_txt.shape[2]
    for t in (k_txt, v_txt) + (() if q_txt is None else (q_txt,)):
        if tuple(t.shape) != (B, H, Nt, D) or t.dtype != q.dtype:
            raise ValueError("text tensors must be [B, H, Nt, D] in the image dtype")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:5], dtype=torch.float32, device=q.device)
    out_txt = lse_txt = None
    if q_txt is not None:
        out_txt = torch.empty_like(q_txt)
        lse_txt = torch.empty((B, H, Nt), dtype=torch.float32, device=q.device)
    _dev(*[t for t in (q, k, v, k_txt, v_txt, q_txt, out, lse, out_txt, lse_txt) if t is not None])
    need = joint_workspace_bytes(B, H, N, Nt, D, ulysses, ring, q.dtype, mode, q_txt is not None)
    if need and (workspace is None or workspace.numel() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    check("usp_attention_fwd_joint", _lib.lib().usp_attention_fwd_joint(
        _p(q), _p(k), _p(v), _p(q_txt), _p(k_txt), _p(v_txt), _p(out), _p(lse), _p(out_txt), _p(lse_txt),
        B, H, N, Nt, D, ulysses, ring, scale, _dt(q), _MODES[mode], _p(workspace) if need else None, need,
        _stream()))
    res = (out, lse) if q_txt is None else (out, lse, out_txt, lse_txt)
    if host:
        res = tuple(_to_host(t) for t in res)
        torch.cuda.current_stream().synchronize()
    return res


def cross_attention_fwd(q, k_txt, v_txt, ulysses: int, ring: int, scale: float | None = None, out=None, lse=None):
    """Cross-attention of the token-sharded image queries [ring, ulysses, B, H,
    Ns, D] to the replicated text K/V [B, H, Nt, D] -> (out, lse) in the
    stack layout.  CPU inputs take the host path of :func:`attention_fwd`."""
    host = not q.is_cuda
    if host:
        q, k_txt, v_txt = _to_device((q, k_txt, v_txt), torch.device("cuda", torch.cuda.current_device()))
    B, H, N, D = _stack_dims(q, ulysses, ring)
    Nt = k_txt.shape[2]
    for t in (k_txt, v_txt):
        if tuple(t.shape) != (B, H, Nt, D) or t.dtype != q.dtype:
            raise ValueError("text K/V must be [B, H, Nt, D] in the query dtype")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty(q.shape[:5], dtype=torch.float32, device=q.device) if lse is None else lse
    _dev(q, k_txt, v_txt, out, lse)
    check("usp_cross_attention_fwd", _lib.lib().usp_cross_attention_fwd(
        _p(q), _p(k_txt), _p(v_txt), _p(out), _p(lse), B, H, N, Nt, D, ulysses, ring, scale, _dt(q), _stream()))
    if host:
        out, lse = _to_host(out), _to_host(lse)
        torch.cuda.current_stream().synchronize()
    return out, lse


def quantize_e4m3(x, ulysses: int, ring: int):
    """Per-head E4M3 codes (uint8, same stack layout) and dequantisation
    scales [B, H] fp32 of a bf16 token-sharded stack."""
    B, H, N, D = _stack_dims(x, ulysses, ring)
    x8 = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    scales = torch.empty((B, H), dtype=torch.float32, device=x.device)
    _dev(x, x8, scales)
    check("usp_quantize_e4m3", _lib.lib().usp_quantize_e4m3(
        _p(x), _p(x8), _p(scales), B, H, N, D, ulysses, ring, _stream()))
    return x8, scales


def attention_fwd_fp8(q, k, v, ulysses: int, ring: int, scale: float | None = None, out=None, lse=None,
                      workspace=None):
    """FP8 (E4M3) fused USP forward of bf16 token-sharded stacks -> (out bf16, lse fp32)."""
    host = not q.is_cuda
    if host:
        q, k, v = _to_device((q, k, v), torch.device("cuda", torch.cuda.current_device()))
    B, H, N, D = _stack_dims(q, ulysses, ring)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty(q.shape[:5], dtype=torch.float32, device=q.device) if lse is None else lse
    _dev(q, k, v, out, lse)
    need = int(_lib.lib().usp_attention_fp8_workspace_bytes(B, H, N, D, ulysses, ring))
    if need and (workspace is None or workspace.numel() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    check("usp_attention_fwd_fp8", _lib.lib().usp_attention_fwd_fp8(
        _p(q), _p(k), _p(v), _p(out), _p(lse), B, H, N, D, ulysses, ring, scale, _p(workspace) if need else None,
        need, _stream()))
    if host:
        out, lse = _to_host(out), _to_host(lse)
        torch.cuda.current_stream().synchronize()
    return out, lse


def attention_bwd(q, k, v, out, lse, dout, ulysses: int, ring: int, scale: float | None = None,
                  workspace=None, mode: str = "fused"):
    """USP attention backward over token-sharded stacks -> (dq, dk, dv).

    mode "fused" reads the stacks in place; "materialised" re-lays q, k, v,
    O, dO and lse out head-sharded, runs the per-rank chunk backward there
    and re-lays the gradients back (usp_attention_bwd_materialised)."""
    if mode not in ("fused", "materialised"):
        raise ValueError("mode must be 'fused' or 'materialised'")
    host = not q.is_cuda
    if host:
        q, k, v, out, lse, dout = _to_device((q, k, v, out, lse, dout),
                                             torch.device("cuda", torch.cuda.current_device()))
    B, H, N, D = _stack_dims(q, ulysses, ring)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    _dev(q, k, v, out, lse, dout, dq, dk, dv)
    need = workspace_bytes(B, H, N, D, ulysses, ring, q.dtype, mode, backward=True)
    if need and (workspace is None or workspace.numel() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    name = "usp_attention_bwd" if mode == "fused" else "usp_attention_bwd_materialised"
    check(name, getattr(_lib.lib(), name)(
        _p(q), _p(k), _p(v), _p(out), _p(lse), _p(dout), _p(dq), _p(dk), _p(dv), B, H, N, D, ulysses, ring,
        scale, _dt(q), _p(workspace) if need else None, need, _stream()))
    if host:
        dq, dk, dv = _to_host(dq), _to_host(dk), _to_host(dv)
        torch.cuda.current_stream().synchronize()
    return dq, dk, dv


def device_status() -> int:
    """Synchronise the current stream and return (and clear) the device error status."""
    return int(_lib.lib().usp_device_status(_stream()))


def set_spin_limit(polls: int) -> None:
    """Test hook: polls a device-side wait may make before it gives up
    (usp_set_debug_spin_limit; negative restores the default)."""
    _lib.lib().usp_set_debug_spin_limit(int(polls))
