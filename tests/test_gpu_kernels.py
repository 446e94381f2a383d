"""GPU parity of the individual kernels against the CPU oracle, through the C ABI:
the Ulysses re-layouts (bit-exact), the LSE merge and the chunk attention
(fp32 and bf16), with ragged shapes, canary guards and double-run determinism."""
import math

import numpy as np
import pytest
import torch

import oracle
from diffusion_transformer_sequence_gb300 import workloads as wl
from tests.helpers import Canary, bits, check_out, ensure_built, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()
    import diffusion_transformer_sequence_gb300 as usp
    usp.lib()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _api():
    import diffusion_transformer_sequence_gb300 as usp
    return usp


def _randbits(shape, dtype, seed):
    """Arbitrary bit patterns (NaN and inf encodings included): a re-layout must move bits."""
    g = torch.Generator().manual_seed(seed)
    esz = torch.tensor([], dtype=dtype).element_size()
    it = {2: torch.int16, 4: torch.int32}[esz]
    lo, hi = (-(2 ** 15), 2 ** 15) if esz == 2 else (-(2 ** 31), 2 ** 31 - 1)
    return torch.randint(lo, hi, shape, generator=g, dtype=torch.int64).to(it).view(dtype)


RELAYOUT_CASES = [
    ("f32", 4, 1, 1, 8, 256, 32),        # handbook demo
    ("bf16", 2, 2, 1, 24, 4096, 128),    # Qwen-Image 1024^2, u2 x r2
    ("bf16", 4, 1, 1, 24, 16384, 128),   # Qwen-Image 2048^2, u4
    ("bf16", 8, 4, 1, 40, 32768, 128),   # Wan shapes, u8 x r4
    ("bf16", 8, 2, 1, 40, 75600, 128),   # Wan 720p, u8 x r2 (Ns = 4725)
    ("f32", 3, 2, 2, 6, 42, 5),          # ragged: 4-byte vector path
    ("bf16", 2, 1, 1, 2, 6, 3),          # 2-byte path
    ("bf16", 1, 1, 1, 1, 1, 1),          # single element
    ("f32", 2, 3, 3, 4, 6, 1),           # LSE-like layout (D = 1)
    ("bf16", 2, 2, 2, 4, 800, 128),      # 51200-byte runs: several CTAs per run, partial last chunk
    ("f32", 2, 2, 1, 4, 64, 4),          # 256-byte runs: one partly used CTA per run
    ("f32", 2, 2, 1, 4, 64, 1),          # LSE with Ns = 16: 64-byte runs
]


@pytest.mark.parametrize("dtype,u,r,B,H,N,D", RELAYOUT_CASES)
def test_relayout_bit_exact(dtype, u, r, B, H, N, D):
    usp = _api()
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    x = _randbits((B, H, N, D), tdt, seed=N + H)
    T = wl.to_token_stack(x, u, r)
    Td = T.cuda()
    Xc = Canary((r, u, B, H // u, N // r, D), tdt)
    X = usp.relayout_tok2head(Td, u, r, out=Xc.view)
    ref = oracle.tok2head(bits(T), u, r)
    assert np.array_equal(bits(X), ref)
    Bc = Canary(tuple(T.shape), tdt)
    back = usp.relayout_head2tok(X, u, r, out=Bc.view)
    assert np.array_equal(bits(back), bits(T))
    assert np.array_equal(bits(back), oracle.head2tok(ref, u, r))
    Xc.check()
    Bc.check()
    # a second run is bitwise identical
    X2 = usp.relayout_tok2head(Td, u, r)
    assert torch.equal(X2.view(torch.uint8), X.view(torch.uint8))


def test_relayout_lse_stack():
    usp = _api()
    u, r, B, H, N = 8, 2, 1, 40, 75600
    L = _randbits((B, H, N), torch.float32, seed=3)
    T = wl.to_token_stack(L, u, r)
    X = usp.relayout_tok2head(T.cuda(), u, r)
    assert np.array_equal(bits(X), oracle.tok2head(bits(T), u, r))
    assert np.array_equal(bits(usp.relayout_head2tok(X, u, r)), bits(T))


MERGE_CASES = [("bf16", 2, 1, 24, 4096, 128), ("bf16", 4, 1, 5, 8192, 128), ("f32", 3, 2, 3, 37, 32),
               ("f32", 1, 1, 2, 9, 16), ("bf16", 2, 1, 2, 5, 3), ("f32", 5, 1, 1, 1, 128), ("bf16", 8, 1, 1, 300, 128)]


@pytest.mark.parametrize("dtype,R,B,H,Nq,D", MERGE_CASES)
def test_lse_merge(dtype, R, B, H, Nq, D):
    usp = _api()
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    g = torch.Generator().manual_seed(R * 1000 + Nq)
    outs = torch.randn(R, B, H, Nq, D, generator=g).to(tdt)
    lses = (torch.randn(R, B, H, Nq, generator=g) * 3 + 5).float()
    oc, lc = Canary((B, H, Nq, D), tdt), Canary((B, H, Nq), torch.float32)
    o, l = usp.lse_merge(outs.cuda(), lses.cuda(), out=oc.view, lse=lc.view)
    ro, rl = oracle.lse_merge(f64(outs), f64(lses))
    if dtype == "f32":
        check_out(o, l, ro, rl, "f32", "merge")
    else:  # output rounded to bf16 once: |err| <= 2^-8 |value| + fp32 noise
        go = f64(o)
        assert np.all(np.abs(go - ro) <= 2.0 ** -8 * np.abs(ro) + 1e-5)
        assert np.abs(f64(l) - rl).max() <= 1e-5 * np.abs(rl).max()
    oc.check()
    lc.check()


F32_CHUNK = [(1, 8, 256, 256, 32), (2, 3, 37, 53, 16), (1, 2, 1, 129, 8), (1, 1, 130, 1, 4), (1, 2, 70, 300, 128)]
BF16_CHUNK = [(1, 2, 128, 128), (1, 3, 300, 200), (2, 2, 1, 1), (1, 1, 129, 4097), (1, 4, 1000, 257),
              (1, 1, 384, 384), (1, 2, 256, 1), (3, 1, 17, 2000),
              # more items (head x query-tile pair) than SMs: each CTA of the persistent
              # grid walks several, with odd query-tile counts (a lone last tile) and
              # 1, 2 or 3 KV tiles per item (the last one ragged), so the barrier
              # phases wrap across items in every parity pattern
              (2, 160, 300, 100), (2, 160, 300, 200), (1, 200, 300, 300),
              # 32 KV tiles per item (the longest run persistent) and 33 (one CTA per item)
              (1, 8, 1000, 4064), (1, 8, 1000, 4097)]


@pytest.mark.parametrize("B,H,Nq,Nk,D", F32_CHUNK)
def test_chunk_fwd_f32(B, H, Nq, Nk, D):
    usp = _api()
    g = torch.Generator().manual_seed(Nq * 7 + Nk)
    q, k, v = (torch.randn(B, H, n, D, generator=g) for n in (Nq, Nk, Nk))
    scale = 1 / math.sqrt(D)
    oc, lc = Canary((B, H, Nq, D), torch.float32), Canary((B, H, Nq), torch.float32)
    o, l = usp.attn_chunk_fwd(q.cuda(), k.cuda(), v.cuda(), scale, out=oc.view, lse=lc.view)
    ro, rl = oracle.attention(f64(q), f64(k), f64(v), scale)
    check_out(o, l, ro, rl, "f32", "chunk f32")
    oc.check()
    lc.check()


@pytest.mark.parametrize("B,H,Nq,Nk", BF16_CHUNK)
def test_chunk_fwd_bf16(B, H, Nq, Nk):
    usp = _api()
    D = 128
    g = torch.Generator().manual_seed(Nq * 13 + Nk)
    q, k, v = (torch.randn(B, H, n, D, generator=g).to(torch.bfloat16) for n in (Nq, Nk, Nk))
    scale = 1 / math.sqrt(D)
    oc, lc = Canary((B, H, Nq, D), torch.bfloat16), Canary((B, H, Nq), torch.float32)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, l = usp.attn_chunk_fwd(qd, kd, vd, scale, out=oc.view, lse=lc.view)
    assert usp.device_status() == 0
    ro, rl = oracle.attention(f64(q), f64(k), f64(v), scale)
    check_out(o, l, ro, rl, "bf16", "chunk bf16")
    oc.check()
    lc.check()
    o2, l2 = usp.attn_chunk_fwd(qd, kd, vd, scale)          # deterministic
    assert torch.equal(o2.view(torch.int16), o.view(torch.int16)) and torch.equal(l2, l)


def test_chunk_fwd_bf16_large_logits():
    """Scores spanning a wide range exercise the deferred-rescale path."""
    usp = _api()
    B, H, Nq, Nk, D = 1, 2, 256, 1024, 128
    g = torch.Generator().manual_seed(11)
    q = (torch.randn(B, H, Nq, D, generator=g) * 4).to(torch.bfloat16)
    k = (torch.randn(B, H, Nk, D, generator=g) * torch.linspace(0.1, 4, Nk)[None, None, :, None]).to(torch.bfloat16)
    v = torch.randn(B, H, Nk, D, generator=g).to(torch.bfloat16)
    o, l = usp.attn_chunk_fwd(q.cuda(), k.cuda(), v.cuda(), 1 / math.sqrt(D))
    ro, rl = oracle.attention(f64(q), f64(k), f64(v), 1 / math.sqrt(D))
    check_out(o, l, ro, rl, "bf16", "large logits")


def test_bounded_wait_timeout_path():
    """A poll limit of 0 makes the kernel's waits expire: it must return an error
    status instead of hanging, and the context must stay usable afterwards."""
    usp = _api()
    B, H, N, D = 1, 2, 512, 128
    g = torch.Generator().manual_seed(5)
    q, k, v = (torch.randn(B, H, N, D, generator=g).to(torch.bfloat16).cuda() for _ in range(3))
    assert usp.device_status() == 0
    try:
        usp.set_spin_limit(0)
        usp.attn_chunk_fwd(q, k, v)
        st = usp.device_status()
    finally:
        usp.set_spin_limit(-1)
    assert st == 6, f"expected USP_ERR_TIMEOUT, got {st}"
    assert usp.device_status() == 0          # cleared
    o, l = usp.attn_chunk_fwd(q, k, v)
    assert usp.device_status() == 0
    ro, rl = oracle.attention(f64(q), f64(k), f64(v), 1 / math.sqrt(D))
    check_out(o, l, ro, rl, "bf16", "after timeout")


@pytest.mark.parametrize("path", ["backward", "fp8"])
def test_bounded_wait_timeout_other_kernels(path):
    """The same expiring-wait check for the backward kernels (dK/dV, and dQ on
    the side stream) and the FP8 forward: error status, no hang, a cleared
    status, and correct results on the next call."""
    usp = _api()
    w = wl.custom("to", "bf16", 1, 2, 512, 128, 2, 2, seed=8, backward=True)
    inp = wl.make_inputs(w)
    st = {n: wl.to_token_stack(t, 2, 2).cuda() for n, t in inp.items()}
    o, l = usp.attention_fwd(st["q"], st["k"], st["v"], 2, 2, w.scale, mode="fused")
    assert usp.device_status() == 0

    def call():
        if path == "fp8":
            return usp.attention_fwd_fp8(st["q"], st["k"], st["v"], 2, 2, w.scale)
        return usp.attention_bwd(st["q"], st["k"], st["v"], o, l, st["dout"], 2, 2, w.scale)

    try:
        usp.set_spin_limit(0)
        call()
        status = usp.device_status()
    finally:
        usp.set_spin_limit(-1)
    assert status == 6, f"expected USP_ERR_TIMEOUT, got {status}"
    assert usp.device_status() == 0          # cleared
    res = call()
    assert usp.device_status() == 0
    stacks = [f64(wl.to_token_stack(inp[n], 2, 2)) for n in ("q", "k", "v")]
    if path == "fp8":
        ro, _, _, _ = oracle.usp_forward_fp8(*stacks, 2, 2, w.scale)
        assert np.abs(f64(res[0]) - ro).max() < 5e-2
    else:
        ro, rl = oracle.attention(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), w.scale)
        rdq, _, _ = oracle.attention_bwd(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), ro, rl, f64(inp["dout"]),
                                         w.scale)
        got = f64(wl.from_token_stack(res[0].cpu()))
        assert np.abs(got - rdq).max() / np.abs(rdq).max() < 2e-2
