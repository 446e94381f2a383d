"""GPU parity of the FP8 (OCP E4M3) path against the oracle, through the C ABI.

Quantisation is integer work on a float decision taken in fp32 on both sides,
so codes and scales must match the oracle bit for bit.  The FP8 attention is
compared with the oracle's attention of the dequantised q, k, v; the only
remaining difference is the kernel's E4M3 rounding of P, which the error model
in tests/fp8_error_model.py bounds per element (7 sigma + bf16 output rounding
+ 1e-4); LSE within 1e-3 relative.  Small problems: every row.  Qwen-Image
1024^2 and the Wan shapes: 4096 sampled query rows per head (Wan: four heads,
two on either side of a Ulysses group boundary)."""
import numpy as np
import pytest
import torch

import oracle
from oracle import pool
from diffusion_transformer_sequence_gb300 import workloads as wl
from tests.fp8_error_model import check_fp8, sigma_rows
from tests.helpers import Canary, ensure_built, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()
    assert torch.cuda.is_available()


def _usp():
    import diffusion_transformer_sequence_gb300 as usp
    return usp


def _codes_as_values(x8):
    return x8.cpu().view(torch.float8_e4m3fn).double().numpy()


@pytest.mark.parametrize("B,H,N,D,u,r,mag", [
    (1, 4, 512, 128, 2, 2, 1.0),
    (2, 3, 300, 64, 3, 1, 40.0),      # ragged shards, larger magnitudes
    (1, 8, 800, 128, 8, 1, 1e-3),     # small magnitudes: subnormal codes
    (1, 2, 1000, 16, 2, 4, 300.0),
])
def test_quantize_e4m3_bit_exact(B, H, N, D, u, r, mag):
    usp = _usp()
    g = torch.Generator().manual_seed(N + D)
    x = (torch.randn(B, H, N, D, generator=g) * mag).to(torch.bfloat16)
    x[:, -1, : N // 3] *= 50                      # one head with a few large values
    if H > 2:
        x[0, 1] = 0                               # an all-zero head
    st = wl.to_token_stack(x, u, r)
    x8, sc = usp.quantize_e4m3(st.cuda(), u, r)
    assert usp.device_status() == 0
    codes, scales = oracle.quantize_e4m3_heads(f64(st))
    np.testing.assert_array_equal(_codes_as_values(x8), codes)
    np.testing.assert_array_equal(sc.cpu().double().numpy(), scales)


def _oracle_fp8(w, stacks):
    O, L, codes, scales = oracle.usp_forward_fp8(*[f64(t) for t in stacks], w.ulysses, w.ring, w.scale)
    return O, L, codes, scales


SMALL = [
    (1, 2, 512, 2, 2),
    (2, 6, 960, 3, 2),     # ragged tiles in every shard
    (1, 8, 800, 8, 1),     # shards shorter than one tile
    (1, 2, 1000, 2, 4),    # Ns = 125: V^T rows padded to 128
    (1, 2, 384, 1, 1),
]


@pytest.mark.parametrize("B,H,N,u,r", SMALL)
def test_fp8_attention_small_full_rows(B, H, N, u, r):
    usp = _usp()
    w = wl.custom("fp8", "bf16", B, H, N, 128, u, r, seed=N + 11 * H)
    inp = wl.make_inputs(w, with_dout=False)
    stacks = [wl.to_token_stack(inp[n], u, r) for n in ("q", "k", "v")]
    O, L, codes, scales = _oracle_fp8(w, stacks)
    oc = Canary(w.stack_shape, torch.bfloat16)
    lc = Canary(w.lse_stack_shape, torch.float32)
    usp.attention_fwd_fp8(*[t.cuda() for t in stacks], u, r, w.scale, out=oc.view, lse=lc.view)
    assert usp.device_status() == 0
    oc.check()
    lc.check()
    deq = [wl.from_token_stack(torch.from_numpy(c * s[None, None, :, :, None, None])).reshape(B * H, N, 128).numpy()
           for c, s in zip(codes, scales)]
    sig = np.stack([sigma_rows(deq[0][h], deq[1][h], deq[2][h], np.arange(N), w.scale) for h in range(B * H)])
    go = wl.from_token_stack(oc.view.cpu()).reshape(B * H, N, 128)
    gl = wl.from_token_stack(lc.view.cpu()).reshape(B * H, N)
    ro = wl.from_token_stack(torch.from_numpy(O)).reshape(B * H, N, 128).numpy()
    rl = wl.from_token_stack(torch.from_numpy(L)).reshape(B * H, N).numpy()
    check_fp8(f64(go), f64(gl), ro, rl, sig, f"fp8 B{B} H{H} N{N} u{u} r{r}")


@pytest.mark.parametrize("name,heads", [("qwen1024", None), ("wan_s32k", [0, 4, 5, 39]), ("wan720p", [4, 5])])
def test_fp8_attention_workloads_sampled(name, heads):
    usp = _usp()
    w = wl.WORKLOADS[name]
    inp = wl.make_inputs(w, with_dout=False)
    stacks = [wl.to_token_stack(inp[n], w.ulysses, w.ring) for n in ("q", "k", "v")]
    o, l = usp.attention_fwd_fp8(*[t.cuda() for t in stacks], w.ulysses, w.ring, w.scale)
    assert usp.device_status() == 0
    BH = w.B * w.H
    heads = list(range(BH)) if heads is None else heads
    rows = wl.sample_rows(w, 4096)
    deq = []
    for t in stacks:
        c, s = oracle.quantize_e4m3_heads(f64(t))
        deq.append(wl.from_token_stack(torch.from_numpy(c * s[None, None, :, :, None, None]))
                   .reshape(BH, w.N, w.D)[heads].numpy())
    ro, rl = pool.sampled_attention(deq[0], deq[1], deq[2], rows.numpy(), w.scale)
    sig = np.stack([sigma_rows(deq[0][i], deq[1][i], deq[2][i], rows.numpy(), w.scale) for i in range(len(heads))])
    go = wl.from_token_stack(o).reshape(BH, w.N, w.D)[heads][:, rows.cuda()]
    gl = wl.from_token_stack(l).reshape(BH, w.N)[heads][:, rows.cuda()]
    err, worst = check_fp8(f64(go), f64(gl), ro, rl, sig, f"fp8 {name}")
    # the same rows against unquantised bf16-input attention: the FP8 error itself (reported, loose bound)
    exact = [inp[n].reshape(BH, w.N, w.D)[heads].float().numpy() for n in ("q", "k", "v")]
    eo, _ = pool.sampled_attention(*exact, rows.numpy(), w.scale)
    e_fp8 = np.abs(f64(go) - eo).max()
    print(f"\nfp8 {name}: max |O - oracle(dequantised)| = {err:.3e} ({worst:.2f} of the model bound); "
          f"max |O - exact attention| = {e_fp8:.3e}")
    assert e_fp8 < 0.1
