"""Pins for the CPU oracle: each oracle function is checked against something
other than itself -- a library routine (torch fp64 SDPA, logsumexp, autograd
on CPU), a closed form, an invariant, brute force on tiny inputs, or the value
the handbook prints for its four-card Ulysses demo.  A mutation suite at the
end plants plausible mistakes in copies of the oracle and checks that these
pins catch every one.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import usp_oracle as uo
from diffusion_transformer_sequence_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g, dtype=torch.float64)


def _sdpa(q, k, v, scale):
    """torch's own attention routine in fp64 on CPU plus torch.logsumexp."""
    o = F.scaled_dot_product_attention(q, k, v, scale=scale)
    lse = torch.logsumexp(scale * torch.matmul(q, k.transpose(-1, -2)), dim=-1)
    return o, lse


# ---------------------------------------------------------------- attention

@pytest.mark.parametrize("shape", [(2, 3, 37, 53, 16), (1, 8, 256, 256, 32), (1, 2, 1, 129, 8), (1, 1, 130, 1, 4)])
def test_attention_matches_torch_sdpa(shape):
    B, H, Nq, Nk, D = shape
    q, k, v = _rand((B, H, Nq, D), 1), _rand((B, H, Nk, D), 2), _rand((B, H, Nk, D), 3)
    scale = 1.0 / math.sqrt(D)
    o, lse = uo.attention(q.numpy(), k.numpy(), v.numpy(), scale, row_block=7)
    ro, rl = _sdpa(q, k, v, scale)
    np.testing.assert_allclose(o, ro.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, rl.numpy(), rtol=0, atol=1e-12)


def test_attention_bruteforce_tiny():
    """Direct one-pass evaluation with math.exp over Python lists."""
    Nq, Nk, D, scale = 3, 5, 4, 0.7
    q, k, v = _rand((Nq, D), 4).tolist(), _rand((Nk, D), 5).tolist(), _rand((Nk, D), 6).tolist()
    o, lse = uo.attention(np.array(q), np.array(k), np.array(v), scale)
    for i in range(Nq):
        w = [math.exp(scale * sum(q[i][d] * k[j][d] for d in range(D))) for j in range(Nk)]
        z = sum(w)
        assert abs(lse[i] - math.log(z)) < 1e-12
        for d in range(D):
            assert abs(o[i, d] - sum(w[j] * v[j][d] for j in range(Nk)) / z) < 1e-12


def test_attention_closed_forms():
    D, scale = 8, 0.3
    q, k, v = _rand((5, D), 7).numpy(), _rand((1, D), 8).numpy(), _rand((1, D), 9).numpy()
    # one key: every weight is 1, O = v, lse = scale q.k
    o, lse = uo.attention(q, k, v, scale)
    np.testing.assert_allclose(o, np.repeat(v, 5, 0), atol=1e-14)
    np.testing.assert_allclose(lse, scale * (q @ k[0]), atol=1e-13)
    # identical keys: uniform weights, O = mean(V), lse = s + ln Nk
    Nk = 11
    kk = np.repeat(k, Nk, 0)
    vv = _rand((Nk, D), 10).numpy()
    o, lse = uo.attention(q, kk, vv, scale)
    np.testing.assert_allclose(o, np.repeat(vv.mean(0, keepdims=True), 5, 0), atol=1e-13)
    np.testing.assert_allclose(lse, scale * (q @ k[0]) + math.log(Nk), atol=1e-13)


def test_attention_rows_is_row_subset():
    q, k, v = _rand((2, 40, 8), 11).numpy(), _rand((2, 33, 8), 12).numpy(), _rand((2, 33, 8), 13).numpy()
    rows = [0, 5, 39, 17]
    o, l = uo.attention(q, k, v, 0.5)
    o2, l2 = uo.attention_rows(q, k, v, rows, 0.5)
    np.testing.assert_array_equal(o2, o[:, rows])
    np.testing.assert_array_equal(l2, l[:, rows])


# -------------------------------------------------------------------- merge

def test_merge_of_chunks_equals_full_attention():
    """Ring paragraph: merging per-chunk results by log-sum-exp gives full attention."""
    B, H, Nq, D = 1, 3, 21, 16
    q = _rand((B, H, Nq, D), 20)
    ks = [_rand((B, H, n, D), 21 + i) for i, n in enumerate((5, 17, 1, 30))]
    vs = [_rand((B, H, n, D), 31 + i) for i, n in enumerate((5, 17, 1, 30))]
    scale = 0.25
    parts = [uo.attention(q.numpy(), kc.numpy(), vc.numpy(), scale) for kc, vc in zip(ks, vs)]
    o, l = uo.lse_merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
    ro, rl = _sdpa(q, torch.cat(ks, 2), torch.cat(vs, 2), scale)
    np.testing.assert_allclose(o, ro.numpy(), atol=1e-12)
    np.testing.assert_allclose(l, rl.numpy(), atol=1e-12)


def test_merge_special_cases():
    o, l = _rand((1, 4, 9, 8), 40).numpy(), _rand((1, 4, 9), 41).numpy()
    mo, ml = uo.lse_merge(o[None], l[None])                  # one partial: unchanged
    np.testing.assert_allclose(mo, o, atol=1e-15)
    np.testing.assert_allclose(ml, l, atol=1e-15)
    mo, ml = uo.lse_merge(np.stack([o, o]), np.stack([l, l]))  # two equal partials
    np.testing.assert_allclose(mo, o, atol=1e-14)
    np.testing.assert_allclose(ml, l + math.log(2.0), atol=1e-14)
    # a partial with a much smaller lse contributes ~nothing
    o2 = _rand((1, 4, 9, 8), 42).numpy()
    mo, ml = uo.lse_merge(np.stack([o, o2]), np.stack([l, l - 200.0]))
    np.testing.assert_allclose(mo, o, atol=1e-12)
    np.testing.assert_allclose(ml, l, atol=1e-12)


# ----------------------------------------------------------------- re-layout

def _heads_exchange(shards, H, P):
    """The handbook's head exchange, built independently of the oracle's run
    loops from tensor views: P source cards each hold [B, H, n, D] (their
    tokens, every head); destination card j receives head group j of every
    source, the sources' token segments laid end to end in source order.
    Stack the sources, split H into (P, H/P), and move the destination axis
    to the front and the source axis next to the token axis."""
    S = torch.stack(shards)                                   # [src, B, H, n, D]
    src, B, _, n, D = S.shape
    S = S.reshape(src, B, P, H // P, n, D)                    # [src, B, dst, h', n, D]
    S = S.permute(2, 1, 3, 0, 4, 5)                           # [dst, B, h', src, n, D]
    return list(S.reshape(P, B, H // P, src * n, D))          # per dst: [B, h', src*n, D]


def _tokens_exchange(parts, N, P):
    """The inverse exchange: P cards each hold [B, H/P, N, D] (all tokens of
    their head group); source card s receives token segment s of every card's
    heads, the head groups stacked in card order."""
    S = torch.stack(parts)                                    # [grp, B, h', N, D]
    grp, B, hp, _, D = S.shape
    S = S.reshape(grp, B, hp, P, N // P, D)                   # [grp, B, h', seg, n, D]
    S = S.permute(3, 1, 0, 2, 4, 5)                           # [seg, B, grp, h', n, D]
    return list(S.reshape(P, B, grp * hp, N // P, D))        # per seg: [B, H, n, D]


@pytest.mark.parametrize("u,r,B,H,N,D", [(4, 1, 1, 8, 256, 32), (2, 2, 2, 6, 24, 3), (3, 2, 1, 9, 42, 5), (1, 3, 1, 2, 9, 4), (2, 1, 1, 2, 2, 1)])
def test_relayout_matches_page_construction(u, r, B, H, N, D):
    x = torch.arange(B * H * N * D, dtype=torch.int64).reshape(B, H, N, D)
    Ns, Nr = N // (u * r), N // r
    T = wl.to_token_stack(x, u, r)
    X = uo.tok2head(T.numpy(), u, r)
    for g in range(r):
        shards = [x[:, :, (g * u + s) * Ns:(g * u + s + 1) * Ns] for s in range(u)]
        ref = _heads_exchange(shards, H, u)
        for j in range(u):
            assert torch.equal(torch.from_numpy(X[g, j]), ref[j])
        back = _tokens_exchange([torch.from_numpy(X[g, j]) for j in range(u)], Nr, u)
        Tb = uo.head2tok(X, u, r)
        for s in range(u):
            assert torch.equal(torch.from_numpy(Tb[g, s]), back[s])
    np.testing.assert_array_equal(uo.head2tok(X, u, r), T.numpy())           # roundtrip
    assert np.array_equal(np.sort(X.ravel()), np.arange(x.numel()))         # a permutation


def test_relayout_lse_layout():
    u, r, B, H, N = 2, 2, 1, 4, 12
    L = torch.arange(B * H * N, dtype=torch.int64).reshape(B, H, N)
    T = wl.to_token_stack(L, u, r)
    X = uo.tok2head(T.numpy(), u, r)
    assert X.shape == (r, u, B, H // u, N // r)
    np.testing.assert_array_equal(uo.head2tok(X, u, r), T.numpy())
    # head-sharded rank (g, j) row n holds global token g*Nr + n of head j*Hu + h'
    for g in range(r):
        for j in range(u):
            for h in range(H // u):
                np.testing.assert_array_equal(X[g, j, 0, h], L[0, j * (H // u) + h, g * (N // r):(g + 1) * (N // r)].numpy())


# ------------------------------------------------------------ USP simulation

def test_page_demo_golden():
    gd = json.load(open(os.path.join(GOLDEN, "ulysses_demo.json")))
    w = wl.WORKLOADS["demo"]
    assert (w.B, w.H, w.N, w.D, w.ulysses, w.ring) == (gd["B"], gd["H"], gd["N"], gd["D"], gd["P"], 1)
    inp = wl.make_inputs(w)
    torch.manual_seed(0)                         # the page's own draw order
    q0, k0, v0 = (torch.randn(gd["B"], gd["H"], gd["N"], gd["D"]) for _ in range(3))
    assert torch.equal(inp["q"], q0) and torch.equal(inp["k"], k0) and torch.equal(inp["v"], v0)
    Tq, Tk, Tv = (wl.to_token_stack(inp[n], w.ulysses, w.ring).numpy() for n in ("q", "k", "v"))
    O, L = uo.usp_forward(Tq, Tk, Tv, w.ulysses, w.ring, w.scale)
    full = wl.from_token_stack(torch.from_numpy(O))
    sdpa_o = F.scaled_dot_product_attention(q0, k0, v0)
    assert torch.allclose(full.float(), sdpa_o, atol=gd["atol"]) == gd["printed_result"]
    ro, rl = _sdpa(q0.double(), k0.double(), v0.double(), w.scale)
    np.testing.assert_allclose(full.numpy(), ro.numpy(), atol=1e-12)
    np.testing.assert_allclose(wl.from_token_stack(torch.from_numpy(L)).numpy(), rl.numpy(), atol=1e-12)


@pytest.mark.parametrize("u,r,H,N", [(2, 2, 4, 24), (1, 4, 2, 32), (2, 3, 2, 18), (4, 2, 8, 40), (1, 1, 3, 7)])
def test_usp_forward_equals_unsharded(u, r, H, N):
    B, D = 2, 8
    q, k, v = _rand((B, H, N, D), 50), _rand((B, H, N, D), 51), _rand((B, H, N, D), 52)
    scale = 0.35
    T = [wl.to_token_stack(x, u, r).numpy() for x in (q, k, v)]
    O, L = uo.usp_forward(*T, u, r, scale)
    ro, rl = _sdpa(q, k, v, scale)
    np.testing.assert_allclose(wl.from_token_stack(torch.from_numpy(O)).numpy(), ro.numpy(), atol=1e-12)
    np.testing.assert_allclose(wl.from_token_stack(torch.from_numpy(L)).numpy(), rl.numpy(), atol=1e-12)


@pytest.mark.parametrize("u,r,H,N,Nt", [(2, 2, 4, 24, 5), (1, 3, 2, 18, 7), (4, 1, 8, 16, 3), (1, 1, 2, 8, 1)])
def test_usp_joint_equals_attention_over_concatenated_tokens(u, r, H, N, Nt):
    """Joint attention with replicated text == unsharded attention over [text; image]."""
    B, D, scale = 2, 8, 0.3
    q, k, v = _rand((B, H, N, D), 150), _rand((B, H, N, D), 151), _rand((B, H, N, D), 152)
    qt, kt, vt = _rand((B, H, Nt, D), 153), _rand((B, H, Nt, D), 154), _rand((B, H, Nt, D), 155)
    T = [wl.to_token_stack(x, u, r).numpy() for x in (q, k, v)]
    O, L, Ot, Lt = uo.usp_forward_joint(*T, kt.numpy(), vt.numpy(), u, r, scale, q_txt=qt.numpy())
    K, V = torch.cat([kt, k], 2), torch.cat([vt, v], 2)
    ro, rl = _sdpa(q, K, V, scale)
    np.testing.assert_allclose(wl.from_token_stack(torch.from_numpy(O)).numpy(), ro.numpy(), atol=1e-12)
    np.testing.assert_allclose(wl.from_token_stack(torch.from_numpy(L)).numpy(), rl.numpy(), atol=1e-12)
    to, tl = _sdpa(qt, K, V, scale)
    np.testing.assert_allclose(Ot, to.numpy(), atol=1e-12)
    np.testing.assert_allclose(Lt, tl.numpy(), atol=1e-12)


@pytest.mark.parametrize("u,r,N,Nt", [(2, 2, 16, 5), (4, 1, 12, 7), (1, 3, 9, 1)])
def test_usp_cross_attention_equals_unsharded(u, r, N, Nt):
    """Cross-attention of sharded image queries to replicated text K/V ==
    unsharded SDPA of all image queries against the text."""
    B, H, D, scale = 2, 4, 8, 0.4
    q = _rand((B, H, N, D), 160)
    kt, vt = _rand((B, H, Nt, D), 161), _rand((B, H, Nt, D), 162)
    O, L = uo.usp_cross_attention(wl.to_token_stack(q, u, r).numpy(), kt.numpy(), vt.numpy(), u, r, scale)
    ro, rl = _sdpa(q, kt, vt, scale)
    np.testing.assert_allclose(wl.from_token_stack(torch.from_numpy(O)).numpy(), ro.numpy(), atol=1e-12)
    np.testing.assert_allclose(wl.from_token_stack(torch.from_numpy(L)).numpy(), rl.numpy(), atol=1e-12)


def test_ring_chunk_schedule_visits_every_chunk_once():
    for r in range(1, 9):
        for g in range(r):
            assert sorted(uo.ring_chunk(g, t, r) for t in range(r)) == list(range(r))
            assert uo.ring_chunk(g, 0, r) == g


# ------------------------------------------------------------------ FP8 E4M3

def _e4m3_table():
    """Every finite E4M3 value, decoded from the bit fields: (value, code)."""
    vals = []
    for code in range(256):
        sgn, e, m = code >> 7, (code >> 3) & 15, code & 7
        if e == 15 and m == 7:
            continue                                   # NaN encodings
        mag = (m / 8) * 2.0 ** -6 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
        vals.append(((-1) ** sgn * mag, code))
    return vals


def test_e4m3_grid_fixed_points_and_extremes():
    table = _e4m3_table()
    v = np.array([t[0] for t in table])
    np.testing.assert_array_equal(uo.e4m3_round(v), v)
    assert v.max() == 448.0 and v.min() == -448.0
    assert np.min(np.abs(v[v != 0])) == 2.0 ** -9


def test_e4m3_round_is_nearest_ties_to_even_brute_force():
    table = [t for t in _e4m3_table() if t[0] >= 0 and not (t[0] == 0 and t[1] == 128)]
    vals = np.array([t[0] for t in table])
    codes = np.array([t[1] for t in table])
    rng = np.random.default_rng(31)
    x = np.concatenate([rng.uniform(0, 500, 4000), rng.uniform(0, 0.05, 2000), 2.0 ** rng.uniform(-12, 9, 2000),
                        (vals[:-1] + vals[1:]) / 2])                        # every midpoint: ties
    got = uo.e4m3_round(x)
    for xi, gi in zip(x, got):
        d = np.abs(vals - min(xi, 448.0))
        best = np.flatnonzero(d == d.min())
        pick = best[0] if len(best) == 1 else best[np.argmin(codes[best] & 1)]   # tie: even mantissa
        assert gi == vals[pick], (xi, gi, vals[pick])
    np.testing.assert_array_equal(uo.e4m3_round(-x), -got)


def test_e4m3_round_matches_torch_float8():
    rng = np.random.default_rng(32)
    x = np.concatenate([rng.standard_normal(20000) * 50, rng.standard_normal(5000) * 0.01])
    x = x[np.abs(x) <= 464]                            # torch's cast turns larger values into NaN, not 448
    x = x.astype(np.float32).astype(np.float64)        # torch rounds fp64 through fp32 first; feed fp32 values
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).double().numpy()
    np.testing.assert_array_equal(uo.e4m3_round(x), ref)


def test_quantize_e4m3_heads_against_torch_fp32_and_float8():
    rng = np.random.default_rng(33)
    T = (rng.standard_normal((2, 2, 2, 3, 10, 16)) * rng.uniform(0.1, 30, (1, 1, 2, 3, 1, 1))).astype(np.float32)
    T[:, :, 1, 2] = 0.0                                # an all-zero head
    codes, scales = uo.quantize_e4m3_heads(T)
    t = torch.from_numpy(T)
    amax = t.abs().amax(dim=(0, 1, 4, 5))
    inv = torch.where(amax > 0, torch.tensor(448.0, dtype=torch.float32) / torch.where(amax > 0, amax, 1.0),
                      torch.ones_like(amax))
    ref = (t * inv[None, None, :, :, None, None]).to(torch.float8_e4m3fn).double().numpy()
    np.testing.assert_array_equal(codes, ref)
    np.testing.assert_array_equal(scales, torch.where(amax > 0, amax / 448.0, 1.0).double().numpy())
    assert np.all(np.abs(codes).max(axis=(0, 1, 4, 5))[amax.numpy() > 0] == 448.0)   # amax -> +-448
    assert np.all(codes[:, :, 1, 2] == 0) and scales[1, 2] == 1.0
    deq = codes * scales[None, None, :, :, None, None]
    assert np.all(np.abs(deq - T) <= 2.0 ** -4 * np.abs(T) + 2.0 ** -10 * scales[None, None, :, :, None, None])
    T2 = T.copy()
    T2[:, :, 0, 0] *= 2                                # heads are independent
    c2, _ = uo.quantize_e4m3_heads(T2)
    mask = np.ones((2, 3), bool)
    mask[0, 0] = False
    np.testing.assert_array_equal(c2[:, :, mask], codes[:, :, mask])


def test_usp_forward_fp8_equals_sdpa_of_dequantised():
    u, r, B, H, N, D, scale = 2, 2, 1, 4, 32, 16, 0.25
    q, k, v = (_rand((B, H, N, D), s) * f for s, f in ((170, 3.0), (171, 1.0), (172, 2.0)))
    T = [wl.to_token_stack(x, u, r).numpy() for x in (q, k, v)]
    O, L, codes, scales = uo.usp_forward_fp8(*T, u, r, scale)
    deq = [wl.from_token_stack(torch.from_numpy(c * sc[None, None, :, :, None, None])) for c, sc in zip(codes, scales)]
    ro, rl = _sdpa(*deq, scale)
    np.testing.assert_allclose(wl.from_token_stack(torch.from_numpy(O)).numpy(), ro.numpy(), atol=1e-12)
    np.testing.assert_allclose(wl.from_token_stack(torch.from_numpy(L)).numpy(), rl.numpy(), atol=1e-12)
    # and it stays near unquantised attention (E4M3 keeps 3 mantissa bits)
    eo, _ = _sdpa(q / 3, k, v, scale)
    O2, _, _, _ = uo.usp_forward_fp8(wl.to_token_stack(q / 3, u, r).numpy(), T[1], T[2], u, r, scale)
    assert np.abs(wl.from_token_stack(torch.from_numpy(O2)).numpy() - eo.numpy()).max() < 0.25


# ----------------------------------------------------------------- backward

def test_bwd_matches_autograd():
    B, H, N, D = 1, 2, 45, 16
    scale = 0.2
    q, k, v, do = (_rand((B, H, N, D), s).requires_grad_(s < 63) for s in (60, 61, 62, 63))
    o = F.scaled_dot_product_attention(q, k, v, scale=scale)
    o.backward(do)
    oo, ll = uo.attention(q.detach().numpy(), k.detach().numpy(), v.detach().numpy(), scale)
    dq, dk, dv = uo.attention_bwd(q.detach().numpy(), k.detach().numpy(), v.detach().numpy(), oo, ll, do.numpy(), scale)
    np.testing.assert_allclose(dq, q.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dk, k.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dv, v.grad.numpy(), atol=1e-12)


def test_bwd_finite_differences():
    N, D, scale, eps = 4, 3, 0.9, 1e-6
    q, k, v, do = (_rand((N, D), s).numpy() for s in (70, 71, 72, 73))

    def loss(q_, k_, v_):
        return float((uo.attention(q_, k_, v_, scale)[0] * do).sum())

    o, l = uo.attention(q, k, v, scale)
    grads = uo.attention_bwd(q, k, v, o, l, do, scale)
    for idx, (x, g) in enumerate(zip((q, k, v), grads)):
        for i in range(N):
            for d in range(D):
                xp, xm = x.copy(), x.copy()
                xp[i, d] += eps
                xm[i, d] -= eps
                args_p = [q, k, v]
                args_m = [q, k, v]
                args_p[idx], args_m[idx] = xp, xm
                fd = (loss(*args_p) - loss(*args_m)) / (2 * eps)
                assert abs(fd - g[i, d]) < 1e-7


def test_bwd_sampled_matches_full():
    N, D, scale = 70, 8, 0.3
    q, k, v, do = (_rand((N, D), s).numpy() for s in (80, 81, 82, 83))
    o, l = uo.attention(q, k, v, scale)
    dq, dk, dv = uo.attention_bwd(q, k, v, o, l, do, scale)
    qr, kr = [0, 13, 69], [1, 2, 68, 69]
    sq, sk, sv = uo.attention_bwd_sampled(q, k, v, do, scale, qr, kr, row_block=16)
    np.testing.assert_allclose(sq, dq[qr], atol=1e-12)
    np.testing.assert_allclose(sk, dk[kr], atol=1e-12)
    np.testing.assert_allclose(sv, dv[kr], atol=1e-12)


def test_pool_matches_serial():
    from oracle import pool
    q, k, v = (_rand((3, 50, 8), s).numpy() for s in (90, 91, 92))
    rows = [0, 7, 49]
    o, l = pool.sampled_attention(q, k, v, rows, 0.4, workers=2)
    o1, l1 = uo.attention_rows(q, k, v, rows, 0.4)
    np.testing.assert_allclose(o, o1, atol=1e-13)
    np.testing.assert_allclose(l, l1, atol=1e-13)


# ----------------------------------------------------------- mutation suite

def _pins_pass(mod) -> bool:
    """Run the core pins against a (possibly mutated) oracle module."""
    try:
        rng = np.random.default_rng(5)
        q, k, v = (rng.standard_normal((2, 2, 12, 4)) for _ in range(3))
        ro, rl = _sdpa(*(torch.from_numpy(x) for x in (q, k, v)), 0.5)
        o, l = mod.attention(q, k, v, 0.5)
        if not (np.allclose(o, ro.numpy(), atol=1e-10) and np.allclose(l, rl.numpy(), atol=1e-10)):
            return False
        parts = [mod.attention(q, k[..., s:s + 4, :], v[..., s:s + 4, :], 0.5) for s in (0, 4, 8)]
        mo, ml = mod.lse_merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
        if not (np.allclose(mo, ro.numpy(), atol=1e-10) and np.allclose(ml, rl.numpy(), atol=1e-10)):
            return False
        x = torch.arange(1 * 4 * 12 * 2).reshape(1, 4, 12, 2)
        for u, r in ((2, 2), (2, 1), (1, 3)):
            T = wl.to_token_stack(x, u, r).numpy()
            X = mod.tok2head(T, u, r)
            Ns = 12 // (u * r)
            for g in range(r):
                sh = [x[:, :, (g * u + s) * Ns:(g * u + s + 1) * Ns] for s in range(u)]
                ref = _heads_exchange(sh, 4, u)
                if not all(torch.equal(torch.from_numpy(X[g, j]), ref[j]) for j in range(u)):
                    return False
            if not np.array_equal(mod.head2tok(X, u, r), T):
                return False
        T = [wl.to_token_stack(torch.from_numpy(a), 2, 2).numpy() for a in (q, k, v)]
        O, L = mod.usp_forward(*T, 2, 2, 0.5)
        if not np.allclose(wl.from_token_stack(torch.from_numpy(O)).numpy(), ro.numpy(), atol=1e-10):
            return False
        kt, vt = rng.standard_normal((2, 2, 3, 4)), rng.standard_normal((2, 2, 3, 4))
        qtx = rng.standard_normal((2, 2, 3, 4))
        Oj, Lj, Otj, Ltj = mod.usp_forward_joint(*T, kt, vt, 2, 2, 0.5, q_txt=qtx)
        Kc, Vc = torch.from_numpy(np.concatenate([kt, k], 2)), torch.from_numpy(np.concatenate([vt, v], 2))
        rj, _ = _sdpa(torch.from_numpy(q), Kc, Vc, 0.5)
        if not np.allclose(wl.from_token_stack(torch.from_numpy(Oj)).numpy(), rj.numpy(), atol=1e-10):
            return False
        rtj, _ = _sdpa(torch.from_numpy(qtx), Kc, Vc, 0.5)
        if not np.allclose(Otj, rtj.numpy(), atol=1e-10):
            return False
        Oc, _ = mod.usp_cross_attention(T[0], kt, vt, 2, 2, 0.5)
        rc, _ = _sdpa(torch.from_numpy(q), torch.from_numpy(kt), torch.from_numpy(vt), 0.5)
        if not np.allclose(wl.from_token_stack(torch.from_numpy(Oc)).numpy(), rc.numpy(), atol=1e-10):
            return False
        # FP8: rounding against torch's float8 cast, per-head quantisation, dequantised attention
        xs = (rng.standard_normal(4000) * 60).astype(np.float32).astype(np.float64)
        xs = xs[np.abs(xs) <= 464]
        if not np.array_equal(mod.e4m3_round(xs), torch.from_numpy(xs).to(torch.float8_e4m3fn).double().numpy()):
            return False
        Tq8 = (T[0] * np.array([1.0, 7.0])[None, None, None, :, None, None]).astype(np.float32)
        c8, s8 = mod.quantize_e4m3_heads(Tq8)
        t8 = torch.from_numpy(Tq8)
        am = t8.abs().amax(dim=(0, 1, 4, 5))
        if not np.array_equal(c8, (t8 * (448.0 / am)[None, None, :, :, None, None]).to(torch.float8_e4m3fn).double().numpy()):
            return False
        O8, _, cq, sq = mod.usp_forward_fp8(*T, 2, 2, 0.5)
        dq8 = [wl.from_token_stack(torch.from_numpy(c * sc[None, None, :, :, None, None])) for c, sc in zip(cq, sq)]
        r8, _ = _sdpa(*dq8, 0.5)
        if not np.allclose(wl.from_token_stack(torch.from_numpy(O8)).numpy(), r8.numpy(), atol=1e-10):
            return False
        oo, ll = uo.attention(q, k, v, 0.5)
        do = rng.standard_normal(q.shape)
        qt, kt, vt = (torch.from_numpy(a).requires_grad_() for a in (q, k, v))
        F.scaled_dot_product_attention(qt, kt, vt, scale=0.5).backward(torch.from_numpy(do))
        g = mod.attention_bwd(q, k, v, oo, ll, do, 0.5)
        return all(np.allclose(a, b.grad.numpy(), atol=1e-10) for a, b in zip(g, (qt, kt, vt)))
    except Exception:
        return False


def _mutant(src_old: str, src_new: str):
    import importlib.util
    import types
    src = open(uo.__file__).read()
    assert src.count(src_old) >= 1, src_old
    src = src.replace(src_old, src_new, 1)
    mod = types.ModuleType("oracle_mutant")
    exec(compile(src, "oracle_mutant", "exec"), mod.__dict__)
    return mod


MUTATIONS = [
    ("S = scale * (q[..., r0:r1, :] @ kT)", "S = (q[..., r0:r1, :] @ kT)"),                       # dropped scale
    ("np.exp(S - lse[..., None]) @ v", "np.exp(S - m) @ v"),                                      # unnormalised O
    ("m[..., 0] + np.log(", "np.log("),                                                           # dropped max term
    ("L = m + np.log(np.exp(lses - m[None]).sum(axis=0))", "L = m"),                              # merge without sum
    ("O += np.exp(lses[t] - L)[..., None] * outs[t]", "O += np.exp(lses[t] - m)[..., None] * outs[t]"),  # wrong weight
    ("= T[g, s, :, j * Hu:(j + 1) * Hu]", "= T[g, j, :, s * Hu:(s + 1) * Hu]"),                   # swapped rank roles
    ("X[g, j, :, :, s * Ns:(s + 1) * Ns] = T", "X[g, (j + 1) % u, :, :, s * Ns:(s + 1) * Ns] = T"),  # wrong destination
    ("return (g - t) % ring", "return g"),                                                         # no ring rotation
    ("    Xo, Xl = lse_merge(parts_o, parts_l)\n    out =", "    Xo, Xl = lse_merge(parts_o[:ring], parts_l[:ring])\n    out ="),  # text chunk dropped
    ("po[c], pl[c] = attention(qt[:, hs], Xk[c, j]", "po[c], pl[c] = attention(qt[:, hs], Xk[c, (j + 1) % ulysses]"),  # text queries, wrong head group
    ("O[g, j], L[g, j] = attention(Tq[g, j], kt", "O[g, j], L[g, j] = attention(Tq[g, (j + 1) % ulysses], kt"),  # cross: wrong rank's tokens
    ("y = np.round(a / quantum) * quantum", "y = np.trunc(a / quantum) * quantum"),              # E4M3: truncation
    ("E4M3_MAX = 448.0", "E4M3_MAX = 240.0"),                                                     # E4M3: wrong range
    ("amax = np.abs(T32).max(axis=(0, 1, 4, 5))", "amax = np.abs(T32).max() + np.zeros(T32.shape[2:4], np.float32)"),  # one scale for all heads
    ("deq = [c * sc[None, None, :, :, None, None] for c, sc in zip(codes, scales)]", "deq = [c for c in codes]"),  # no dequantisation
    ("dS = P * (dP - delta[..., None])", "dS = P * (dP + delta[..., None])"),                    # wrong sign
    ("dk = scale * (np.swapaxes(dS, -1, -2) @ q)", "dk = scale * (np.swapaxes(dS, -1, -2) @ k)"), # wrong operand
    ("dv = np.swapaxes(P, -1, -2) @ dout", "dv = P @ dout"),                                      # missing transpose
]


def test_pins_accept_the_oracle():
    assert _pins_pass(uo)


@pytest.mark.parametrize("old,new", MUTATIONS)
def test_pins_catch_planted_mistakes(old, new):
    assert not _pins_pass(_mutant(old, new))
