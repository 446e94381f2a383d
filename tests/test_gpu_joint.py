"""GPU parity of the joint text + image USP forward (usp_attention_fwd_joint)
and of SP cross-attention (usp_cross_attention_fwd) against the oracle,
through the C ABI.

Joint attention: image tokens are sharded over the ulysses x ring virtual
ranks, the text tokens' q/k/v are replicated on every rank ("Parallelism
Acceleration Guide", "How to parallelize a new model": dual-stream joint
attention over the concatenated text + image sequence).  Small problems are
checked on every row against the oracle's own joint USP simulation
(oracle.usp_forward_joint); the two full-size joint workloads are checked on
4096 seeded image query rows per head plus every text query row against the
oracle's unsharded attention over the concatenated keys.  Tolerances are the
forward's: 1e-5 (fp32), 2e-2 on O and 1e-3 relative on LSE (bf16)."""
import numpy as np
import pytest
import torch

import oracle
from oracle import pool
from diffusion_transformer_sequence_gb300 import workloads as wl
from tests.helpers import Canary, check_out, ensure_built, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()
    assert torch.cuda.is_available()


def _usp():
    import diffusion_transformer_sequence_gb300 as usp
    return usp


def _joint_c(w, st, txt, mode, text_queries):
    """Call the C entry point with guarded output buffers; returns (o, l[, ot, lt])."""
    usp = _usp()
    from diffusion_transformer_sequence_gb300 import _lib
    L = usp.lib()
    B, H, N, Nt, D = w.B, w.H, w.N, w.Nt, w.D
    oc = Canary(w.stack_shape, w.torch_dtype)
    lc = Canary(w.lse_stack_shape, torch.float32)
    cans = [oc, lc]
    otc = ltc = None
    if text_queries:
        otc = Canary((B, H, Nt, D), w.torch_dtype)
        ltc = Canary((B, H, Nt), torch.float32)
        cans += [otc, ltc]
    dt = _lib.USP_F32 if w.dtype == "f32" else _lib.USP_BF16
    md = _lib.USP_FUSED if mode == "fused" else _lib.USP_MATERIALISED
    need = L.usp_attention_joint_workspace_bytes(B, H, N, Nt, D, w.ulysses, w.ring, dt, md, int(text_queries))
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
    p = lambda t: None if t is None else t.data_ptr()
    rc = L.usp_attention_fwd_joint(
        p(st[0]), p(st[1]), p(st[2]), p(txt["q_txt"]) if text_queries else None, p(txt["k_txt"]),
        p(txt["v_txt"]), oc.view.data_ptr(), lc.view.data_ptr(), p(otc.view) if otc else None,
        p(ltc.view) if ltc else None, B, H, N, Nt, D, w.ulysses, w.ring, w.scale, dt, md,
        ws.data_ptr() if need else None, need, torch.cuda.current_stream().cuda_stream)
    assert rc == 0, _lib.lib().usp_status_string(rc)
    assert usp.device_status() == 0
    for c in cans:
        c.check()
    res = (oc.view, lc.view)
    if text_queries:
        res += (otc.view, ltc.view)
    return res


SMALL = [
    ("bf16", 1, 2, 512, 256, 2, 2),
    ("bf16", 2, 6, 960, 77, 3, 2),      # text shorter than one tile; ragged image shards
    ("bf16", 1, 8, 800, 300, 8, 1),     # shards shorter than one tile, ragged text
    ("bf16", 1, 2, 1000, 130, 2, 4),    # Ns = 125
    ("f32", 1, 4, 96, 40, 2, 3),
    ("f32", 2, 2, 50, 7, 1, 5),
]


@pytest.mark.parametrize("dtype,B,H,N,Nt,u,r", SMALL)
@pytest.mark.parametrize("mode", ["materialised", "fused"])
def test_joint_small_full_rows(dtype, B, H, N, Nt, u, r, mode):
    D = 128 if dtype == "bf16" else 32
    w = wl.custom("joint", dtype, B, H, N, D, u, r, seed=N + 3 * Nt, Nt=Nt)
    inp = wl.make_inputs(w)
    txt = wl.make_text_inputs(w)
    stacks = [wl.to_token_stack(inp[n], u, r) for n in ("q", "k", "v")]
    ref = oracle.usp_forward_joint(*[f64(t) for t in stacks], f64(txt["k_txt"]), f64(txt["v_txt"]), u, r,
                                   w.scale, q_txt=f64(txt["q_txt"]))
    st = [t.cuda() for t in stacks]
    txt_d = {n: t.cuda() for n, t in txt.items()}
    for tq in (True, False):
        got = _joint_c(w, st, txt_d, mode, tq)
        tag = f"{mode} {dtype} B{B} H{H} N{N} Nt{Nt} u{u} r{r} text_q={tq}"
        check_out(got[0], got[1], ref[0], ref[1], dtype, "image " + tag)
        if tq:
            check_out(got[2], got[3], ref[2], ref[3], dtype, "text " + tag)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("mode", ["materialised", "fused"])
def test_joint_no_image_tokens(dtype, mode):
    """N = 0: the text queries attend to the text keys alone."""
    D = 128 if dtype == "bf16" else 64
    w = wl.custom("joint0", dtype, 1, 4, 0, D, 2, 2, seed=11, Nt=200)
    txt = wl.make_text_inputs(w)
    empty = torch.empty(w.stack_shape, dtype=w.torch_dtype, device="cuda")
    got = _joint_c(w, [empty] * 3, {n: t.cuda() for n, t in txt.items()}, mode, True)
    ro, rl = oracle.attention(f64(txt["q_txt"]), f64(txt["k_txt"]), f64(txt["v_txt"]), w.scale)
    check_out(got[2], got[3], ro, rl, dtype, f"text only {mode} {dtype}")


@pytest.mark.parametrize("mode", ["materialised", "fused"])
def test_joint_without_text_is_plain_usp(mode):
    """Nt = 0 is usp_attention_fwd: bitwise the same result."""
    usp = _usp()
    w = wl.custom("joint_nt0", "bf16", 1, 4, 1024, 128, 2, 2, seed=5)
    inp = wl.make_inputs(w)
    st = [wl.to_token_stack(inp[n], 2, 2).cuda() for n in ("q", "k", "v")]
    empty = torch.empty((1, 4, 0, 128), dtype=torch.bfloat16, device="cuda")
    o1, l1 = usp.attention_fwd_joint(*st, empty, empty, 2, 2, w.scale, mode=mode)
    o2, l2 = usp.attention_fwd(*st, 2, 2, w.scale, mode=mode)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(l1, l2)


@pytest.mark.parametrize("name", wl.JOINT)
def test_joint_workloads_sampled(name):
    """Full-size joint workloads, both modes, against one oracle evaluation."""
    w = wl.WORKLOADS[name]
    inp = wl.make_inputs(w)
    txt = wl.make_text_inputs(w)
    st = [wl.to_token_stack(inp[n], w.ulysses, w.ring).cuda() for n in ("q", "k", "v")]
    txt_d = {n: t.cuda() for n, t in txt.items()}
    rows = wl.sample_rows(w, 4096)
    BH = w.B * w.H
    f = lambda t, n: t.reshape(BH, n, w.D).float().numpy()
    kcat = np.concatenate([f(txt["k_txt"], w.Nt), f(inp["k"], w.N)], axis=1)
    vcat = np.concatenate([f(txt["v_txt"], w.Nt), f(inp["v"], w.N)], axis=1)
    # image rows, then every text row, through one oracle call
    qsel = np.concatenate([f(inp["q"], w.N)[:, rows.numpy()], f(txt["q_txt"], w.Nt)], axis=1)
    ro, rl = pool.sampled_attention(qsel, kcat, vcat, np.arange(qsel.shape[1]), w.scale)
    R = len(rows)
    for mode in ("materialised", "fused"):
        o, l, ot, lt = _joint_c(w, st, txt_d, mode, True)
        go = wl.from_token_stack(o).reshape(BH, w.N, w.D)[:, rows.cuda()]
        gl = wl.from_token_stack(l).reshape(BH, w.N)[:, rows.cuda()]
        check_out(go, gl, ro[:, :R], rl[:, :R], w.dtype, f"{name} {mode} image")
        check_out(ot.reshape(BH, w.Nt, w.D), lt.reshape(BH, w.Nt), ro[:, R:], rl[:, R:], w.dtype,
                  f"{name} {mode} text")
        del o, l, ot, lt
        torch.cuda.empty_cache()


def test_joint_host_buffers_end_to_end():
    """CPU tensors in, CPU tensors out through the public joint call."""
    usp = _usp()
    w = wl.custom("joint_e2e", "bf16", 1, 4, 1024, 128, 2, 2, seed=9, Nt=256)
    inp = wl.make_inputs(w)
    txt = wl.make_text_inputs(w)
    stacks = [wl.to_token_stack(inp[n], 2, 2) for n in ("q", "k", "v")]
    o, l, ot, lt = usp.attention_fwd_joint(*stacks, txt["k_txt"], txt["v_txt"], 2, 2, w.scale,
                                           q_txt=txt["q_txt"], mode="materialised")
    assert not o.is_cuda and not ot.is_cuda
    ref = oracle.usp_forward_joint(*[f64(t) for t in stacks], f64(txt["k_txt"]), f64(txt["v_txt"]), 2, 2,
                                   w.scale, q_txt=f64(txt["q_txt"]))
    check_out(o, l, ref[0], ref[1], "bf16", "joint host e2e image")
    check_out(ot, lt, ref[2], ref[3], "bf16", "joint host e2e text")


CROSS = [
    ("bf16", 1, 2, 512, 77, 2, 2),
    ("bf16", 2, 6, 960, 300, 3, 2),
    ("bf16", 1, 8, 800, 128, 8, 1),
    ("f32", 1, 4, 96, 40, 2, 3),
    ("f32", 2, 2, 50, 1, 1, 5),        # a single text token
]


@pytest.mark.parametrize("dtype,B,H,N,Nt,u,r", CROSS)
def test_cross_attention_small_full_rows(dtype, B, H, N, Nt, u, r):
    usp = _usp()
    from diffusion_transformer_sequence_gb300 import _lib
    D = 128 if dtype == "bf16" else 32
    w = wl.custom("cross", dtype, B, H, N, D, u, r, seed=N + 5 * Nt, Nt=Nt)
    inp = wl.make_inputs(w, with_dout=False)
    txt = wl.make_text_inputs(w)
    tq = wl.to_token_stack(inp["q"], u, r)
    ro, rl = oracle.usp_cross_attention(f64(tq), f64(txt["k_txt"]), f64(txt["v_txt"]), u, r, w.scale)
    oc = Canary(w.stack_shape, w.torch_dtype)
    lc = Canary(w.lse_stack_shape, torch.float32)
    kt, vt = txt["k_txt"].cuda(), txt["v_txt"].cuda()
    rc = usp.lib().usp_cross_attention_fwd(
        tq.cuda().data_ptr(), kt.data_ptr(), vt.data_ptr(), oc.view.data_ptr(), lc.view.data_ptr(), B, H, N, Nt, D,
        u, r, w.scale, _lib.USP_F32 if dtype == "f32" else _lib.USP_BF16, torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    assert usp.device_status() == 0
    oc.check()
    lc.check()
    check_out(oc.view, lc.view, ro, rl, dtype, f"cross {dtype} B{B} H{H} N{N} Nt{Nt} u{u} r{r}")


def test_cross_attention_wan720p_sampled():
    """Wan 720p image queries (B1 H40 N75600, u8 x r2) against 512 replicated
    text tokens, 4096 sampled query rows per head, through the public call."""
    usp = _usp()
    w = wl.WORKLOADS["wan720p_joint"]
    inp = wl.make_inputs(w, with_dout=False)
    txt = wl.make_text_inputs(w)
    q = wl.to_token_stack(inp["q"], w.ulysses, w.ring).cuda()
    o, l = usp.cross_attention_fwd(q, txt["k_txt"].cuda(), txt["v_txt"].cuda(), w.ulysses, w.ring, w.scale)
    assert usp.device_status() == 0
    rows = wl.sample_rows(w, 4096)
    BH = w.B * w.H
    go = wl.from_token_stack(o).reshape(BH, w.N, w.D)[:, rows.cuda()]
    gl = wl.from_token_stack(l).reshape(BH, w.N)[:, rows.cuda()]
    f = lambda t, n: t.reshape(BH, n, w.D).float().numpy()
    ro, rl = pool.sampled_attention(f(inp["q"], w.N), f(txt["k_txt"], w.Nt), f(txt["v_txt"], w.Nt), rows.numpy(),
                                    w.scale)
    check_out(go, gl, ro, rl, w.dtype, "cross wan720p")
