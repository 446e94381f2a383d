"""GPU parity of usp_attention_bwd and usp_attention_bwd_materialised against
the oracle, through the C ABI.

Small problems: every row of dq, dk, dv against oracle.attention_bwd, with the
backward fed the oracle's own forward (out rounded to the input dtype, lse to
fp32, both on the test side).  Wan shapes (u8 x r4, N = 32768): the GPU
forward feeds the GPU backward; the oracle recomputes everything from q, k,
v, dO and checks 4096 sampled query rows (dq) and 4096 sampled key rows (dk,
dv) on four heads, two of them on either side of a Ulysses head-group
boundary.  Tolerance (no bound is stated for gradients): per tensor
max|err| / max|ref| <= 2e-2 in bf16, max|err| <= 1e-5 in fp32."""
import numpy as np
import pytest
import torch

import oracle
from oracle import pool
from diffusion_transformer_sequence_gb300 import workloads as wl
from tests.helpers import BF16_GRAD_REL, F32_GRAD_ATOL, Canary, ensure_built, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()
    assert torch.cuda.is_available()


def _usp():
    import diffusion_transformer_sequence_gb300 as usp
    return usp


def _check_grad(got, ref, dtype, what):
    g = f64(got)
    assert np.isfinite(g).all(), f"{what}: non-finite"
    err = np.abs(g - ref).max()
    if dtype == "f32":
        assert err <= F32_GRAD_ATOL, f"{what}: max err {err:.3e}"
    else:
        rel = err / max(np.abs(ref).max(), 1e-30)
        assert rel <= BF16_GRAD_REL, f"{what}: rel err {rel:.3e} (abs {err:.3e})"


SMALL = [
    ("bf16", 1, 2, 512, 2, 2),
    ("bf16", 2, 6, 960, 3, 2),     # ragged tiles in every shard
    ("bf16", 1, 8, 800, 8, 1),     # shards shorter than one tile
    ("bf16", 1, 2, 384, 1, 1),
    ("bf16", 1, 2, 1000, 2, 4),    # Ns = 125: row pitch padding of the per-row vectors
    ("f32", 1, 4, 96, 2, 3),
    ("f32", 2, 2, 50, 1, 5),
]


@pytest.mark.parametrize("mode", ["fused", "materialised"])
@pytest.mark.parametrize("dtype,B,H,N,u,r", SMALL)
def test_bwd_small_full_rows(dtype, B, H, N, u, r, mode):
    usp = _usp()
    D = 128 if dtype == "bf16" else 32
    w = wl.custom("bwd", dtype, B, H, N, D, u, r, seed=N + 7 * H, backward=True)
    inp = wl.make_inputs(w)
    q, k, v, do = (inp[n] for n in ("q", "k", "v", "dout"))
    o_ref, l_ref = oracle.attention(f64(q), f64(k), f64(v), w.scale)
    dq_r, dk_r, dv_r = oracle.attention_bwd(f64(q), f64(k), f64(v), o_ref, l_ref, f64(do), w.scale)
    o_in = torch.from_numpy(o_ref).to(w.torch_dtype)
    l_in = torch.from_numpy(l_ref).float()
    st = lambda t: wl.to_token_stack(t, u, r).cuda()
    cans = [Canary(w.stack_shape, w.torch_dtype) for _ in range(3)]
    dq, dk, dv = (c.view for c in cans)
    L = usp.lib()
    from diffusion_transformer_sequence_gb300 import _lib
    need = usp.workspace_bytes(B, H, N, D, u, r, w.torch_dtype, mode=mode, backward=True)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    args = [st(q), st(k), st(v), st(o_in), st(l_in), st(do)]
    fn = L.usp_attention_bwd if mode == "fused" else L.usp_attention_bwd_materialised
    rc = fn(*[a.data_ptr() for a in args], dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, D,
            u, r, w.scale, _lib.USP_F32 if dtype == "f32" else _lib.USP_BF16, ws.data_ptr(), need,
            torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    assert usp.device_status() == 0
    for c in cans:
        c.check()
    for name, got, ref in (("dq", dq, dq_r), ("dk", dk, dk_r), ("dv", dv, dv_r)):
        _check_grad(wl.from_token_stack(got.cpu()), ref, dtype, f"{name} {mode} {dtype} B{B} H{H} N{N} u{u} r{r}")


def test_bwd_wan_shapes_sampled():
    """Wan shapes (B1 H40 N32768 D128, u8 x r4), forward + backward on the GPU."""
    usp = _usp()
    w = wl.WORKLOADS["wan_s32k"]
    inp = wl.make_inputs(w)
    st = {n: wl.to_token_stack(t, w.ulysses, w.ring).cuda() for n, t in inp.items()}
    o, l = usp.attention_fwd(st["q"], st["k"], st["v"], w.ulysses, w.ring, w.scale, mode="fused")
    dq, dk, dv = usp.attention_bwd(st["q"], st["k"], st["v"], o, l, st["dout"], w.ulysses, w.ring, w.scale)
    assert usp.device_status() == 0
    dq2, dk2, dv2 = usp.attention_bwd(st["q"], st["k"], st["v"], o, l, st["dout"], w.ulysses, w.ring, w.scale)
    for a, b in ((dq, dq2), (dk, dk2), (dv, dv2)):    # deterministic: no atomics anywhere
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    # The materialised path re-lays the same tokens out head-sharded; with
    # Ns = 1024 a multiple of the 128-row tile, every tile and every sum runs
    # in the same order, so its gradients equal the fused ones bit for bit.
    mq, mk, mv = usp.attention_bwd(st["q"], st["k"], st["v"], o, l, st["dout"], w.ulysses, w.ring, w.scale,
                                   mode="materialised")
    assert usp.device_status() == 0
    for name, a, b in (("dq", dq, mq), ("dk", dk, mk), ("dv", dv, mv)):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), f"materialised {name} differs from fused"
    heads = [0, 4, 5, 39]   # Hu = 5: heads 4 | 5 sit on either side of a Ulysses group boundary
    qrows = wl.sample_rows(w, 4096)
    g = torch.Generator().manual_seed(w.row_seed + 1)
    krows = torch.unique(torch.cat([qrows[::2], torch.randperm(w.N, generator=g)[:2048]]))
    flat = {n: inp[n].reshape(w.B * w.H, w.N, w.D) for n in inp}
    sel = lambda t, rows: wl.from_token_stack(t).reshape(w.B * w.H, w.N, w.D)[heads][:, rows.cuda()]
    g_dq, g_dk, g_dv = sel(dq, qrows), sel(dk, krows), sel(dv, krows)
    f = lambda n: flat[n].float().numpy()
    r_dq, r_dk, r_dv = pool.sampled_backward(f("q"), f("k"), f("v"), f("dout"), w.scale, heads, qrows.numpy(),
                                             krows.numpy())
    _check_grad(g_dq, r_dq, "bf16", "wan dq")
    _check_grad(g_dk, r_dk, "bf16", "wan dk")
    _check_grad(g_dv, r_dv, "bf16", "wan dv")


def test_bwd_wan720p_sampled():
    """Wan 720p (B1 H40 N75600 D128, u8 x r2; Ns = 4725, so every shard ends in
    a ragged tile), forward + both backward calls on the GPU against the
    oracle at 2048 sampled query rows (dq) and 2048 sampled key rows (dk, dv)
    of two heads on either side of a Ulysses head-group boundary."""
    usp = _usp()
    w = wl.WORKLOADS["wan720p"]
    inp = wl.make_inputs(w, with_dout=True)
    st = {n: wl.to_token_stack(t, w.ulysses, w.ring).cuda() for n, t in inp.items()}
    o, l = usp.attention_fwd(st["q"], st["k"], st["v"], w.ulysses, w.ring, w.scale, mode="fused")
    heads = [4, 5]   # Hu = 5
    qrows = wl.sample_rows(w, 2048)
    g = torch.Generator().manual_seed(w.row_seed + 2)
    krows = torch.unique(torch.cat([qrows[::2], torch.randperm(w.N, generator=g)[:1024]]))
    flat = {n: inp[n].reshape(w.B * w.H, w.N, w.D) for n in inp}
    f = lambda n: flat[n][heads].float().numpy()
    r_dq, r_dk, r_dv = pool.sampled_backward(f("q"), f("k"), f("v"), f("dout"), w.scale, list(range(len(heads))),
                                             qrows.numpy(), krows.numpy())
    for mode in ("fused", "materialised"):
        dq, dk, dv = usp.attention_bwd(st["q"], st["k"], st["v"], o, l, st["dout"], w.ulysses, w.ring, w.scale,
                                       mode=mode)
        assert usp.device_status() == 0
        sel = lambda t, rows: wl.from_token_stack(t).reshape(w.B * w.H, w.N, w.D)[heads][:, rows.cuda()]
        _check_grad(sel(dq, qrows), r_dq, "bf16", f"wan720p {mode} dq")
        _check_grad(sel(dk, krows), r_dk, "bf16", f"wan720p {mode} dk")
        _check_grad(sel(dv, krows), r_dv, "bf16", f"wan720p {mode} dv")
        del dq, dk, dv
        torch.cuda.empty_cache()


@pytest.mark.parametrize("name,heads", [("qwen1024", [0, 11, 12, 23]), ("qwen2048", [0, 5, 6, 23])])
def test_bwd_qwen_workloads_sampled(name, heads):
    """Qwen-Image 1024² (u2 x r2, the benchmark's step) and 2048² (u4 x r1):
    the GPU forward feeds both backward calls at full size; 2048 sampled query
    rows (dq) and 2048 sampled key rows (dk, dv) of four heads, two of them on
    either side of a Ulysses head-group boundary, against the oracle."""
    usp = _usp()
    w = wl.WORKLOADS[name]
    inp = wl.make_inputs(w, with_dout=True)
    st = {n: wl.to_token_stack(t, w.ulysses, w.ring).cuda() for n, t in inp.items()}
    o, l = usp.attention_fwd(st["q"], st["k"], st["v"], w.ulysses, w.ring, w.scale, mode="fused")
    qrows = wl.sample_rows(w, 2048)
    g = torch.Generator().manual_seed(w.row_seed + 3)
    krows = torch.unique(torch.cat([qrows[::2], torch.randperm(w.N, generator=g)[:1024]]))
    flat = {n: inp[n].reshape(w.B * w.H, w.N, w.D) for n in inp}
    f = lambda n: flat[n][heads].float().numpy()
    r_dq, r_dk, r_dv = pool.sampled_backward(f("q"), f("k"), f("v"), f("dout"), w.scale, list(range(len(heads))),
                                             qrows.numpy(), krows.numpy())
    sel = lambda t, rows: wl.from_token_stack(t).reshape(w.B * w.H, w.N, w.D)[heads][:, rows.cuda()]
    for mode in ("fused", "materialised"):
        dq, dk, dv = usp.attention_bwd(st["q"], st["k"], st["v"], o, l, st["dout"], w.ulysses, w.ring, w.scale,
                                       mode=mode)
        assert usp.device_status() == 0
        _check_grad(sel(dq, qrows), r_dq, "bf16", f"{name} {mode} dq")
        _check_grad(sel(dk, krows), r_dk, "bf16", f"{name} {mode} dk")
        _check_grad(sel(dv, krows), r_dv, "bf16", f"{name} {mode} dv")


# (B, H, N, ulysses, ring): Qwen-Image 2048^2 (u4, Ns = 4096), a u8 grid with
# Ns = 256, and a hybrid u2 x r2 grid with Ns = 512.  Every shard is a whole
# number of 128-row tiles.
BITWISE = [(1, 24, 16384, 4, 1), (1, 8, 2048, 8, 1), (2, 4, 2048, 2, 2)]


@pytest.mark.parametrize("B,H,N,u,r", BITWISE)
def test_bwd_sharded_bitwise_equals_unsharded(B, H, N, u, r):
    """The USP PR page (Validation, Numerics) finds Ulysses-only USP equal to
    sp = 1 bit for bit, the input gradients included: the exchange only moves
    data.  Here both backward calls over the sharded stacks, given the same
    forward out and lse, must equal the unsharded (u = r = 1) backward bit for
    bit.  This holds when every shard is a whole number of 128-row tiles: the
    kernels then see the same global tiles in the same order whatever the
    grid.  (With a ragged shard the last tile of each shard is short, the
    per-tile partial sums are grouped differently and results agree to
    rounding only; the small-problem tests above check those grids against
    the oracle.)  The hybrid u x r case checks the same for the backward
    alone: its forward merges ring partials and is not bitwise sp = 1, so
    the test feeds both calls one out and lse."""
    usp = _usp()
    w = wl.custom("bwdbit", "bf16", B, H, N, 128, u, r, seed=31, backward=True)
    assert w.Ns % 128 == 0
    g = {n: t.cuda() for n, t in wl.make_inputs(w, with_dout=True).items()}
    one = {n: wl.to_token_stack(t, 1, 1) for n, t in g.items()}      # u = r = 1: the plain layout
    o, l = usp.attention_fwd(one["q"], one["k"], one["v"], 1, 1, w.scale, mode="fused")
    ref = [wl.from_token_stack(t) for t in
           usp.attention_bwd(one["q"], one["k"], one["v"], o, l, one["dout"], 1, 1, w.scale, mode="fused")]
    st = {n: wl.to_token_stack(t, u, r) for n, t in g.items()}
    so, sl = wl.to_token_stack(wl.from_token_stack(o), u, r), wl.to_token_stack(wl.from_token_stack(l), u, r)
    for mode in ("fused", "materialised"):
        got = usp.attention_bwd(st["q"], st["k"], st["v"], so, sl, st["dout"], u, r, w.scale, mode=mode)
        assert usp.device_status() == 0
        for name, a, b in zip(("dq", "dk", "dv"), got, ref):
            a = wl.from_token_stack(a)
            assert torch.equal(a.view(torch.int16), b.view(torch.int16)), \
                f"{mode} u{u} r{r}: {name} differs from the unsharded backward " \
                f"({int((a != b).sum())} elements, max |diff| {float((a.float() - b.float()).abs().max()):.3e})"


def _small_bwd_inputs(seed=21):
    w = wl.custom("bwdc", "bf16", 1, 4, 1024, 128, 2, 2, seed=seed, backward=True)
    inp = wl.make_inputs(w)
    st = {n: wl.to_token_stack(t, 2, 2).cuda() for n, t in inp.items()}
    return w, st


@pytest.mark.parametrize("mode", ["fused", "materialised"])
def test_bwd_concurrent_kernels_graph_capture(mode):
    """The backward's dQ kernel runs on a library-owned side stream, forked and
    joined with events: captured into a CUDA graph and replayed it must give
    the eager result bit for bit (the materialised call adds its re-layouts
    to the graph)."""
    usp = _usp()
    w, st = _small_bwd_inputs()
    o, l = usp.attention_fwd(st["q"], st["k"], st["v"], 2, 2, w.scale, mode="fused")
    ref = usp.attention_bwd(st["q"], st["k"], st["v"], o, l, st["dout"], 2, 2, w.scale, mode=mode)
    torch.cuda.synchronize()
    ws = torch.empty(usp.workspace_bytes(w.B, w.H, w.N, w.D, 2, 2, torch.bfloat16, mode=mode, backward=True),
                     dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):   # warm-up on the capture stream
        usp.attention_bwd(st["q"], st["k"], st["v"], o, l, st["dout"], 2, 2, w.scale, workspace=ws, mode=mode)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        got = usp.attention_bwd(st["q"], st["k"], st["v"], o, l, st["dout"], 2, 2, w.scale, workspace=ws,
                                mode=mode)
    for _ in range(2):
        for t in got:
            t.zero_()
        g.replay()
        torch.cuda.synchronize()
        for a, b in zip(got, ref):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert usp.device_status() == 0


@pytest.mark.parametrize("mode", ["fused", "materialised"])
def test_bwd_two_host_threads(mode):
    """Two host threads, each on its own stream, share the device's side stream
    (it is locked per call): every result equals the single-thread one."""
    import threading
    usp = _usp()
    w, st = _small_bwd_inputs(seed=22)
    o, l = usp.attention_fwd(st["q"], st["k"], st["v"], 2, 2, w.scale, mode="fused")
    ref = usp.attention_bwd(st["q"], st["k"], st["v"], o, l, st["dout"], 2, 2, w.scale, mode=mode)
    torch.cuda.synchronize()
    errors = []

    def worker():
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                for _ in range(8):
                    got = usp.attention_bwd(st["q"], st["k"], st["v"], o, l, st["dout"], 2, 2, w.scale, mode=mode)
                    s.synchronize()
                    for a, b in zip(got, ref):
                        if not torch.equal(a.view(torch.int16), b.view(torch.int16)):
                            errors.append("mismatch")
        except Exception as e:  # reported below
            errors.append(repr(e))

    ts = [threading.Thread(target=worker) for _ in range(2)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    assert not errors, errors
    assert usp.device_status() == 0
