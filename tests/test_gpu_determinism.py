"""Run-to-run determinism of every entry point on the GPU, through the C ABI.

The pages run their parity suite in a deterministic mode (the PR page's
"Op-level parity" and deterministic double-runs) and single out atomics as
the only source of run-to-run variation; none of these kernels uses
floating-point atomics, so every call, run twice on the same inputs, must
give bit-identical outputs.  Shapes are small but span several tiles, a
ragged tail and every rank of a 2 x 2 grid."""
import pytest
import torch

from diffusion_transformer_sequence_gb300 import workloads as wl
from tests.helpers import ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()
    assert torch.cuda.is_available()


def _usp():
    import diffusion_transformer_sequence_gb300 as usp
    return usp


def _same(a, b):
    va = a.view(torch.int16) if a.dtype == torch.bfloat16 else a.view(torch.int32)
    vb = b.view(torch.int16) if b.dtype == torch.bfloat16 else b.view(torch.int32)
    return torch.equal(va, vb)


def _twice(fn):
    first = [t.clone() for t in fn()]
    torch.cuda.synchronize()
    second = fn()
    torch.cuda.synchronize()
    return first, second


@pytest.fixture(scope="module")
def inputs():
    w = wl.custom("det", "bf16", 1, 4, 1000, 128, 2, 2, seed=2024, backward=True, Nt=200)  # Ns = 250: ragged
    inp = wl.make_inputs(w)
    txt = wl.make_text_inputs(w)
    st = {n: wl.to_token_stack(t, 2, 2).cuda() for n, t in inp.items()}
    tx = {n: t.cuda() for n, t in txt.items()}
    return w, st, tx


CALLS = ["fwd_fused", "fwd_materialised", "bwd_fused", "bwd_materialised", "joint_fused", "joint_materialised",
         "cross", "fp8"]


@pytest.mark.parametrize("call", CALLS)
def test_double_run_bitwise(inputs, call):
    usp = _usp()
    w, st, tx = inputs
    q, k, v, do = st["q"], st["k"], st["v"], st["dout"]
    if call.startswith("fwd_"):
        fn = lambda: usp.attention_fwd(q, k, v, 2, 2, w.scale, mode=call[4:])
    elif call.startswith("bwd_"):
        o, l = usp.attention_fwd(q, k, v, 2, 2, w.scale, mode="fused")
        fn = lambda: usp.attention_bwd(q, k, v, o, l, do, 2, 2, w.scale, mode=call[4:])
    elif call.startswith("joint_"):
        fn = lambda: [t for t in usp.attention_fwd_joint(q, k, v, tx["k_txt"], tx["v_txt"], 2, 2, w.scale,
                                                         q_txt=tx["q_txt"], mode=call[6:]) if t is not None]
    elif call == "cross":
        fn = lambda: usp.cross_attention_fwd(q, tx["k_txt"], tx["v_txt"], 2, 2, w.scale)
    else:
        fn = lambda: usp.attention_fwd_fp8(q, k, v, 2, 2, w.scale)
    first, second = _twice(fn)
    assert usp.device_status() == 0
    assert len(first) == len(second) and len(first) >= 2
    for i, (a, b) in enumerate(zip(first, second)):
        assert _same(a, b), f"{call}: output {i} differs between two runs"


CAPTURED = ["fwd_materialised", "fwd_fused", "joint_materialised", "fp8"]


@pytest.mark.parametrize("call", CAPTURED)
def test_graph_capture_replays_bitwise(inputs, call):
    """Each call captured into a CUDA graph (its launches chained by
    programmatic dependent launch; the joint call forks its text launch onto
    the side stream) and replayed gives the eager result bit for bit."""
    usp = _usp()
    w, st, tx = inputs
    q, k, v = st["q"], st["k"], st["v"]
    B, H, N, D = w.B, w.H, w.N, w.D
    if call.startswith("fwd_"):
        mode = call[4:]
        ws = torch.empty(max(1, usp.workspace_bytes(B, H, N, D, 2, 2, torch.bfloat16, mode)), dtype=torch.uint8,
                         device="cuda")
        outs = (torch.empty_like(q), torch.empty(w.lse_stack_shape, device="cuda"))
        fn = lambda: usp.attention_fwd(q, k, v, 2, 2, w.scale, mode=mode, out=outs[0], lse=outs[1], workspace=ws)
    elif call == "joint_materialised":
        ws = torch.empty(usp.joint_workspace_bytes(B, H, N, w.Nt, D, 2, 2, torch.bfloat16, "materialised", False),
                         dtype=torch.uint8, device="cuda")
        fn = lambda: usp.attention_fwd_joint(q, k, v, tx["k_txt"], tx["v_txt"], 2, 2, w.scale, mode="materialised",
                                             workspace=ws)
    else:
        L = usp.lib()
        ws = torch.empty(int(L.usp_attention_fp8_workspace_bytes(B, H, N, D, 2, 2)), dtype=torch.uint8, device="cuda")
        outs = (torch.empty_like(q), torch.empty(w.lse_stack_shape, device="cuda"))
        fn = lambda: usp.attention_fwd_fp8(q, k, v, 2, 2, w.scale, out=outs[0], lse=outs[1], workspace=ws)
    ref = [t.clone() for t in fn()]
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):    # warm-up on the capture stream
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        got = fn()
    for _ in range(2):
        for t in got:
            t.zero_()
        g.replay()
        torch.cuda.synchronize()
        for i, (a, b) in enumerate(zip(got, ref)):
            assert _same(a, b), f"{call}: output {i} differs after graph replay"
    assert usp.device_status() == 0
