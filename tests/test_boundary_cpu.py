"""C-ABI boundary tests that need no GPU: the library builds and loads, exports
every symbol include/usp.h declares, and rejects invalid arguments on the host
before touching CUDA (the USP PR page's Limitations: every configuration
outside the supported envelope fails loudly)."""
import ctypes

import pytest

from tests.helpers import ensure_built


@pytest.fixture(scope="module")
def L():
    ensure_built()
    from diffusion_transformer_sequence_gb300 import _lib
    return _lib.lib()


def test_exports_every_declared_symbol(L):
    from diffusion_transformer_sequence_gb300 import _lib
    declared = _lib.header_symbols()
    assert len(declared) >= 11
    handle = ctypes.CDLL(_lib.LIB_PATH)
    for name in declared:
        assert hasattr(handle, name), f"libusp.so does not export {name}"
    assert set(declared) == set(_lib.SIGNATURES), "binding signatures out of sync with usp.h"


def test_boundary_names_of_the_scope_table(L):
    """The C ABI carries every entry point the hot path's scope names,
    including the bounded-wait test hook under its listed name (the earlier
    name stays as an alias)."""
    for name in ("usp_relayout_tok2head", "usp_relayout_head2tok", "usp_attn_chunk_fwd", "usp_lse_merge",
                 "usp_attention_workspace_bytes", "usp_attention_fwd", "usp_attention_bwd",
                 "usp_status_string", "usp_last_cuda_error", "usp_set_debug_spin_limit", "usp_set_spin_limit"):
        assert hasattr(L, name), name
    L.usp_set_debug_spin_limit(-1)   # host-side only: restores the default poll limit


def _header_prototypes():
    """name -> list of (C type of each parameter) parsed from include/usp.h."""
    import re
    from diffusion_transformer_sequence_gb300 import _lib
    txt = open(_lib.HEADER).read()
    txt = re.sub(r"/\*.*?\*/", " ", txt, flags=re.S)          # drop comments
    protos = {}
    for m in re.finditer(r"([A-Za-z_][A-Za-z0-9_ \*]*?)\b(usp_[a-z0-9_]+)\s*\(([^;{]*?)\)\s*;", txt):
        args = [a.strip() for a in re.sub(r"\s+", " ", m.group(3)).split(",")]
        protos[m.group(2)] = [] if args == ["void"] or args == [""] else args
    return protos


def test_binding_signatures_match_header():
    """Every ctypes signature has the header's parameter count, and each
    parameter's ctypes type has the width and kind of its C type."""
    import ctypes
    from diffusion_transformer_sequence_gb300 import _lib
    protos = _header_prototypes()
    assert set(protos) == set(_lib.SIGNATURES)
    for name, (res, args) in _lib.SIGNATURES.items():
        cargs = protos[name]
        assert len(cargs) == len(args), f"{name}: header has {len(cargs)} parameters, binding {len(args)}"
        for c, t in zip(cargs, args):
            ctype = c.rsplit(" ", 1)[0]
            if "*" in c or "usp_stream_t" in c:   # every pointer (and the stream handle) passes as an address
                assert t is ctypes.c_void_p or issubclass(t, ctypes._Pointer), \
                    f"{name}: pointer parameter {c!r} bound as {t}"
            elif "int64_t" in ctype:
                assert t is ctypes.c_int64, f"{name}: {c!r} bound as {t}"
            elif "size_t" in ctype:
                assert t is ctypes.c_size_t, f"{name}: {c!r} bound as {t}"
            elif "float" in ctype:
                assert t is ctypes.c_float, f"{name}: {c!r} bound as {t}"
            elif "long long" in ctype:
                assert t is ctypes.c_longlong, f"{name}: {c!r} bound as {t}"
            else:   # int and the enums (usp_dtype, usp_mode)
                assert t is ctypes.c_int, f"{name}: {c!r} bound as {t}"


def test_status_strings(L):
    from diffusion_transformer_sequence_gb300 import _lib
    for code, name in [(0, "USP_OK"), (1, "USP_ERR_INVALID_ARG"), (2, "USP_ERR_DIVISIBILITY"),
                       (3, "USP_ERR_UNSUPPORTED"), (4, "USP_ERR_WORKSPACE"), (5, "USP_ERR_CUDA"),
                       (6, "USP_ERR_TIMEOUT")]:
        assert L.usp_status_string(code).decode() == name
    assert L.usp_last_cuda_error() == 0


FAKE = 0x10000  # never dereferenced: every call below is rejected on the host


@pytest.mark.parametrize("fn", ["usp_relayout_tok2head", "usp_relayout_head2tok"])
def test_relayout_validation(L, fn):
    f = getattr(L, fn)
    assert f(FAKE, FAKE, 1, 6, 256, 32, 4, 1, 0, None) == 2      # H % ulysses
    assert f(FAKE, FAKE, 1, 8, 250, 32, 4, 1, 0, None) == 2      # N % sp
    assert f(FAKE, FAKE, 1, 8, 256, 32, 2, 3, 0, None) == 2      # N % (u*r)
    assert f(FAKE, FAKE, 1, 8, 256, 32, 0, 1, 0, None) == 1      # ulysses < 1
    assert f(FAKE, FAKE, 1, 8, 256, 32, 1, 0, 0, None) == 1      # ring < 1
    assert f(FAKE, FAKE, -1, 8, 256, 32, 1, 1, 0, None) == 1     # negative size
    assert f(FAKE, FAKE, 1, 8, 256, 0, 1, 1, 0, None) == 1       # D < 1
    assert f(None, FAKE, 1, 8, 256, 32, 4, 1, 0, None) == 1      # null src
    assert f(FAKE, None, 1, 8, 256, 32, 4, 1, 0, None) == 1      # null dst
    assert f(FAKE, FAKE, 1, 8, 256, 32, 4, 1, 7, None) == 3      # unknown dtype
    assert f(None, None, 0, 8, 256, 32, 4, 1, 0, None) == 0      # empty problem: no-op
    assert f(None, None, 1, 8, 0, 32, 4, 1, 0, None) == 0


def test_chunk_validation(L):
    f = L.usp_attn_chunk_fwd
    a = (FAKE, FAKE, FAKE, FAKE, FAKE)
    assert f(*a, 1, 2, 256, 0, 128, 0.1, 1, None) == 1           # no keys
    assert f(*a, 1, 2, 256, 256, 64, 0.1, 1, None) == 3          # bf16 needs D = 128
    assert f(*a, 1, 2, 256, 256, 256, 0.1, 0, None) == 3         # fp32 D > 128
    assert f(*a, 1, 2, 256, 256, 128, float("nan"), 1, None) == 1
    assert f(*a, 1, 2, 256, 256, 128, float("inf"), 1, None) == 1
    assert f(FAKE, FAKE, FAKE, FAKE, None, 1, 2, 256, 256, 128, 0.1, 1, None) == 1
    assert f(FAKE + 8, FAKE, FAKE, FAKE, FAKE, 1, 2, 256, 256, 128, 0.1, 1, None) == 1  # misaligned for TMA
    assert f(None, None, None, None, None, 1, 2, 0, 256, 128, 0.1, 1, None) == 0     # no queries: no-op


def test_merge_validation(L):
    f = L.usp_lse_merge
    assert f(FAKE, FAKE, 0, FAKE, FAKE, 1, 2, 8, 128, 1, None) == 1   # R < 1
    assert f(None, FAKE, 2, FAKE, FAKE, 1, 2, 8, 128, 1, None) == 1
    assert f(FAKE, FAKE, 2, FAKE, FAKE, 1, 2, 8, 128, 9, None) == 3
    assert f(None, None, 2, None, None, 1, 2, 0, 128, 1, None) == 0


def test_attention_validation_and_workspace(L):
    f = L.usp_attention_fwd
    a = (FAKE, FAKE, FAKE, FAKE, FAKE)
    assert f(*a, 1, 40, 32768, 128, 16, 1, 0.1, 1, 0, None, 0, None) == 2   # ulysses > H (40 % 16)
    assert f(*a, 1, 40, 32770, 128, 8, 4, 0.1, 1, 0, None, 0, None) == 2    # N % sp
    assert f(*a, 1, 40, 32768, 128, 8, 4, 0.1, 1, 5, None, 0, None) == 1    # bad mode
    assert f(*a, 1, 40, 32768, 64, 8, 4, 0.1, 1, 0, None, 0, None) == 3     # bf16 D != 128
    assert f(*a, 1, 40, 32768, 128, 8, 4, 0.1, 1, 0, None, 0, None) == 4    # no workspace
    ws = L.usp_attention_workspace_bytes(1, 40, 32768, 128, 8, 4, 1, 0, 0)
    t = 40 * 32768 * 128 * 2
    lb = 40 * 32768 * 4
    assert ws == 3 * t + 4 * t + 4 * lb          # head-sharded q, k, v and the ring partials (merged into out)
    assert f(*a, 1, 40, 32768, 128, 8, 4, 0.1, 1, 0, FAKE, ws - 1, None) == 4
    assert L.usp_attention_workspace_bytes(1, 40, 32768, 128, 8, 4, 1, 1, 0) == 0   # fused: none
    assert L.usp_attention_workspace_bytes(1, 24, 16384, 128, 4, 1, 1, 0, 0) == 4 * 24 * 16384 * 128 * 2 + 24 * 16384 * 4
    assert L.usp_attention_workspace_bytes(1, 6, 256, 128, 4, 1, 1, 0, 0) == 0      # invalid -> 0
    assert f(None, None, None, None, None, 1, 8, 0, 32, 4, 1, 0.1, 0, 1, None, 0, None) == 0  # empty


def test_backward_validation_and_workspace(L):
    a = (FAKE,) * 5 + (FAKE,) * 4
    for f in (L.usp_attention_bwd, L.usp_attention_bwd_materialised):
        assert f(*a, 1, 40, 32768, 128, 16, 1, 0.1, 1, None, 0, None) == 2   # ulysses > H (40 % 16)
        assert f(*a, 1, 40, 32770, 128, 8, 4, 0.1, 1, None, 0, None) == 2    # N % sp
        assert f(*a, 1, 40, 32768, 64, 8, 4, 0.1, 1, None, 0, None) == 3     # bf16 D != 128
        assert f(*a, 1, 40, 32768, 128, 8, 4, float("nan"), 1, None, 0, None) == 1
        assert f(*a, 1, 40, 32768, 128, 8, 4, 0.1, 1, None, 0, None) == 4    # no workspace
        assert f(*((None,) * 9), 1, 8, 0, 32, 4, 1, 0.1, 0, None, 0, None) == 0  # empty
    # fused: Delta and lse*log2(e), rows of each (rank, head) padded to 4
    fused = L.usp_attention_workspace_bytes(1, 40, 32768, 128, 8, 4, 1, 1, 1)
    assert fused == 2 * 32 * 40 * 1024 * 4
    # materialised: q, k, v, O, dO, dq, dk, dv head-sharded, the lse, and the
    # two vectors over [ring * ulysses][B * Hu][Nr]
    mat = L.usp_attention_workspace_bytes(1, 40, 32768, 128, 8, 4, 1, 0, 1)
    t = 40 * 32768 * 128 * 2
    assert mat == 8 * t + 40 * 32768 * 4 + 2 * 4 * 40 * 8192 * 4
    assert L.usp_attention_bwd_materialised(*a, 1, 40, 32768, 128, 8, 4, 0.1, 1, FAKE, mat - 1, None) == 4
    # Nr = 75600 / 2 = 37800 rows per ring chunk (a multiple of 4 already)
    assert L.usp_attention_workspace_bytes(1, 40, 75600, 128, 8, 2, 1, 0, 1) == \
        8 * 40 * 75600 * 128 * 2 + 40 * 75600 * 4 + 2 * 2 * 40 * 37800 * 4
    # ragged: Nr = 6 rows pad to 8, every buffer rounded to 256 bytes
    got = L.usp_attention_workspace_bytes(1, 4, 12, 32, 2, 2, 0, 0, 1)
    rnd = lambda x: (x + 255) // 256 * 256
    assert got == 8 * rnd(4 * 12 * 32 * 4) + rnd(4 * 12 * 4) + 2 * rnd(2 * 4 * 8 * 4)


def test_grid_limits(L):
    """One past the largest launch grid (B*H = 65536 units) is rejected on the host."""
    a = (FAKE,) * 5
    assert L.usp_attention_fwd(*a, 2, 32768, 16, 128, 1, 1, 0.1, 1, 1, None, 0, None) == 3   # fused
    ws = L.usp_attention_workspace_bytes(2, 32768, 16, 128, 1, 1, 1, 0, 0)
    assert L.usp_attention_fwd(*a, 2, 32768, 16, 128, 1, 1, 0.1, 1, 0, FAKE, ws, None) == 3   # materialised
    g = (FAKE,) * 9
    ws = L.usp_attention_workspace_bytes(2, 32768, 16, 128, 1, 1, 1, 1, 1)
    assert L.usp_attention_bwd(*g, 2, 32768, 16, 128, 1, 1, 0.1, 1, FAKE, ws, None) == 3
    ws = L.usp_attention_workspace_bytes(2, 32768, 16, 128, 1, 1, 1, 0, 1)
    assert L.usp_attention_bwd_materialised(*g, 2, 32768, 16, 128, 1, 1, 0.1, 1, FAKE, ws, None) == 3
    # materialised forward: r*r*u*B*Hu units (here 2*2*1*B*H) past the grid
    ws = L.usp_attention_workspace_bytes(1, 16384, 32, 128, 1, 2, 1, 0, 0)
    assert L.usp_attention_fwd(*a, 1, 16384, 32, 128, 1, 2, 0.1, 1, 0, FAKE, ws, None) == 3


def test_joint_validation_and_workspace(L):
    f = L.usp_attention_fwd_joint
    img = (FAKE, FAKE, FAKE)
    txt = (FAKE, FAKE, FAKE)
    outs = (FAKE, FAKE, FAKE, FAKE)
    base = (1, 24, 4096, 512, 128, 2, 2, 0.1, 1)
    assert f(*img, *txt, *outs, 1, 24, 4096, -1, 128, 2, 2, 0.1, 1, 0, None, 0, None) == 1   # negative Nt
    assert f(*img, *txt, *outs, 1, 24, 4098, 512, 128, 2, 2, 0.1, 1, 0, None, 0, None) == 2  # N % sp
    assert f(*img, *txt, *outs, 1, 24, 4096, 512, 64, 2, 2, 0.1, 1, 0, None, 0, None) == 3   # bf16 D != 128
    assert f(*img, FAKE, None, FAKE, *outs, *base, 0, None, 0, None) == 1                      # k_txt missing
    assert f(*img, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, *base, 0, None, 0, None) == 1     # out_txt missing
    assert f(*img, *txt, *outs, *base, 0, None, 0, None) == 4                                   # no workspace
    assert f(*img, *txt, *outs, *base, 7, None, 0, None) == 1                                   # bad mode
    assert f(*img, FAKE + 2, FAKE, FAKE, *outs, *base, 1, None, 0, None) == 1                  # misaligned q_txt
    t, lb = 24 * 4096 * 128 * 2, 24 * 4096 * 4
    tt, tlb = 24 * 512 * 128 * 2, 24 * 512 * 4
    ws = L.usp_attention_joint_workspace_bytes(1, 24, 4096, 512, 128, 2, 2, 1, 0, 1)
    assert ws == 3 * t + 3 * t + 3 * lb + 3 * tt + 3 * tlb
    assert L.usp_attention_joint_workspace_bytes(1, 24, 4096, 512, 128, 2, 2, 1, 0, 0) == ws - 3 * tt - 3 * tlb
    assert f(*img, *txt, *outs, *base, 0, FAKE, ws - 1, None) == 4
    assert L.usp_attention_joint_workspace_bytes(1, 24, 4096, 512, 128, 2, 2, 1, 1, 1) == 0   # fused: none
    assert L.usp_attention_joint_workspace_bytes(1, 24, 4096, 0, 128, 2, 2, 1, 0, 1) == \
        L.usp_attention_workspace_bytes(1, 24, 4096, 128, 2, 2, 1, 0, 0)                        # Nt = 0
    assert f(None, None, None, None, FAKE, FAKE, None, None, None, None, 0, 24, 4096, 512, 128, 2, 2, 0.1, 1, 1,
             None, 0, None) == 0                                                                # empty batch


def test_cross_attention_validation(L):
    f = L.usp_cross_attention_fwd
    a = (FAKE, FAKE, FAKE, FAKE, FAKE)
    assert f(*a, 1, 40, 75600, 0, 128, 8, 2, 0.1, 1, None) == 1        # no text keys
    assert f(*a, 1, 40, 75601, 512, 128, 8, 2, 0.1, 1, None) == 2     # N % sp
    assert f(*a, 1, 40, 75600, 512, 64, 8, 2, 0.1, 1, None) == 3      # bf16 D != 128
    assert f(*a, 1, 40, 75600, 512, 128, 8, 2, float("nan"), 1, None) == 1
    assert f(FAKE + 8, *a[1:], 1, 40, 75600, 512, 128, 8, 2, 0.1, 1, None) == 1   # misaligned q
    assert f(None, None, None, None, None, 1, 40, 0, 512, 128, 8, 2, 0.1, 1, None) == 0  # empty


def test_fp8_validation_and_workspace(L):
    q = L.usp_quantize_e4m3
    assert q(FAKE, FAKE, FAKE, 1, 24, 4096, 120, 2, 2, None) == 3     # D % 16
    assert q(FAKE, FAKE, FAKE, 1, 24, 4098, 128, 2, 2, None) == 2     # N % sp
    assert q(FAKE + 8, FAKE, FAKE, 1, 24, 4096, 128, 2, 2, None) == 1  # misaligned
    assert q(None, None, FAKE, 0, 24, 4096, 128, 2, 2, None) == 0     # empty
    ws = L.usp_attention_fp8_workspace_bytes(1, 24, 4096, 128, 2, 2)
    assert ws == 3 * (4 * 24 * 1024 * 128) + 512                       # q, k codes, V^T codes, amax (256-aligned)
    # Ns = 4725 (Wan 720p, u8 x r2): V^T rows padded to 4736
    assert L.usp_attention_fp8_workspace_bytes(1, 40, 75600, 128, 8, 2) == \
        2 * ((16 * 40 * 4725 * 128 + 255) // 256 * 256) + (16 * 40 * 128 * 4736 + 255) // 256 * 256 + 512
    assert L.usp_attention_fp8_workspace_bytes(1, 24, 4096, 64, 2, 2) == 0
    f = L.usp_attention_fwd_fp8
    a = (FAKE, FAKE, FAKE, FAKE, FAKE)
    assert f(*a, 1, 24, 4096, 64, 2, 2, 0.1, None, 0, None) == 3       # D != 128
    assert f(*a, 1, 24, 4096, 128, 2, 2, float("inf"), None, 0, None) == 1
    assert f(*a, 1, 24, 4096, 128, 2, 2, 0.1, None, 0, None) == 4      # no workspace
    assert f(*a, 1, 24, 4096, 128, 2, 2, 0.1, FAKE, ws - 1, None) == 4
    assert f(*a, 1, 23, 4096, 128, 2, 2, 0.1, FAKE, ws, None) == 2     # H % ulysses


def test_product_path_does_not_import_oracle():
    import subprocess
    import sys
    code = ("import sys, diffusion_transformer_sequence_gb300 as u; u.lib(); "
            "import diffusion_transformer_sequence_gb300.api, diffusion_transformer_sequence_gb300.workloads; "
            "assert not any(m == 'oracle' or m.startswith('oracle.') for m in sys.modules), sorted(sys.modules)")
    subprocess.run([sys.executable, "-c", code], check=True)


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    from diffusion_transformer_sequence_gb300 import _lib
    monkeypatch.setattr(_lib, "_LIB", None)
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "libusp.so"))
    with pytest.raises(RuntimeError, match="no fallback"):
        _lib.lib()
