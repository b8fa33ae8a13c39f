"""The C-ABI library loads, exports every symbol include/fv.h declares, and
rejects bad arguments on the host before touching a GPU.  No compute call
runs here: every call below fails validation first (or is host-only)."""
import ctypes
import os
import re

import pytest

import video_diffusion_transformer_gb300 as fv
from video_diffusion_transformer_gb300 import build as fbuild

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "fv.h")


@pytest.fixture(scope="module")
def lib():
    fbuild.build()
    return fv.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fv_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for need in ("fv_attn_fwd", "fv_adaln_modulate", "fv_gated_residual", "fv_step_for_timestep",
                 "fv_sync_status", "fv_status_string"):
        assert need in names
    assert set(names) == set(fv.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert lib.fv_version() >= 100


def test_status_strings(lib):
    for code, name in fv.STATUS.items():
        assert fv.status_string(code).startswith(name)
    assert fv.status_string(-123) == "unknown fv_status"


def test_step_for_timestep():
    ladder = [999.0, 749.0, 500.0, 250.0]
    assert fv.step_for_timestep(ladder, 500.0) == 2
    assert fv.step_for_timestep(ladder, 999.0) == 0
    with pytest.raises(fv.FvError) as e:
        fv.step_for_timestep(ladder, 501.0)
    assert e.value.code == -4


# Fake but well-aligned addresses: validation rejects every call below before
# any CUDA call, so these are never dereferenced.
A = 1 << 40
B = A + (1 << 34)
C = B + (1 << 34)
O = C + (1 << 34)
T = O + (1 << 34)


def attn(lib, q=A, k=B, v=C, o=O, n=1008, h=4, d=128, scale=0.088, g=4, lse=None):
    return lib.fv_attn_fwd(q, k, v, o, n, h, d, scale, g, lse, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), -1), (dict(o=None), -1),
    (dict(d=64), -2), (dict(n=0), -2), (dict(n=-5), -2), (dict(n=1 << 31), -2), (dict(h=0), -2),
    (dict(h=257), -2), (dict(g=0), -2), (dict(g=5), -2),
    (dict(scale=-1.0), -8), (dict(scale=float("nan")), -8), (dict(scale=float("inf")), -8),
    (dict(q=A + 8), -3), (dict(o=O + 2), -3), (dict(lse=T + 2), -3),
    (dict(o=A + 4096), -9), (dict(o=B), -9), (dict(lse=A + 64), -9),
])
def test_attn_rejects_bad_arguments(lib, kw, code):
    assert attn(lib, **kw) == code


def modulate(lib, x=A, y=O, fp32=0, n=1008, c=5376, sh=B, sc=C, ld=5376, steps=8, step=3, eps=1e-6):
    return lib.fv_adaln_modulate(x, y, fp32, n, c, sh, sc, ld, steps, step, eps, None)


@pytest.mark.parametrize("kw,code", [
    (dict(x=None), -1), (dict(sh=None), -1),
    (dict(n=0), -2), (dict(c=5377), -2), (dict(c=8200), -2), (dict(ld=5000), -2), (dict(steps=0), -2),
    (dict(step=8), -4), (dict(step=-1), -4),
    (dict(eps=-1e-6), -8), (dict(eps=float("nan")), -8),
    (dict(x=A + 2), -3), (dict(sh=B + 4), -3), (dict(ld=5378), -3),
    (dict(y=A + 1024), -9),
])
def test_modulate_rejects_bad_arguments(lib, kw, code):
    assert modulate(lib, **kw) == code


def gres(lib, x=A, a=B, out=O, n=5040, c=5376, g=C, ld=5376, steps=8, step=3):
    return lib.fv_gated_residual(x, a, out, n, c, g, ld, steps, step, None)


@pytest.mark.parametrize("kw,code", [
    (dict(a=None), -1), (dict(g=None), -1),
    (dict(n=0), -2), (dict(c=12), -2), (dict(ld=100), -2),
    (dict(step=8), -4),
    (dict(out=O + 8), -3), (dict(g=C + 4), -3),
    (dict(out=B), -9), (dict(out=A + 16), -9),
])
def test_gated_residual_rejects_bad_arguments(lib, kw, code):
    assert gres(lib, **kw) == code


def test_python_binding_requires_cuda_tensors():
    import torch
    q = torch.zeros((128, 128), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fv.attn_fwd(q, q, q)


def test_product_package_never_imports_the_oracle():
    pkg = os.path.dirname(fv.__file__)
    for root, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cc", ".cpp")):
                text = open(os.path.join(root, f)).read()
                assert "oracle" not in text.lower(), f


def window(lib, n=4032, t=1008, c=5, w=1, **kw):
    return lib.fv_attn_fwd_window(A, B, C, O, n, 4, 128, 0.088, 4, t, c, w, None, None)


@pytest.mark.parametrize("kw,code", [
    (dict(t=0), -2), (dict(t=1000), -2), (dict(c=0), -2), (dict(w=-1), -2), (dict(n=0), -2),
])
def test_window_rejects_bad_arguments(lib, kw, code):
    assert window(lib, **kw) == code


def test_window_null_pointers(lib):
    assert lib.fv_attn_fwd_window(None, B, C, O, 4032, 4, 128, 0.088, 4, 1008, 5, 1, None, None) == -1
    assert lib.fv_attn_fwd_window(A, B, C, O, 4032, 4, 128, 0.088, 4, 1008, 5, 1, T + 2, None) == -3
    assert lib.fv_attn_fwd_window(A, B, C, O, 4032, 4, 128, 0.088, 4, 1008, 5, 1, A + 4, None) == -9


def test_tagged_ops_reject_bad_arguments(lib):
    # modulate: missing tags, zero modalities, off-ladder step
    assert lib.fv_adaln_modulate_tagged(A, O, 0, 1008, 5376, B, C, 5376, 8, 3, 3, None, 1e-6, None) == -1
    assert lib.fv_adaln_modulate_tagged(A, O, 0, 1008, 5376, B, C, 5376, 8, 0, 3, T, 1e-6, None) == -2
    assert lib.fv_adaln_modulate_tagged(A, O, 0, 1008, 5376, B, C, 5376, 8, 256, 3, T, 1e-6, None) == -2
    assert lib.fv_adaln_modulate_tagged(A, O, 0, 1008, 5376, B, C, 5376, 8, 3, 8, T, 1e-6, None) == -4
    # gated residual
    assert lib.fv_gated_residual_tagged(A, B, O, 5040, 5376, C, 5376, 8, 3, 3, None, None) == -1
    assert lib.fv_gated_residual_tagged(A, B, O, 5040, 5376, C, 5376, 8, 3, -1, T, None) == -4
    assert lib.fv_gated_residual_tagged(A, B, B, 5040, 5376, C, 5376, 8, 3, 3, T, None) == -9


def vsa(lib, q=A, k=B, v=C, o=O, n=4 * 8 * 12, h=2, d=128, scale=0.088, f=4, hh=8, w=12, topk=2, sel=T,
        ws=T + (1 << 30), wsb=1 << 30, lse=None):
    return lib.fv_vsa_attn(q, k, v, o, n, h, d, scale, f, hh, w, topk, sel, ws, wsb, lse, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), -1), (dict(sel=None), -1), (dict(ws=None), -1),
    (dict(d=64), -2), (dict(f=3), -2), (dict(w=2), -2), (dict(n=4 * 8 * 12 - 1), -2), (dict(topk=0), -2),
    (dict(topk=7), -2), (dict(h=0), -2), (dict(f=4, hh=4, w=4 * 16385, n=4 * 4 * 4 * 16385), -2),
    (dict(scale=0.0), -8), (dict(scale=float("nan")), -8), (dict(wsb=64), -8),
    (dict(q=A + 8), -3), (dict(ws=T + (1 << 30) + 16), -3), (dict(sel=T + 2), -3),
    (dict(o=A), -9), (dict(sel=A + 64), -9), (dict(sel=T + 224, ws=T + 256), -9), (dict(lse=O + 1024), -9),
])
def test_vsa_rejects_bad_arguments(lib, kw, code):
    assert vsa(lib, **kw) == code


def test_vsa_host_helpers_follow_the_printed_count(lib):
    from oracle import vsa as VS
    for grid in [(72, 24, 42), (5, 6, 7), (4, 4, 4), (102, 24, 42)]:
        assert fv.vsa_num_tiles(*grid) == len(VS.tile_tokens(*grid))
    assert fv.vsa_num_tiles(0, 4, 4) == 0 and fv.vsa_num_tiles(4, 4, 4 * 16385) == -1
    for n in (1, 2, 7, 64, 594, 1188, 1716):
        for s in (0.0, 0.5, 0.75, 0.9, 0.95, 1.0, -0.5, 1.5):
            assert fv.vsa_topk(n, s) == VS.topk_count(n, s), (n, s)
    assert fv.vsa_topk(0, 0.9) == 0 and fv.vsa_topk(10, float("nan")) == 0
    assert lib.fv_vsa_workspace_bytes(2, 4, 8, 12, 2) > 0
    assert lib.fv_vsa_workspace_bytes(2, 4, 8, 12, 7) == -1
