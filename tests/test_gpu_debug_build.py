"""The debug build (libfv_debug.so, FV_DEBUG_CHECKS=1): the same kernels with
in-kernel index checks compiled in -- tile coordinates against N and the
head range, tensor-memory columns against the allocation, kept-tile list
entries against the grid.  On the ragged lengths and the windowed and
block-sparse variants no check may fire (the status word stays clear), and
the outputs still match the oracle and, bit for bit, the release build."""
import ctypes
import math

import numpy as np
import pytest
import torch

import video_diffusion_transformer_gb300 as fv
from tests import parity as P

pytestmark = pytest.mark.gpu
SCALE = 1.0 / math.sqrt(128)


@pytest.fixture(scope="module")
def dbg(cuda_ok):
    from video_diffusion_transformer_gb300 import build
    build.build()
    build.build(debug=True)
    fv.load_library()
    return fv.load_library(fv.DEBUG_LIB_PATH)


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _rand(n, heads, seed):
    g = torch.Generator().manual_seed(seed)
    return [torch.randn((n, heads * 128), generator=g).to(torch.bfloat16) for _ in range(3)]


def _sync(lib):
    rc = lib.fv_sync_status(_stream())
    assert rc == 0, fv.STATUS.get(rc, rc)


@pytest.mark.parametrize("n", [1, 2, 127, 129, 255, 1000])
def test_debug_build_dense_ragged_lengths(dbg, n):
    heads = 2
    q, k, v = _rand(n, heads, 300 + n)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o = torch.empty_like(qd)
    lse = torch.empty((heads, n), dtype=torch.float32, device="cuda")
    rc = dbg.fv_attn_fwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), n, heads, 128, SCALE, 1,
                         lse.data_ptr(), _stream())
    assert rc == 0
    _sync(dbg)
    P.assert_attention_ok(P.attention_errors(q, k, v, o, heads, 0, SCALE, lse))
    ref = fv.attn_fwd(qd, kd, vd, head_group=1)
    fv.sync_status()
    assert torch.equal(o, ref)


def test_debug_build_window(dbg):
    t_f, frames, heads = 96, 11, 2
    n = t_f * frames
    q, k, v = _rand(n, heads, 401)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o = torch.empty_like(qd)
    rc = dbg.fv_attn_fwd_window(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), n, heads, 128, SCALE,
                                heads, t_f, 2, 1, None, _stream())
    assert rc == 0
    _sync(dbg)
    ref = fv.attn_fwd_window(qd, kd, vd, frame_tokens=t_f, chunk_frames=2, window_chunks=1, head_group=heads)
    fv.sync_status()
    assert torch.equal(o, ref)


def test_debug_build_vsa(dbg):
    from tests import test_gpu_vsa as TV
    grid, heads, topk = (5, 6, 7), 2, 2
    n = grid[0] * grid[1] * grid[2]
    q, k, v = TV.rand(n, heads, 402)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    nt = fv.vsa_num_tiles(*grid)
    o = torch.empty_like(qd)
    sel = torch.empty((heads, nt, topk), dtype=torch.int32, device="cuda")
    need = dbg.fv_vsa_workspace_bytes(heads, *grid, topk)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    rc = dbg.fv_vsa_attn(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), n, heads, 128, SCALE, *grid,
                         topk, sel.data_ptr(), ws.data_ptr(), need, None, _stream())
    assert rc == 0
    _sync(dbg)
    ref, ref_sel = fv.vsa_attn(qd, kd, vd, frames=grid[0], height=grid[1], width=grid[2], topk=topk)
    fv.sync_status()
    assert torch.equal(sel, ref_sel) and torch.equal(o, ref)
    assert np.isfinite(o.float().cpu().numpy()).all()


def test_debug_status_code_is_known(dbg):
    assert fv.STATUS[-10] == "FV_ERR_DEVICE_CHECK"
    assert "debug" in dbg.fv_status_string(-10).decode()
