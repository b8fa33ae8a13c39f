"""fv_attn_fwd_noalloc: the attention entry point for callers that must not
allocate device memory (their memory belongs to a pool they manage, such as a
framework's caching allocator or a serving process with a fixed budget).

It must give what fv_attn_fwd gives, on consecutive calls that reuse the
library's fixed scratch array.  This file is collected last on purpose, so a
run that stops at the first failure has already run every other test.
"""
import ctypes
import math

import pytest
import torch

import video_diffusion_transformer_gb300 as fv
from tests import parity as P

pytestmark = pytest.mark.gpu
SCALE = 1.0 / math.sqrt(128)


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_ok):
    from video_diffusion_transformer_gb300 import build
    build.build()
    fv.load_library()


def _call_noalloc(q, k, v, o, lse, heads, head_group):
    lib = fv.load_library()
    dev_status = ctypes.c_int(-99)
    rc = lib.fv_attn_fwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), q.shape[0], heads, 128,
                                 SCALE, head_group, lse.data_ptr(), torch.cuda.current_stream().cuda_stream,
                                 ctypes.byref(dev_status))
    return rc, dev_status.value


def test_noalloc_matches_allocating_entry_point_on_two_calls():
    n, heads, group = 3000, 10, 4          # 3 launches: 4 + 4 + 2 heads, ragged tail
    g = torch.Generator().manual_seed(77)
    q, k, v = [torch.randn((n, heads * 128), generator=g).to(torch.bfloat16).cuda() for _ in range(3)]
    lse_ref = torch.empty((heads, n), dtype=torch.float32, device="cuda")
    o_ref = fv.attn_fwd(q, k, v, head_group=group, lse=lse_ref)
    fv.sync_status()
    for call in range(2):
        o = torch.full_like(q, float("nan"))
        lse = torch.full_like(lse_ref, float("nan"))
        rc, dev_status = _call_noalloc(q, k, v, o, lse, heads, group)
        assert rc == 0, fv.status_string(rc)
        assert dev_status == 0, fv.status_string(dev_status)
        d = (o.float() - o_ref.float()).abs()
        assert not torch.isnan(o.float()).any()
        assert float(d.max()) <= P.MAX_ABS and float(d.mean()) <= P.MEAN_ABS, (call, float(d.max()))
        assert float((lse - lse_ref).abs().max()) <= P.LSE_ABS


def test_noalloc_rejects_more_launches_than_scratch_words():
    q = torch.zeros((16, 65 * 128), dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((65, 16), dtype=torch.float32, device="cuda")
    rc, _ = _call_noalloc(q, q.clone(), q.clone(), o, lse, 65, 1)   # 65 launches > 64 words
    assert rc == -2
    rc, dev_status = _call_noalloc(q, q.clone(), q.clone(), o, lse, 65, 2)  # 33 launches: fine
    assert rc == 0 and dev_status == 0
