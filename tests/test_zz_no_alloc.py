"""fv_attn_fwd_noalloc: the attention entry point for callers that must not
allocate device memory (their memory belongs to a pool they manage, such as a
framework's caching allocator or a serving process with a fixed budget).

It must give exactly what fv_attn_fwd gives, on consecutive calls that reuse
the library's fixed scratch array; it must report a device-side timeout
through its own scratch words and clear them for the next call; and a process
that only ever calls it must see no change in free device memory.  This file
is collected last on purpose, so a run that stops at the first failure has
already run every other test.
"""
import ctypes
import json
import math
import os
import subprocess
import sys

import pytest
import torch

import video_diffusion_transformer_gb300 as fv

pytestmark = pytest.mark.gpu
SCALE = 1.0 / math.sqrt(128)
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


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


def _inputs(n, heads, seed):
    g = torch.Generator().manual_seed(seed)
    return [torch.randn((n, heads * 128), generator=g).to(torch.bfloat16).cuda() for _ in range(3)]


def test_noalloc_matches_allocating_entry_point_on_two_calls():
    """Same kernel, same inputs: the outputs must be bit-identical, so reusing
    the scratch array changes nothing."""
    n, heads, group = 3000, 10, 4          # 3 launches: 4 + 4 + 2 heads, ragged tail
    q, k, v = _inputs(n, heads, 77)
    lse_ref = torch.empty((heads, n), dtype=torch.float32, device="cuda")
    o_ref = fv.attn_fwd(q, k, v, head_group=group, lse=lse_ref)
    fv.sync_status()
    for call in range(2):
        o = torch.full_like(q, float("nan"))
        lse = torch.full_like(lse_ref, float("nan"))
        rc, dev_status = _call_noalloc(q, k, v, o, lse, heads, group)
        assert rc == 0, fv.status_string(rc)
        assert dev_status == 0, fv.status_string(dev_status)
        assert torch.equal(o, o_ref), call
        assert torch.equal(lse, lse_ref), call


def test_noalloc_rejects_more_launches_than_scratch_words():
    q = torch.zeros((16, 65 * 128), dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((65, 16), dtype=torch.float32, device="cuda")
    rc, _ = _call_noalloc(q, q.clone(), q.clone(), o, lse, 65, 1)   # 65 launches > 64 words
    assert rc == -2
    rc, dev_status = _call_noalloc(q, q.clone(), q.clone(), o, lse, 65, 2)  # 33 launches: fine
    assert rc == 0 and dev_status == 0


def test_noalloc_reports_a_timeout_and_the_next_call_clears_it():
    """A bounded wait made to run out (the fv_test_skip_load hook, first
    launch of two) is reported through the call's own scratch word as
    FV_ERR_DEVICE_TIMEOUT; the next call clears the words it uses and
    reports nothing, with the exact output of fv_attn_fwd."""
    n, heads = 4096, 2
    q, k, v = _inputs(n, heads, 78)
    o = torch.empty_like(q)
    lse = torch.empty((heads, n), dtype=torch.float32, device="cuda")
    fv.test_skip_load(fv.TEST_ATTN, 5)
    try:
        rc, dev_status = _call_noalloc(q, k, v, o, lse, heads, 1)
    finally:
        fv.test_skip_load(fv.TEST_ATTN, -1)
    assert rc == 0, fv.status_string(rc)
    assert dev_status == -7, fv.status_string(dev_status)
    rc, dev_status = _call_noalloc(q, k, v, o, lse, heads, 1)
    assert rc == 0 and dev_status == 0, (rc, dev_status)
    lse_ref = torch.empty_like(lse)
    o_ref = fv.attn_fwd(q, k, v, head_group=1, lse=lse_ref)
    fv.sync_status()
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)


_FRESH = r"""
import ctypes, json, math, sys
sys.path.insert(0, sys.argv[1])
import torch
import video_diffusion_transformer_gb300 as fv
lib = fv.load_library()            # the library's kernels are registered before the context exists
n, heads = 2048, 4
q, k, v = [torch.randn((n, heads * 128), device="cuda").to(torch.bfloat16) for _ in range(3)]
o = torch.empty_like(q)
lse = torch.empty((heads, n), dtype=torch.float32, device="cuda")
torch.cuda.synchronize()
s = torch.cuda.current_stream().cuda_stream
free0 = torch.cuda.mem_get_info()[0]
codes = []
for _ in range(2):
    st = ctypes.c_int(-99)
    rc = lib.fv_attn_fwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), n, heads, 128,
                                 1.0 / math.sqrt(128), 2, lse.data_ptr(), s, ctypes.byref(st))
    codes.append((rc, st.value))
torch.cuda.synchronize()
free1 = torch.cuda.mem_get_info()[0]
# control: the allocating entry point's first call allocates its status word
rc2 = lib.fv_attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), n, heads, 128,
                      1.0 / math.sqrt(128), 2, None, s)
torch.cuda.synchronize()
free2 = torch.cuda.mem_get_info()[0]
print(json.dumps({"codes": codes, "free0": free0, "free1": free1, "rc2": rc2, "free2": free2}))
"""


def test_noalloc_allocates_nothing_in_a_fresh_process():
    """A process that only calls fv_attn_fwd_noalloc: free device memory is the
    same before and after two calls.  Modules load eagerly (at context
    creation), so no lazy code loading shows up in between; the control call
    to fv_attn_fwd afterwards shows that its one status-word allocation is
    visible to the same measurement."""
    env = dict(os.environ, CUDA_MODULE_LOADING="EAGER")
    res = subprocess.run([sys.executable, "-c", _FRESH, ROOT], capture_output=True, text=True, env=env,
                         timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    r = json.loads(res.stdout.strip().splitlines()[-1])
    assert r["codes"] == [[0, 0], [0, 0]], r
    assert r["free1"] == r["free0"], r
    assert r["rc2"] == 0 and r["free2"] < r["free1"], r
