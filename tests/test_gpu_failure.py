"""Failure detection on the GPU without a fault.  In every kernel that waits
on a copy, a bounded wait is made to run out: the test hook
fv_test_skip_load makes the first CTA of the next launch never issue one
copy.  The call must report FV_ERR_DEVICE_TIMEOUT through the status word,
drain its in-flight copies and MMAs, release tensor memory, and leave the
context usable: the next call in the same process passes parity."""
import math
import time

import numpy as np
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


def _inputs(n=4096, heads=2, seed=21):
    g = torch.Generator().manual_seed(seed)
    return [torch.randn((n, heads * 128), generator=g).to(torch.bfloat16) for _ in range(3)]


def _expect_timeout(kernel, load_index, call):
    """Arm the hook, run the call, and check it reports the device timeout
    within a bounded wall time; the hook is disarmed afterwards either way."""
    fv.sync_status()
    fv.test_skip_load(kernel, load_index)
    try:
        t0 = time.time()
        call()
        with pytest.raises(fv.FvError) as e:
            fv.sync_status()
        elapsed = time.time() - t0
    finally:
        fv.test_skip_load(kernel, -1)
    assert e.value.code == -7, e.value
    assert elapsed < 30.0
    fv.sync_status()  # the read cleared the word


def test_hook_rejects_unknown_kernel_and_is_one_shot():
    with pytest.raises(fv.FvError) as e:
        fv.test_skip_load(99, 0)
    assert e.value.code == -8
    q, k, v = _inputs(n=512)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    _expect_timeout(fv.TEST_ATTN, 1, lambda: fv.attn_fwd(qd, kd, vd, head_group=1))
    # two launches (head_group 1): the first consumed the hook, and now
    # nothing is armed: a plain call reports nothing
    fv.attn_fwd(qd, kd, vd, head_group=1)
    fv.sync_status()


def test_attention_wait_times_out_and_context_survives():
    q, k, v = _inputs()
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    _expect_timeout(fv.TEST_ATTN, 5, lambda: fv.attn_fwd(qd, kd, vd, head_group=2))
    lse = torch.empty((2, q.shape[0]), dtype=torch.float32, device="cuda")
    o = fv.attn_fwd(qd, kd, vd, head_group=2, lse=lse)
    fv.sync_status()
    P.assert_attention_ok(P.attention_errors(q, k, v, o, 2, 64, SCALE, lse))


def test_window_attention_wait_times_out():
    q, k, v = _inputs(n=10 * 96)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    _expect_timeout(fv.TEST_ATTN, 2, lambda: fv.attn_fwd_window(qd, kd, vd, frame_tokens=96, chunk_frames=2,
                                                                 window_chunks=1, head_group=2))
    fv.attn_fwd_window(qd, kd, vd, frame_tokens=96, chunk_frames=2, window_chunks=1, head_group=2)
    fv.sync_status()


def test_vsa_fine_wait_times_out_and_context_survives():
    from tests import test_gpu_vsa as TV
    grid, heads, topk = (8, 8, 12), 2, 3
    n = grid[0] * grid[1] * grid[2]
    q, k, v = TV.rand(n, heads, 5)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    # CTA 0's loads: K_0, K_1, V_0, K_2, ...; V_0 never arrives
    _expect_timeout(fv.TEST_VSA_FINE, 2,
                    lambda: fv.vsa_attn(qd, kd, vd, frames=grid[0], height=grid[1], width=grid[2], topk=topk))
    TV.check(q, k, v, grid, topk)


def _delta_case():
    from tests import test_gpu_delta as TD
    frames, t, c, w = 9, 40, 2, 1
    args = TD.make(frames, t, 2, 4242)
    return TD, args, (t, c, w)


@pytest.mark.parametrize("kernel,load_index", [
    (fv.TEST_VDA_STATS, 0),    # CTA 0's only 64-token stage (frame 1, head 0)
    (fv.TEST_VDA_SCAN, 3),     # the inverse M of the fourth step of the forward scan of head 0
    (fv.TEST_VDA_READOUT, 0),  # the first Q tile of CTA 0
], ids=["stats", "scan", "readout"])
def test_delta_wait_times_out_and_context_survives(kernel, load_index):
    TD, (q, k, v, beta, alpha, ts), (t, c, w) = _delta_case()
    dev = [x.cuda() for x in (q, k, v, beta, alpha, ts)]
    _expect_timeout(kernel, load_index,
                    lambda: fv.delta_attn(*dev[:5], frame_tokens=t, chunk_frames=c, window_chunks=w,
                                          text_state=dev[5]))
    ws, wo = TD.check(q, k, v, beta, alpha, ts, t, c, w)
    assert ws <= 1e-4 and wo <= 1e-2, (ws, wo)
