"""Failure detection on the GPU without a fault: a bounded wait inside the
attention kernel is made to run out (a K/V load that is never issued, set by
the FV_TEST_SKIP_KV_LOAD test hook), and the call must report
FV_ERR_DEVICE_TIMEOUT through the status word, drain its in-flight copies and
MMAs, release tensor memory, and leave the context usable."""
import math
import os
import time

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


def test_bounded_wait_times_out_reports_status_and_context_survives():
    q, k, v = _inputs()
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    fv.sync_status()
    os.environ["FV_TEST_SKIP_KV_LOAD"] = "5"
    try:
        t0 = time.time()
        fv.attn_fwd(qd, kd, vd, head_group=2)
        with pytest.raises(fv.FvError) as e:
            fv.sync_status()
        elapsed = time.time() - t0
    finally:
        del os.environ["FV_TEST_SKIP_KV_LOAD"]
    assert e.value.code == -7, e.value
    assert elapsed < 30.0
    # the status word was cleared by the read, and the context still computes
    fv.sync_status()
    lse = torch.empty((2, q.shape[0]), dtype=torch.float32, device="cuda")
    o = fv.attn_fwd(qd, kd, vd, head_group=2, lse=lse)
    fv.sync_status()
    P.assert_attention_ok(P.attention_errors(q, k, v, o, 2, 64, SCALE, lse))
