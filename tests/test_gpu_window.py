"""GPU parity of the windowed attention (the Video DeltaNet softmax branch)
against the fp64 oracle, through the C ABI."""
import math

import numpy as np
import pytest
import torch

import oracle
import video_diffusion_transformer_gb300 as fv
import workloads as W
from tests import parity as P

pytestmark = pytest.mark.gpu
SCALE = 1.0 / math.sqrt(128)


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_ok):
    from video_diffusion_transformer_gb300 import build
    build.build()
    fv.load_library()


def rand(n, heads, seed):
    g = torch.Generator().manual_seed(seed)
    return [torch.randn((n, heads * 128), generator=g).to(torch.bfloat16) for _ in range(3)]


def check(q, k, v, heads, hg, t, c, w, rows_per_head=0, rows=None):
    n = q.shape[0]
    lse = torch.full((heads, n), float("nan"), dtype=torch.float32, device="cuda")
    o = fv.attn_fwd_window(q.cuda(), k.cuda(), v.cuda(), frame_tokens=t, chunk_frames=c, window_chunks=w,
                           head_group=hg, lse=lse)
    fv.sync_status()
    o_cpu, lse_cpu = o.cpu(), lse.cpu().numpy()
    worst, tot, cnt, se, sref, lw = 0.0, 0.0, 0, 0.0, 0.0, 0.0
    for h in range(heads):
        r = rows if rows is not None else W.sampled_rows(n, h, rows_per_head).numpy()
        o_ref, l_ref = oracle.attn_rows_window(q, k, v, h, r, SCALE, t, c, w)
        got = o_cpu[r, h * 128:(h + 1) * 128].double().numpy()
        d = np.abs(got - o_ref)
        worst, tot, cnt = max(worst, float(d.max())), tot + float(d.sum()), cnt + d.size
        se, sref = se + float((d * d).sum()), sref + float((o_ref * o_ref).sum())
        lw = max(lw, float(np.abs(lse_cpu[h, r] - l_ref).max()))
    err = {"max_abs": worst, "mean_abs": tot / cnt, "rel_rms": math.sqrt(se / sref), "lse_max_abs": lw}
    P.assert_attention_ok(err)
    return o, err


@pytest.mark.parametrize("frames,t,c,w", [(6, 64, 2, 1), (9, 100, 3, 1), (12, 300, 5, 1), (20, 128, 5, 1),
                                          (11, 96, 2, 0), (13, 77, 2, 2), (3, 1008, 5, 1)])
def test_small_geometries_all_rows(frames, t, c, w):
    n, heads = frames * t, 2
    q, k, v = rand(n, heads, frames * 1000 + t)
    for hg in (1, 2):
        check(q, k, v, heads, hg, t, c, w)


def test_window_wider_than_clip_is_dense_attention():
    n, heads, t = 12 * 100, 3, 100
    q, k, v = rand(n, heads, 5)
    o_win = fv.attn_fwd_window(q.cuda(), k.cuda(), v.cuda(), frame_tokens=t, chunk_frames=2, window_chunks=6,
                               head_group=3)
    o_den = fv.attn_fwd(q.cuda(), k.cuda(), v.cuda(), head_group=3)
    fv.sync_status()
    assert torch.equal(o_win, o_den)


def test_model_geometry_72_frames():
    """10 s clip at 1344x768: 72 latent frames of 1,008 tokens, 56 heads in
    groups of 16; rows in the anchor frames, at chunk edges and at random."""
    w_ = W.WORKLOADS["clip10s_72576"]
    q, k, v = W.qkv(w_)
    t = 1008
    edges = []
    for chunk in range(1, 72 // 5 + 1):
        b = chunk * 5 * t
        edges += [b - 1, b, b + 1]
    rows = np.unique(np.concatenate([[0, 1, t - 1, t, 2 * t + 5, 71 * t - 1, 71 * t, 72 * t - 1], edges,
                                     np.random.default_rng(0).integers(0, 72 * t, 40)]))
    rows = rows[rows < 72 * t]
    _, err = check(q, k, v, 56, 16, t, 5, 1, rows=rows)
    print("72-frame window", err)


def test_window_pairs_accounting():
    # the FLOP accounting's pair count agrees with the oracle's window
    n, t = 9 * 7, 7
    ref = sum(oracle.window_allowed(i, j, n, t, 2, 1) for i in range(n) for j in range(n))
    assert W.window_pairs(n, t, 2, 1) == ref
