"""GPU parity of Video Delta Attention (the VDN linear branch) against the
fp64 oracle (oracle/delta.py), through the C ABI."""
import numpy as np
import pytest
import torch

import video_diffusion_transformer_gb300 as fv
from oracle import delta as VD

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_ok):
    from video_diffusion_transformer_gb300 import build
    build.build()
    fv.load_library()


def make(frames, t, heads, seed, beta_scale=1.0, alpha_lo=0.5, text=True):
    g = torch.Generator().manual_seed(seed)
    n = frames * t
    q, k, v = [torch.randn((n, heads * 128), generator=g).to(torch.bfloat16) for _ in range(3)]
    beta = torch.sigmoid(torch.randn((heads, n), generator=g)) * beta_scale
    alpha = alpha_lo + (1.0 - alpha_lo) * torch.rand((heads, frames, 128), generator=g)
    ts = torch.randn((heads, 128, 128), generator=g) * 0.1 if text else None
    return q, k, v, beta.float(), alpha.float(), ts


def run(q, k, v, beta, alpha, ts, t, c, w):
    o, states = fv.delta_attn(q.cuda(), k.cuda(), v.cuda(), beta.cuda(), alpha.cuda(), frame_tokens=t,
                              chunk_frames=c, window_chunks=w, text_state=None if ts is None else ts.cuda())
    fv.sync_status()
    return o.cpu(), states.cpu().double().numpy()


def check(q, k, v, beta, alpha, ts, t, c, w, rows=None, frames_checked=None):
    n, heads = q.shape[0], q.shape[1] // 128
    o, states = run(q, k, v, beta, alpha, ts, t, c, w)
    rows = np.arange(n) if rows is None else rows
    worst_s, worst_o = 0.0, 0.0
    for h in range(heads):
        sl = slice(h * 128, (h + 1) * 128)
        ref_o, fwd, rev = VD.delta_attn_head(q[:, sl].double().numpy(), k[:, sl].double().numpy(),
                                             v[:, sl].double().numpy(), beta[h].double().numpy(),
                                             alpha[h].double().numpy(),
                                             None if ts is None else ts[h].double().numpy(), rows, t, c, w)
        fr = range(fwd.shape[0]) if frames_checked is None else frames_checked
        for f in fr:
            for got, ref in ((states[0, h, f], fwd[f]), (states[1, h, f], rev[f])):
                worst_s = max(worst_s, float(np.abs(got - ref).max() / max(1e-6, np.abs(ref).max())))
        got_o = o[rows, sl].double().numpy()
        scale = np.maximum(np.abs(ref_o), 1.0)
        worst_o = max(worst_o, float((np.abs(got_o - ref_o) / scale).max()))
    return worst_s, worst_o


@pytest.mark.parametrize("frames,t,c,w", [(9, 40, 2, 1), (12, 64, 3, 1), (7, 33, 1, 0), (16, 128, 5, 1)])
def test_small_geometries(frames, t, c, w):
    ws, wo = check(*make(frames, t, 2, frames * 31 + t), t, c, w)
    assert ws <= 1e-4, ws
    assert wo <= 1e-2, wo


def test_no_text_state_and_short_clips():
    for frames in (1, 2, 3):
        q, k, v, beta, alpha, _ = make(frames, 50, 1, frames, text=False)
        ws, wo = check(q, k, v, beta, alpha, None, 50, 2, 1)
        assert ws <= 1e-4 and wo <= 1e-2


def test_aligned_keys_make_ill_conditioned_frames():
    """Every key of a frame close to one direction and beta = 1: I + A_t has
    one eigenvalue near the frame's token count (256) and the rest near 1,
    so the per-frame inverse is ill-conditioned (~257) and its pivots span
    that range.  States and readout stay within the same bounds as the
    well-conditioned cases."""
    frames, t, heads = 8, 256, 2
    q, k, v, beta, alpha, ts = make(frames, t, heads, 901)
    g = torch.Generator().manual_seed(902)
    for h in range(heads):
        u = torch.randn(128, generator=g)
        noise = 0.05 * torch.randn((frames * t, 128), generator=g)
        k[:, h * 128:(h + 1) * 128] = (u[None, :] + noise).to(torch.bfloat16)
    beta = torch.ones_like(beta)
    ws, wo = check(q, k, v, beta, alpha, ts, t, 2, 1)
    print(f"aligned keys: worst state error {ws:.3g}, worst output error {wo:.3g}")
    assert ws <= 1e-3, ws
    assert wo <= 1e-2, wo


def test_no_writes_is_pure_decay():
    frames, t = 10, 32
    q, k, v, beta, alpha, ts = make(frames, t, 2, 7)
    beta.zero_()
    alpha.fill_(0.5)
    _, states = run(q, k, v, beta, alpha, ts, t, 2, 1)
    for f in range(frames - 1):
        ref = 0.5 * ts.double().numpy() * 0.5 ** f
        assert np.abs(states[0, :, f] - ref).max() <= 1e-6 * max(1.0, np.abs(ref).max())


def test_model_geometry_72_frames():
    """72 latent frames of 1,008 tokens (the 10 s clip), 4 heads; sampled rows."""
    frames, t = 72, 1008
    q, k, v, beta, alpha, ts = make(frames, t, 4, 123, alpha_lo=0.9)
    rng = np.random.default_rng(5)
    rows = np.unique(np.concatenate([[0, t - 1, t, 5 * t, 35 * t + 17, frames * t - 1],
                                     rng.integers(0, frames * t, 60)]))
    ws, wo = check(q, k, v, beta, alpha, ts, t, 5, 1, rows=rows, frames_checked=[0, 1, 2, 30, 70, 71])
    print("delta 72 frames: states rel", ws, "readout rel", wo)
    assert ws <= 1e-3, ws
    assert wo <= 2e-2, wo
