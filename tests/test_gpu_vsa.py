"""GPU parity of VSA-style block-sparse attention against the oracle
(oracle/vsa.py), through the C ABI: the kept tiles (exact, up to coarse
scores that tie within float32 rounding, the precision the kernel scores in)
and the attention output and LSE of every checked query.  Where the kernel
kept a different but valid set of tiles (a tie), the oracle's fine stage runs
on the kernel's set, so no row goes unchecked."""
import math

import numpy as np
import pytest
import torch

import oracle
import video_diffusion_transformer_gb300 as fv
from oracle import vsa as VS
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


def run(q, k, v, grid, topk):
    heads = q.shape[1] // 128
    n = q.shape[0]
    lse = torch.full((heads, n), float("nan"), dtype=torch.float32, device="cuda")
    o, sel = fv.vsa_attn(q.cuda(), k.cuda(), v.cuda(), frames=grid[0], height=grid[1], width=grid[2], topk=topk,
                         lse=lse)
    fv.sync_status()
    return o.cpu(), sel.cpu().numpy(), lse.cpu().numpy()


def compare_selection(sel_gpu, q, k, h, grid, topk):
    """Oracle selection of head h (float64 scores); the tiles whose kept set
    differs from the GPU's must differ only by scores tied within float32
    rounding, and the GPU's set must hold topk distinct, ascending tiles."""
    tiles = VS.tile_tokens(*grid)
    sl = slice(h * 128, (h + 1) * 128)
    scores = VS.coarse_scores(VS.pooled(q[:, sl].float().numpy(), tiles), VS.pooled(k[:, sl].float().numpy(), tiles))
    sel_ref = VS.select(scores, topk)
    same = np.all(sel_gpu == sel_ref, axis=1)
    for b in np.nonzero(~same)[0]:
        a, r = set(sel_gpu[b].tolist()), set(sel_ref[b].tolist())
        assert len(a) == topk and np.all(np.diff(sel_gpu[b]) > 0), (b, sel_gpu[b])
        assert sel_gpu[b].min() >= 0 and sel_gpu[b].max() < len(tiles), (b, sel_gpu[b])
        kth = float(np.sort(scores[b])[::-1][topk - 1])
        tol = 1e-5 * max(1e-3, float(np.abs(scores[b]).max()))
        for c in a ^ r:
            assert abs(float(scores[b, c]) - kth) <= tol, (h, b, c)
    return sel_ref, same, tiles


def check(q, k, v, grid, topk, rows=None, max_mismatch=0.01):
    heads = q.shape[1] // 128
    n = q.shape[0]
    o, sel, lse = run(q, k, v, grid, topk)
    owner = VS.token_tile(*grid)
    worst, tot, cnt, se, sref, lw = 0.0, 0.0, 0, 0.0, 0.0, 0.0
    for h in range(heads):
        sel_ref, same, tiles = compare_selection(sel[h], q, k, h, grid, topk)
        assert (~same).mean() <= max_mismatch, (~same).sum()
        r = np.arange(n) if rows is None else np.asarray(rows)
        # A query tile whose kept set differs from the oracle's (a validated
        # tie) is checked against the oracle's fine stage over the GPU's set.
        sel_use = np.where(same[:, None], sel_ref, sel[h])
        sl = slice(h * 128, (h + 1) * 128)
        qh, kh, vh = (t[:, sl].double().numpy() for t in (q, k, v))
        o_ref = VS.fine_rows(qh, kh, vh, r, owner, sel_use, tiles, SCALE)
        l_ref = VS.fine_lse(qh, kh, r, owner, sel_use, tiles, SCALE)
        got = o[r, sl].double().numpy()
        d = np.abs(got - o_ref)
        worst, tot, cnt = max(worst, float(d.max())), tot + float(d.sum()), cnt + d.size
        se, sref = se + float((d * d).sum()), sref + float((o_ref * o_ref).sum())
        lw = max(lw, float(np.abs(lse[h, r] - l_ref).max()))
    err = {"max_abs": worst, "mean_abs": tot / cnt, "rel_rms": math.sqrt(se / sref), "lse_max_abs": lw}
    P.assert_attention_ok(err)
    return o, sel, err


@pytest.mark.parametrize("grid,heads,topk", [
    ((8, 8, 12), 2, 3),      # 2 x 2 x 3 tiles, no ragged edge
    ((5, 6, 7), 2, 2),       # ragged in every direction
    ((4, 4, 12), 1, 1),      # three tiles: an odd count leaves a lone tile in the last pair
    ((4, 4, 12), 2, 2),
    ((8, 12, 10), 3, 5),     # 2 x 3 x 3 tiles
    ((12, 8, 9), 2, 18),     # every tile kept
])
def test_small_grids(grid, heads, topk):
    n = grid[0] * grid[1] * grid[2]
    q, k, v = rand(n, heads, sum(grid) * 7 + topk)
    check(q, k, v, grid, topk)


def test_all_tiles_kept_is_dense_attention():
    grid, heads = (8, 10, 9), 2
    n = grid[0] * grid[1] * grid[2]
    q, k, v = rand(n, heads, 3)
    nt = fv.vsa_num_tiles(*grid)
    o, sel, _ = check(q, k, v, grid, nt)
    assert np.array_equal(sel, np.broadcast_to(np.arange(nt), sel.shape))
    err = P.attention_errors(q, k, v, o.cuda(), heads, 0, SCALE)
    P.assert_attention_ok(err)


def test_deterministic():
    grid, heads = (8, 8, 8), 2
    q, k, v = rand(512, heads, 9)
    a = run(q, k, v, grid, 3)
    b = run(q, k, v, grid, 3)
    assert torch.equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_ten_second_clip_grid():
    """72 x 24 x 42 latent grid (72,576 tokens), 2 heads, 90% sparsity (119 of
    1,188 tiles kept); sampled rows, including the 2-wide edge tiles."""
    grid, heads = (72, 24, 42), 2
    n = grid[0] * grid[1] * grid[2]
    q, k, v = rand(n, heads, 72)
    topk = fv.vsa_topk(fv.vsa_num_tiles(*grid), 0.9)
    assert topk == 119
    rng = np.random.default_rng(1)
    edge = [(t * 24 + h) * 42 + w for t in (0, 35, 71) for h in (0, 23) for w in (40, 41)]
    rows = np.unique(np.concatenate([[0, 1, 41, n - 1], edge, rng.integers(0, n, 300)]))
    _, _, err = check(q, k, v, grid, topk, rows=rows)
    print("vsa 72x24x42:", err)


@pytest.mark.parametrize("hot_tile", [1, 5, 10])
@pytest.mark.parametrize("gain", [6, 16])
def test_large_scores_late_in_the_list(hot_tile, gain):
    """Keys of one tile scaled up: with every tile kept, its scores exceed the
    running maximum when it is reached, in the second half of the first K/V
    tile (tile 1) or later (tiles 5, 10).  Gain 6 leaves most late halves
    within the kernel's 2^20 bound against the first maximum (summed as they
    are); gain 16 takes them past it, so the kernel must rescale the
    probabilities and the output it already holds."""
    grid, heads = (8, 8, 12), 2
    n = grid[0] * grid[1] * grid[2]
    q, k, v = rand(n, heads, 40 + hot_tile)
    idx = VS.tile_tokens(*grid)[hot_tile]
    k[idx] = (k[idx].float() * gain).to(torch.bfloat16)
    check(q, k, v, grid, fv.vsa_num_tiles(*grid))


def test_fourteen_second_clip_grid_one_head():
    """102 x 24 x 42 latent grid (the 14.4 s clip, 1,716 tiles), one head,
    90% sparsity (172 kept); sampled rows."""
    grid, heads = (102, 24, 42), 1
    n = grid[0] * grid[1] * grid[2]
    q, k, v = rand(n, heads, 102)
    nt = fv.vsa_num_tiles(*grid)
    topk = fv.vsa_topk(nt, 0.9)
    assert (nt, topk) == (1716, 172)
    rng = np.random.default_rng(2)
    rows = np.unique(np.concatenate([[0, n - 1], rng.integers(0, n, 200)]))
    check(q, k, v, grid, topk, rows=rows)


def test_outlier_key_channels():
    """1% of the key channels scaled by 20 (as in the half-resolution
    workload): the coarse scores and the softmax both see the outliers."""
    grid, heads = (8, 12, 16), 2
    n = grid[0] * grid[1] * grid[2]
    q, k, v = rand(n, heads, 21)
    cols = torch.randperm(heads * 128, generator=torch.Generator().manual_seed(2))[: max(1, heads * 128 // 100)]
    k[:, cols] = (k[:, cols].float() * 20).to(torch.bfloat16)
    check(q, k, v, grid, fv.vsa_topk(fv.vsa_num_tiles(*grid), 0.75))
