"""Pins for the VSA-style block-sparse attention oracle (oracle/vsa.py): the
printed top-k count, the tile geometry of the model's latent grid, the tile
means, a brute-force selection with ties, the dense oracle at zero sparsity,
a hand-built single-tile case, and invariances of the fine stage."""
import math

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from oracle import vsa as S

D = 128


def _bf16(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16)


def test_topk_count_follows_the_printed_formula():
    # max(1, min(ceil((1 - sparsity) * n), n)), evaluated by hand
    cases = [((1188, 0.9), 119), ((1188, 0.0), 1188), ((1188, 1.0), 1), ((10, 0.95), 1), ((7, 0.5), 4),
             ((3, -0.5), 3), ((64, 0.75), 16), ((1, 0.9), 1), ((594, 0.9), 60)]
    for (n, s), want in cases:
        assert S.topk_count(n, s) == want, (n, s)


def test_tile_grid_of_the_ten_second_clip():
    """72 latent frames of 24 x 42 tokens: 18 x 6 x 11 tiles; the last tile
    column is 2 tokens wide."""
    frames, height, width = 72, 24, 42
    assert S.tile_grid(frames, height, width) == (18, 6, 11)
    tiles = S.tile_tokens(frames, height, width)
    assert len(tiles) == 1188
    sizes = np.array([len(t) for t in tiles])
    assert (sizes == 64).sum() == 1080 and (sizes == 32).sum() == 108
    allidx = np.sort(np.concatenate(tiles))
    assert np.array_equal(allidx, np.arange(frames * height * width))
    assert list(tiles[0][:8]) == [0, 1, 2, 3, 42, 43, 44, 45]
    assert tiles[1][0] == 4 and tiles[11][0] == 4 * 42 and tiles[66][0] == 4 * 24 * 42
    # token (t=5, h=9, w=41) sits in tile (1, 2, 10)
    owner = S.token_tile(frames, height, width)
    assert owner[(5 * height + 9) * width + 41] == (1 * 6 + 2) * 11 + 10


def test_tile_means_are_over_the_tiles_own_tokens():
    frames, height, width = 5, 6, 7  # ragged in every direction
    tiles = S.tile_tokens(frames, height, width)
    x = np.zeros((frames * height * width, 3), dtype=np.float32)
    for b, idx in enumerate(tiles):
        x[idx] = [b, -2.0 * b, 0.5]
    m = S.pooled(x, tiles)
    assert np.array_equal(m, np.array([[b, -2.0 * b, 0.5] for b in range(len(tiles))], dtype=np.float32))
    y = np.random.default_rng(3).standard_normal((frames * height * width, 5)).astype(np.float32)
    mean = np.stack([[sum(float(y[i, c]) for i in idx) / len(idx) for c in range(5)] for idx in tiles])
    assert np.abs(S.pooled(y, tiles) - mean).max() < 1e-12


def test_selection_brute_force_with_ties():
    rng = np.random.default_rng(4)
    scores = rng.integers(-3, 4, size=(9, 11)).astype(np.float32)  # many ties
    for k in (1, 3, 11):
        sel = S.select(scores, k)
        for r in range(9):
            want = [c for c in range(11)
                    if sum(1 for o in range(11)
                           if scores[r, o] > scores[r, c] or (scores[r, o] == scores[r, c] and o < c)) < k]
            assert list(sel[r]) == want, (k, r)


def test_selection_takes_the_exact_scores():
    """The coarse scores are the plain dot products of the tile means: two key
    tiles whose scores differ by 3e-8 (below float32 resolution at 1.0, where
    they would tie and the lower index would win) are told apart."""
    qbar = np.array([[1.0, 1.0]])
    kbar = np.array([[1.0, 0.0], [1.0, 3e-8]])
    sc = S.coarse_scores(qbar, kbar)
    assert sc[0, 1] - sc[0, 0] == pytest.approx(3e-8, rel=1e-9)
    assert list(S.select(sc, 1)[0]) == [1]
    # means of the tiles' own rows feed the same decision
    frames, height, width = 4, 4, 8  # two tiles side by side
    tiles = S.tile_tokens(frames, height, width)
    x = np.zeros((frames * height * width, 2))
    for idx, row in zip(tiles, kbar):
        x[idx] = row
    kb = S.pooled(x, tiles)
    assert np.abs(kb - kbar).max() <= 1e-20
    assert list(S.select(S.coarse_scores(qbar, kb), 1)[0]) == [1]


def test_zero_sparsity_is_dense_attention():
    frames, height, width, heads = 5, 6, 7, 2
    n = frames * height * width
    q, k, v = (_bf16((n, heads * D), s) for s in (11, 12, 13))
    rows = np.arange(0, n, 7)
    ntiles = len(S.tile_tokens(frames, height, width))
    scale = 1.0 / math.sqrt(D)
    for h in range(heads):
        sl = slice(h * D, (h + 1) * D)
        got, sel = S.vsa_head(q[:, sl].double().numpy(), k[:, sl].double().numpy(), v[:, sl].double().numpy(),
                              rows, frames, height, width, S.topk_count(ntiles, 0.0), scale)
        want, want_lse = oracle.attn_rows(q, k, v, h, rows, scale)
        assert np.abs(got - want).max() < 1e-12
        tiles = S.tile_tokens(frames, height, width)
        lse = S.fine_lse(q[:, sl].double().numpy(), k[:, sl].double().numpy(), rows,
                         S.token_tile(frames, height, width), sel, tiles, scale)
        assert np.abs(lse - want_lse).max() < 1e-12
        assert np.array_equal(sel, np.tile(np.arange(ntiles), (ntiles, 1)))


def test_one_kept_tile_by_hand():
    """k = 1: each query sees only the tile whose key mean best matches its
    tile's query mean, worked with explicit loops."""
    frames, height, width = 4, 4, 8  # two tiles side by side
    n = frames * height * width
    d = 16
    rng = np.random.default_rng(5)
    q = rng.standard_normal((n, d))
    k = rng.standard_normal((n, d))
    v = rng.standard_normal((n, d))
    k[[(t * height + h) * width + w for t in range(4) for h in range(4) for w in range(4, 8)]] += 0.7
    members = [[(t * height + h) * width + w for t in range(4) for h in range(4) for w in range(4 * b, 4 * b + 4)]
               for b in range(2)]
    qm = [np.mean(q[m], axis=0) for m in members]
    km = [np.mean(k[m], axis=0) for m in members]
    rows = list(range(n))
    got, sel = S.vsa_head(q, k, v, rows, frames, height, width, 1, 0.25)
    for b in range(2):
        best = int(np.argmax([float(qm[b] @ km[c]) for c in range(2)]))
        assert sel[b, 0] == best
        for i in members[b]:
            p = scipy.special.softmax(0.25 * (k[members[best]] @ q[i]))
            assert np.abs(got[i] - p @ v[members[best]]).max() < 1e-12


def test_selection_follows_the_queries():
    """Tile 0's queries point along the key mean of tile 1 and tile 1's along
    that of tile 0, so each query tile keeps the other key tile."""
    frames, height, width, d = 4, 4, 8, 16
    n = frames * height * width
    rng = np.random.default_rng(8)
    e1, e2 = np.eye(d)[0], np.eye(d)[1]
    owner = S.token_tile(frames, height, width)
    q = np.where(owner[:, None] == 0, e2, e1) + 0.01 * rng.standard_normal((n, d))
    k = np.where(owner[:, None] == 0, 2.0 * e1, e2) + 0.01 * rng.standard_normal((n, d))
    v = rng.standard_normal((n, d))
    _, sel = S.vsa_head(q, k, v, [0], frames, height, width, 1, 0.1)
    assert sel[0, 0] == 1 and sel[1, 0] == 0


def test_values_of_dropped_tiles_do_not_matter():
    frames, height, width = 4, 8, 8  # four tiles
    n = frames * height * width
    rng = np.random.default_rng(6)
    q, k, v = (rng.standard_normal((n, 16)) for _ in range(3))
    rows = np.arange(n)
    out, sel = S.vsa_head(q, k, v, rows, frames, height, width, 2, 0.3)
    tiles = S.tile_tokens(frames, height, width)
    owner = S.token_tile(frames, height, width)
    for b in range(4):
        dropped = [c for c in range(4) if c not in sel[b]]
        v2 = v.copy()
        for c in dropped:
            v2[tiles[c]] = rng.standard_normal((len(tiles[c]), 16)) * 10
        out2, sel2 = S.vsa_head(q, k, v2, rows, frames, height, width, 2, 0.3)
        assert np.array_equal(sel, sel2)
        mine = owner == b
        assert np.abs(out2[mine] - out[mine]).max() < 1e-12
        v3 = v.copy()
        v3[tiles[sel[b, 0]]] += 1.0  # a kept tile's values shift every output of the tile by 1
        out3, _ = S.vsa_head(q, k, v3, rows, frames, height, width, 2, 0.3)
        assert np.abs(out3[mine] - out[mine]).min() > 1e-3


def test_token_order_inside_a_tile_does_not_matter():
    frames, height, width = 4, 4, 12
    n = frames * height * width
    rng = np.random.default_rng(7)
    q, k, v = (rng.standard_normal((n, 16)) for _ in range(3))
    rows = np.arange(n)
    out, sel = S.vsa_head(q, k, v, rows, frames, height, width, 2, 0.3)
    tiles = S.tile_tokens(frames, height, width)
    perm = np.arange(n)
    for idx in tiles:
        perm[idx] = rng.permutation(idx)
    out2, sel2 = S.vsa_head(q, k[perm], v[perm], rows, frames, height, width, 2, 0.3)
    assert np.array_equal(sel, sel2)
    assert np.abs(out2 - out).max() < 1e-12


# Plausible mistakes planted in copies of the oracle module; each must fail a pin.
MUTANTS = {
    "keeps_lowest": ("np.lexsort((index, -s), axis=-1)", "np.lexsort((index, s), axis=-1)"),
    "ties_to_higher_index": ("np.lexsort((index, -s), axis=-1)", "np.lexsort((-index, -s), axis=-1)"),
    "floor_count": ("int(math.ceil((1.0 - sparsity) * num_tiles))", "int(math.floor((1.0 - sparsity) * num_tiles))"),
    "no_minimum_of_one": ("max(1, min(int(", "max(0, min(int("),
    "grid_rounds_down": ("-(-width // TILE[2])", "(width // TILE[2])"),
    "height_width_swapped": ("(t * height + h) * width + w", "(t * width + w) * height + h"),
    "mean_over_full_tile": ("/ float(len(idx))", "/ 64.0"),
    "scale_dropped": ("s = scale * (k64[keys] @ q64[i])\n        e = np.exp", "s = (k64[keys] @ q64[i])\n        e = np.exp"),
    "scores_in_float32": ("return np.asarray(qbar, np.float64) @ np.asarray(kbar, np.float64).T",
                          "return (np.asarray(qbar, np.float32) @ np.asarray(kbar, np.float32).T)"
                          ".astype(np.float64)"),
    "queries_pooled_from_keys": ("select(coarse_scores(pooled(q, tiles), pooled(k, tiles)), topk)",
                                 "select(coarse_scores(pooled(k, tiles), pooled(k, tiles)), topk)"),
    "row_tile_off_by_one": ("for c in selected[row_tile[i]]])\n        s = scale * (k64[keys] @ q64[i])\n        e =",
                            "for c in selected[min(row_tile[i] + 1, len(selected) - 1)]])\n"
                            "        s = scale * (k64[keys] @ q64[i])\n        e ="),
}


def _mutant_module(name):
    import importlib.util
    import os
    import tempfile
    src = open(S.__file__).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, name
    d = tempfile.mkdtemp()
    path = os.path.join(d, f"vsa_{name}.py")
    open(path, "w").write(src.replace(old, new))
    spec = importlib.util.spec_from_file_location(f"vsa_{name}", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_vsa_mutant_is_caught(name, monkeypatch):
    import sys
    monkeypatch.setattr(sys.modules[__name__], "S", _mutant_module(name))
    checks = [test_topk_count_follows_the_printed_formula, test_tile_grid_of_the_ten_second_clip,
              test_tile_means_are_over_the_tiles_own_tokens, test_selection_brute_force_with_ties,
              test_selection_takes_the_exact_scores,
              test_zero_sparsity_is_dense_attention, test_one_kept_tile_by_hand, test_selection_follows_the_queries,
              test_values_of_dropped_tiles_do_not_matter, test_token_order_inside_a_tile_does_not_matter]
    failed = 0
    for fn in checks:
        try:
            fn()
        except (AssertionError, IndexError, ValueError):
            failed += 1
    assert failed >= 1, f"mutant {name} passed every pin"
