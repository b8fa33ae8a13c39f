"""Oracle of VSA-style block-sparse attention over a video latent grid.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Plain numpy, float64
throughout: the tile means, the coarse scores that decide the kept tiles, and
the attention over them.

What it computes, per head, following "FastH3 Preview v1: four calls,
one-tenth the attention, and what the 14x actually measures", section
"Lever two: VSA-H3 makes each of the four calls cheaper":

* the video tokens, laid out as a (frames, height, width) latent grid in
  raster order, are cut into 3D tiles of (4, 4, 4) = 64 tokens (the shape the
  distilled model is trained on); tiles are numbered in raster order over the
  tile grid, and tiles on the far edges hold fewer tokens where a grid side is
  not a multiple of 4;
* a coarse stage scores every (query tile, key tile) pair cheaply: the mean of
  the tile's queries against the mean of the tile's keys;
* each query tile keeps the top-k key tiles, with the page's count
      k = max(1, min(ceil((1 - sparsity) * num_tiles), num_tiles));
* fine stage: every query of the tile attends exactly (softmax over
  scale * q.k) to the keys of its kept tiles, and to nothing else.

Readings where the page leaves the step open:
* pooling is the plain mean over the tile's real tokens (an edge tile's mean
  is over its own, fewer, tokens); the coarse score is the dot product of the
  two means (the softmax scale and a row softmax do not change the ranking);
* ties in the coarse score go to the lower tile index;
* the page gives no precision for the coarse stage, so the oracle takes the
  plain definition (means and dot products) in float64; a GPU path that
  scores in float32 may keep a different tile only where two scores lie
  within float32 rounding of each other;
* the compression branch is left out: its gate is a trained projection that
  the base weights initialise to zero, so untrained it adds nothing;
* only video tokens are present, so there are no exempt (always kept) keys
  and no dense (non-video) queries.
"""
from __future__ import annotations

import math

import numpy as np

TILE = (4, 4, 4)  # (t, h, w) tokens per tile


def topk_count(num_tiles: int, sparsity: float) -> int:
    """Key tiles kept per query tile: max(1, min(ceil((1 - sparsity) n), n))."""
    return max(1, min(int(math.ceil((1.0 - sparsity) * num_tiles)), num_tiles))


def tile_grid(frames: int, height: int, width: int) -> tuple[int, int, int]:
    """Tiles along (t, h, w): each side divided by 4, rounded up."""
    return (-(-frames // TILE[0]), -(-height // TILE[1]), -(-width // TILE[2]))


def tile_tokens(frames: int, height: int, width: int) -> list[np.ndarray]:
    """Token indices of every tile, tiles in raster order over the tile grid,
    tokens of a tile in raster (t, h, w) order."""
    nt, nh, nw = tile_grid(frames, height, width)
    out = []
    for bt in range(nt):
        for bh in range(nh):
            for bw in range(nw):
                ts = range(bt * TILE[0], min(frames, (bt + 1) * TILE[0]))
                hs = range(bh * TILE[1], min(height, (bh + 1) * TILE[1]))
                ws = range(bw * TILE[2], min(width, (bw + 1) * TILE[2]))
                out.append(np.array([(t * height + h) * width + w for t in ts for h in hs for w in ws],
                                    dtype=np.int64))
    return out


def pooled(x: np.ndarray, tiles: list[np.ndarray]) -> np.ndarray:
    """float64 mean of each tile's rows of x ([N, d] -> [num_tiles, d])."""
    x64 = np.asarray(x, dtype=np.float64)
    return np.stack([x64[idx].sum(axis=0) / float(len(idx)) for idx in tiles])


def coarse_scores(qbar: np.ndarray, kbar: np.ndarray) -> np.ndarray:
    """float64 scores of every (query tile, key tile) pair."""
    return np.asarray(qbar, np.float64) @ np.asarray(kbar, np.float64).T


def select(scores: np.ndarray, k: int) -> np.ndarray:
    """The k highest-scoring key tiles of each query tile, ties to the lower
    index; each row returned in ascending tile order ([num_tiles, k])."""
    s = np.asarray(scores, dtype=np.float64)
    index = np.broadcast_to(np.arange(s.shape[1]), s.shape)
    order = np.lexsort((index, -s), axis=-1)  # by descending score, then ascending index
    return np.sort(order[:, :k], axis=-1).astype(np.int64)


def fine_rows(q, k, v, rows, row_tile, selected, tiles, scale: float) -> np.ndarray:
    """float64 attention of each query row over the keys of its tile's kept tiles."""
    q64, k64, v64 = (np.asarray(a, dtype=np.float64) for a in (q, k, v))
    out = np.empty((len(rows), q64.shape[1]))
    for r, i in enumerate(rows):
        keys = np.concatenate([tiles[c] for c in selected[row_tile[i]]])
        s = scale * (k64[keys] @ q64[i])
        e = np.exp(s - s.max())
        out[r] = (e @ v64[keys]) / e.sum()
    return out


def fine_lse(q, k, rows, row_tile, selected, tiles, scale: float) -> np.ndarray:
    """float64 log-sum-exp of each query row's scores over its kept keys."""
    q64, k64 = np.asarray(q, dtype=np.float64), np.asarray(k, dtype=np.float64)
    out = np.empty(len(rows))
    for r, i in enumerate(rows):
        keys = np.concatenate([tiles[c] for c in selected[row_tile[i]]])
        s = scale * (k64[keys] @ q64[i])
        m = s.max()
        out[r] = m + np.log(np.exp(s - m).sum())
    return out


def token_tile(frames: int, height: int, width: int) -> np.ndarray:
    """Tile index of every token ([N])."""
    tiles = tile_tokens(frames, height, width)
    owner = np.empty(frames * height * width, dtype=np.int64)
    for b, idx in enumerate(tiles):
        owner[idx] = b
    return owner


def vsa_head(q, k, v, rows, frames: int, height: int, width: int, topk: int, scale: float):
    """One head: (outputs of ``rows`` [len(rows), d] float64, selection [num_tiles, topk]).

    q, k, v: [N, d] arrays holding the (bf16-exact) inputs of one head."""
    tiles = tile_tokens(frames, height, width)
    sel = select(coarse_scores(pooled(q, tiles), pooled(k, tiles)), topk)
    owner = token_tile(frames, height, width)
    return fine_rows(q, k, v, rows, owner, sel, tiles, scale), sel
