"""fp64 oracle of the Video DeltaNet linear branch (Video Delta Attention).

TEST INFRASTRUCTURE ONLY (see the package docstring).  Plain numpy in
double precision; np.linalg.solve is the one library step.

What it computes, per head, following "FreeVideo: a 66 GB video transformer on
an 8 GB card", section "Where Video DeltaNet comes in":

* q and k of every token are L2-normalised (the branch's "L2 normalization on
  Q and K");
* frame t (T tokens u, write strengths beta_u) has
      A_t = sum_u beta_u k_u k_u^T,   B_t = sum_u beta_u v_u k_u^T;
* the state after writing frame t is the solution of the frame's joint
  least-squares problem, written in closed form on the page:
      S_t = (Sbar_t + B_t) (I + A_t)^{-1},   Sbar_t = S_{t-1} Diag(alpha_t);
* two scans, forward and reverse, each seeded with S_T / 2 (the text state),
  so the two readouts together count it once.

Readings where the page leaves the step open:
* the scans cover the frames the softmax branch does not treat as global
  anchors: forward over frames 1 .. F-2 and reverse over F-2 .. 1 (the first
  and last latent frames are softmax anchors);
* a token of frame t in chunk c = t // C reads the forward state of the last
  frame before its softmax window, p = (c - W) C - 1, and the reverse state of
  the first frame after it, n = (c + W + 1) C:
      o = (Sf + Sr) q,  Sf = state_fwd[max(p, 0)],  Sr = state_rev[min(n, F-1)],
  where state_fwd[0] = state_rev[F-1] = S_T / 2 (nothing written yet);
* the same alpha_t decays the carried state in both directions.
"""
from __future__ import annotations

import numpy as np


def l2_normalize(x: np.ndarray) -> np.ndarray:
    n = np.linalg.norm(x, axis=-1, keepdims=True)
    return x / np.maximum(n, 1e-12)


def frame_stats(k_hat: np.ndarray, v: np.ndarray, beta: np.ndarray):
    """A = sum_u beta_u k_u k_u^T and B = sum_u beta_u v_u k_u^T for one frame."""
    a = (k_hat * beta[:, None]).T @ k_hat
    b = (v * beta[:, None]).T @ k_hat
    return a, b


def update(s_prev: np.ndarray, alpha: np.ndarray, a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """S = (S_prev Diag(alpha) + B) (I + A)^{-1}, solved as (I + A) S^T = (.)^T
    ((I + A) is symmetric)."""
    rhs = s_prev * alpha[None, :] + b
    return np.linalg.solve(np.eye(a.shape[0]) + a, rhs.T).T


def delta_states(q, k, v, beta, alpha, text_state, frame_tokens: int):
    """Per-frame forward and reverse states of one head.

    q, k, v: float64 [N, d]; beta: [N]; alpha: [F, d]; text_state: [d, d] or None.
    Returns (state_fwd [F, d, d], state_rev [F, d, d]).
    """
    n, d = k.shape
    frames = n // frame_tokens
    k_hat = l2_normalize(k)
    seed = np.zeros((d, d)) if text_state is None else 0.5 * np.asarray(text_state, dtype=np.float64)
    fwd = np.empty((frames, d, d))
    rev = np.empty((frames, d, d))
    stats = []
    for t in range(frames):
        sl = slice(t * frame_tokens, (t + 1) * frame_tokens)
        stats.append(frame_stats(k_hat[sl], v[sl], beta[sl]))
    fwd[0] = seed
    for t in range(1, frames):
        fwd[t] = update(fwd[t - 1], alpha[t], *stats[t]) if t <= frames - 2 else fwd[t - 1]
    rev[frames - 1] = seed
    for t in range(frames - 2, -1, -1):
        rev[t] = update(rev[t + 1], alpha[t], *stats[t]) if t >= 1 else rev[t + 1]
    return fwd, rev


def delta_readout(q, fwd, rev, rows, frame_tokens: int, chunk_frames: int, window_chunks: int):
    """o = (state_fwd[p] + state_rev[n]) q_hat for the given token rows."""
    frames = fwd.shape[0]
    q_hat = l2_normalize(q[rows])
    out = np.empty((len(rows), q.shape[1]))
    for r, i in enumerate(rows):
        c = (i // frame_tokens) // chunk_frames
        p = max((c - window_chunks) * chunk_frames - 1, 0)
        nx = min((c + window_chunks + 1) * chunk_frames, frames - 1)
        out[r] = (fwd[p] + rev[nx]) @ q_hat[r]
    return out


def delta_attn_head(q, k, v, beta, alpha, text_state, rows, frame_tokens: int, chunk_frames: int = 5,
                    window_chunks: int = 1):
    """Readout rows and both state sequences of one head (all float64)."""
    fwd, rev = delta_states(q, k, v, beta, alpha, text_state, frame_tokens)
    return delta_readout(q, fwd, rev, rows, frame_tokens, chunk_frames, window_chunks), fwd, rev
