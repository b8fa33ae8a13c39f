"""Checks that pin the oracle to the mathematics rather than to itself.

Every function takes an oracle object (``oracle.default()`` or a deliberately
broken copy) and either returns an error measure or raises AssertionError.
None of them retypes the oracle's formula: they use brute force through
library routines (numpy/scipy/torch float64), closed forms, and invariants of
softmax attention, LayerNorm and rounding.
"""
from __future__ import annotations

import math

import numpy as np
import scipy.special
import torch

D = 128


def _bf16(a) -> torch.Tensor:
    """Exact float64 values (already bf16-representable) -> bf16 tensor."""
    t = torch.as_tensor(np.asarray(a, dtype=np.float64))
    b = t.to(torch.bfloat16)
    assert torch.equal(b.to(torch.float64), t), "test value not representable in bfloat16"
    return b


def _rand_bf16(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g, dtype=torch.float32) * scale).to(torch.bfloat16)


def _head(t: torch.Tensor, h: int) -> np.ndarray:
    return t[:, h * D:(h + 1) * D].to(torch.float64).numpy()


def _rel(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.max(np.abs(a - b)) / max(1e-300, float(np.max(np.abs(b)))))


# ----------------------------------------------------------------- attention
def attn_brute_force(orc, n: int, heads: int, seed: int) -> float:
    """Materialise the whole score matrix, softmax it with scipy, multiply by V."""
    q = _rand_bf16((n, heads * D), seed)
    k = _rand_bf16((n, heads * D), seed + 100)
    v = _rand_bf16((n, heads * D), seed + 200)
    scale = 1.0 / math.sqrt(D)
    worst = 0.0
    for h in range(heads):
        s = scale * (_head(q, h) @ _head(k, h).T)
        p = scipy.special.softmax(s, axis=1)
        o_ref = p @ _head(v, h)
        lse_ref = scipy.special.logsumexp(s, axis=1)
        o, lse = orc.attn_rows(q, k, v, h, np.arange(n), scale)
        worst = max(worst, _rel(o, o_ref), _rel(lse, lse_ref) if n > 1 else abs(lse[0] - lse_ref[0]))
    return worst


def attn_vs_sdpa(orc, n: int, heads: int, seed: int) -> float:
    """torch's float64 scaled_dot_product_attention on the CPU, all rows."""
    q = _rand_bf16((n, heads * D), seed)
    k = _rand_bf16((n, heads * D), seed + 1)
    v = _rand_bf16((n, heads * D), seed + 2)
    scale = 1.0 / math.sqrt(D)

    def bhnd(t):
        return t.to(torch.float64).view(n, heads, D).permute(1, 0, 2).unsqueeze(0)

    ref = torch.nn.functional.scaled_dot_product_attention(bhnd(q), bhnd(k), bhnd(v), scale=scale)[0]
    worst = 0.0
    for h in range(heads):
        o, _ = orc.attn_rows(q, k, v, h, np.arange(n), scale)
        worst = max(worst, _rel(o, ref[h].numpy()))
    return worst


def attn_closed_forms(orc) -> None:
    scale = 1.0 / math.sqrt(D)
    # N = 1: the only key gets weight 1, so O = V and lse = the single score.
    q = _rand_bf16((1, 2 * D), 1)
    k = _rand_bf16((1, 2 * D), 2)
    v = _rand_bf16((1, 2 * D), 3)
    for h in range(2):
        o, lse = orc.attn_rows(q, k, v, h, [0], scale)
        assert np.array_equal(o[0], _head(v, h)[0]), "N=1 must return V"
        s = scale * float(np.dot(_head(q, h)[0], _head(k, h)[0]))
        assert abs(lse[0] - s) <= 1e-12 * max(1.0, abs(s)), "N=1 lse must equal the score"

    # Q = 0 (or scale = 0): uniform weights, O = mean of V, lse = log N.
    n = 300
    k = _rand_bf16((n, D), 4)
    v = _rand_bf16((n, D), 5)
    zero = torch.zeros((n, D), dtype=torch.bfloat16)
    rows = [0, 7, 299]
    mean_v = _head(v, 0).mean(axis=0)
    o, lse = orc.attn_rows(zero, k, v, 0, rows, scale)
    assert _rel(o, np.tile(mean_v, (3, 1))) < 1e-12
    assert np.max(np.abs(lse - math.log(n))) < 1e-12
    qr = _rand_bf16((n, D), 6)
    o, lse = orc.attn_rows(qr, k, v, 0, rows, 0.0)
    assert _rel(o, np.tile(mean_v, (3, 1))) < 1e-12
    assert np.max(np.abs(lse - math.log(n))) < 1e-12

    # V constant over keys: every convex combination returns that vector.
    c = _rand_bf16((1, D), 7)
    vc = c.repeat(n, 1)
    o, _ = orc.attn_rows(qr, k, vc, 0, rows, scale)
    assert _rel(o, np.tile(_head(c, 0), (3, 1))) < 1e-14

    # Two keys on one axis: weights are a logistic function of the score gap.
    a, b0, b1, sc = 1.5, 2.0, -1.0, 0.75
    qv = np.zeros((1, D)); qv[0, 3] = a
    kv = np.zeros((2, D)); kv[0, 3] = b0; kv[1, 3] = b1
    vv = np.zeros((2, D)); vv[0, :] = np.arange(D) / 16.0; vv[1, :] = -np.arange(D) / 32.0
    qt, kt, vt = _bf16(np.vstack([qv, qv])), _bf16(kv), _bf16(vv)
    o, lse = orc.attn_rows(qt, kt, vt, 0, [0], sc)
    s0, s1 = sc * a * b0, sc * a * b1
    w0 = 1.0 / (1.0 + math.exp(s1 - s0))
    expect = w0 * vv[0] + (1.0 - w0) * vv[1]
    assert np.max(np.abs(o[0] - expect)) < 1e-14
    assert abs(lse[0] - math.log(math.exp(s0) + math.exp(s1))) < 1e-14

    # One key far above the rest: O is that key's value row.
    n = 64
    qv = np.zeros((n, D)); qv[:, 0] = 1.0
    kv = np.zeros((n, D)); kv[:, 0] = -1.0; kv[5, 0] = 512.0
    vt = _rand_bf16((n, D), 8)
    o, _ = orc.attn_rows(_bf16(qv), _bf16(kv), vt, 0, [0, 63], scale)
    assert _rel(o, np.tile(_head(vt, 0)[5], (2, 1))) < 1e-14


def attn_invariants(orc) -> None:
    scale = 1.0 / math.sqrt(D)
    n, heads = 200, 2
    q = _rand_bf16((n, heads * D), 21)
    k = _rand_bf16((n, heads * D), 22)
    v = _rand_bf16((n, heads * D), 23)
    rows = np.array([0, 3, 77, 199])
    base = [orc.attn_rows(q, k, v, h, rows, scale) for h in range(heads)]

    # permuting K and V rows together leaves O unchanged
    perm = torch.randperm(n, generator=torch.Generator().manual_seed(3))
    for h in range(heads):
        o, lse = orc.attn_rows(q, k[perm], v[perm], h, rows, scale)
        assert _rel(o, base[h][0]) < 1e-12 and _rel(lse, base[h][1]) < 1e-12

    # permuting Q rows permutes O rows
    qp = q[perm]
    inv = torch.argsort(perm).numpy()
    for h in range(heads):
        o, _ = orc.attn_rows(qp, k, v, h, inv[rows], scale)
        assert _rel(o, base[h][0]) < 1e-12

    # a head reads only its own 128 columns
    q2, k2, v2 = q.clone(), k.clone(), v.clone()
    q2[:, D:] = 0; k2[:, D:] = 3; v2[:, D:] = -1
    o, lse = orc.attn_rows(q2, k2, v2, 0, rows, scale)
    assert np.array_equal(o, base[0][0]) and np.array_equal(lse, base[0][1])
    q2, k2, v2 = q.clone(), k.clone(), v.clone()
    q2[:, :D] = 0; k2[:, :D] = 3; v2[:, :D] = -1
    o, lse = orc.attn_rows(q2, k2, v2, 1, rows, scale)
    assert np.array_equal(o, base[1][0]) and np.array_equal(lse, base[1][1])

    # adding one vector c to every key shifts each score row by a constant:
    # O unchanged, lse shifted by scale * q.c (small integers keep it exact)
    g = torch.Generator().manual_seed(9)
    qi = torch.randint(-3, 4, (n, D), generator=g).to(torch.float64)
    ki = torch.randint(-3, 4, (n, D), generator=g).to(torch.float64)
    ci = torch.randint(-3, 4, (1, D), generator=g).to(torch.float64)
    vi = _rand_bf16((n, D), 10)
    sc = 1.0 / 64.0
    o1, l1 = orc.attn_rows(_bf16(qi), _bf16(ki), vi, 0, rows, sc)
    o2, l2 = orc.attn_rows(_bf16(qi), _bf16(ki + ci), vi, 0, rows, sc)
    assert _rel(o2, o1) < 1e-12
    shift = sc * (qi.numpy()[rows] @ ci.numpy()[0])
    assert np.max(np.abs(l2 - (l1 + shift))) < 1e-10

    # linear in V: O(V1 + V2) = O(V1) + O(V2)
    v1 = torch.randint(-8, 9, (n, D), generator=g).to(torch.float64)
    v2 = torch.randint(-8, 9, (n, D), generator=g).to(torch.float64)
    qa = q[:, :D].contiguous(); ka = k[:, :D].contiguous()
    oa, _ = orc.attn_rows(qa, ka, _bf16(v1), 0, rows, scale)
    ob, _ = orc.attn_rows(qa, ka, _bf16(v2), 0, rows, scale)
    oc, _ = orc.attn_rows(qa, ka, _bf16(v1 + v2), 0, rows, scale)
    assert np.max(np.abs(oc - (oa + ob))) < 1e-12


def attn_probability_rows(orc) -> None:
    """With v_j = e_j (N <= 128) row i of O is row i of the softmax matrix P."""
    n = 100
    scale = 1.0 / math.sqrt(D)
    q = _rand_bf16((n, D), 31)
    k = _rand_bf16((n, D), 32)
    eye = np.zeros((n, D)); eye[np.arange(n), np.arange(n)] = 1.0
    rows = np.arange(n)
    p, lse = orc.attn_rows(q, k, _bf16(eye), 0, rows, scale)
    assert np.all(p >= 0.0)
    assert np.max(np.abs(p.sum(axis=1) - 1.0)) < 1e-13
    assert np.all(p[:, n:] == 0.0)
    # log p_ij - log p_ik equals the score difference, and lse = s_ij - log p_ij
    s = scale * (_head(q, 0) @ _head(k, 0).T)
    logp = np.log(p[:, :n])
    assert np.max(np.abs((logp - logp[:, :1]) - (s - s[:, :1]))) < 1e-10
    assert np.max(np.abs((s - logp) - lse[:, None])) < 1e-10


def attn_large_scores(orc) -> None:
    """Scores near 1e4 overflow exp unless the row maximum is subtracted."""
    n = 8
    qv = np.zeros((n, D)); qv[:, 0] = 64.0
    kv = np.zeros((n, D)); kv[:, 0] = np.array([120.0, 128.0, 96.0, -128.0, 0.0, 112.0, 127.0, 126.0])
    vv = np.zeros((n, D)); vv[:, 1] = np.arange(n)
    o, lse = orc.attn_rows(_bf16(qv), _bf16(kv), _bf16(vv), 0, [0, 5], 1.0)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    s = 64.0 * kv[:, 0]
    w = scipy.special.softmax(s)
    assert np.max(np.abs(o[:, 1] - float(np.dot(w, vv[:, 1])))) < 1e-12
    assert np.max(np.abs(lse - scipy.special.logsumexp(s))) < 1e-9


# ------------------------------------------------------------------ modulate
def modulate_vs_layer_norm(orc) -> float:
    c = 5376
    x = torch.cat([_rand_bf16((32, c), 41), _rand_bf16((32, c), 42, scale=5.0) + 3.0]).to(torch.bfloat16)
    g = torch.Generator().manual_seed(43)
    shift = (torch.randn(c, generator=g) * 0.1).to(torch.float32)
    scl = (torch.randn(c, generator=g) * 0.1).to(torch.float32)
    eps = 1e-6
    x64 = x.to(torch.float64)
    ref = torch.nn.functional.layer_norm(x64, (c,), eps=eps) * (1.0 + scl.to(torch.float64)) + shift.to(torch.float64)
    y = orc.modulate(x, shift.numpy(), scl.numpy(), eps)
    worst = float(np.max(np.abs(y - ref.numpy()) / np.maximum(1.0, np.abs(ref.numpy()))))
    # plain LayerNorm when the table rows are zero
    zero = np.zeros(c, dtype=np.float32)
    y0 = orc.modulate(x, zero, zero, eps)
    ref0 = torch.nn.functional.layer_norm(x64, (c,), eps=eps).numpy()
    return max(worst, float(np.max(np.abs(y0 - ref0))))


def modulate_closed_forms(orc) -> None:
    c = 5376
    g = torch.Generator().manual_seed(51)
    shift = (torch.randn(c, generator=g) * 0.1).to(torch.float32).numpy()
    scl = (torch.randn(c, generator=g) * 0.1).to(torch.float32).numpy()
    # a constant row normalises to 0, so y is the shift row exactly
    x = _bf16(np.full((2, c), 2.5))
    y = orc.modulate(x, shift, scl, 1e-6)
    assert np.array_equal(y, np.tile(shift.astype(np.float64), (2, 1)))
    # alternating +a, -a: mean 0, variance a^2, n = +-a / sqrt(a^2 + eps)
    a, eps = 1.75, 1e-6
    row = np.where(np.arange(c) % 2 == 0, a, -a)
    y = orc.modulate(_bf16(row[None, :]), shift, scl, eps)
    n = row / math.sqrt(a * a + eps)
    assert np.max(np.abs(y[0] - (n * (1.0 + scl.astype(np.float64)) + shift))) < 1e-14
    # LN ignores a constant added to the row (values are multiples of 1/8)
    xi = torch.randint(-40, 41, (3, c), generator=g).to(torch.float64) / 8.0
    y1 = orc.modulate(_bf16(xi), shift, scl, 1e-6)
    y2 = orc.modulate(_bf16(xi + 4.0), shift, scl, 1e-6)
    assert np.max(np.abs(y1 - y2)) < 1e-12
    # with eps = 0 LN ignores a positive scale factor on the row
    y3 = orc.modulate(_bf16(xi), shift, scl, 0.0)
    y4 = orc.modulate(_bf16(xi * 4.0), shift, scl, 0.0)
    assert np.max(np.abs(y3 - y4)) < 1e-12
    # rows are independent: a chosen row equals the same row of a full run
    y5 = orc.modulate(_bf16(xi), shift, scl, 1e-6, rows=[2, 0])
    assert np.array_equal(y5, y1[[2, 0]])


# ------------------------------------------------------------ gated residual
def gated_residual_closed_forms(orc) -> None:
    c = 64
    g = torch.Generator().manual_seed(61)
    x = _rand_bf16((4, c), 62)
    a = _rand_bf16((4, c), 63)
    xbits = x.view(torch.int16).numpy().view(np.uint16)
    # a zero gate or a zero branch leaves x unchanged, bit for bit
    _, yb = orc.gated_residual(x, a, np.zeros(c, dtype=np.float32))
    assert np.array_equal(yb, xbits)
    _, yb = orc.gated_residual(x, torch.zeros_like(a), (torch.randn(c, generator=g)).numpy())
    assert np.array_equal(yb, xbits)
    # per-channel gate read in channel order: x = 0, a = 1 gives the gate itself
    gate = (2.0 ** np.arange(-8, c - 8, dtype=np.float64)).astype(np.float32) * np.where(np.arange(c) % 3 == 0, -1, 1)
    gate = np.clip(gate, -2.0 ** 100, 2.0 ** 100).astype(np.float32)
    y, _ = orc.gated_residual(_bf16(np.zeros((1, c))), _bf16(np.ones((1, c))), gate)
    assert np.array_equal(y[0], gate.astype(np.float64))
    # small exact cases and ties to even at 1.0 (bf16 spacing there is 2^-7)
    cases = [  # (x, gate, a, expected bf16 value)
        (1.0, 0.5, 2.0, 2.0),
        (1.0, 1.0, 2.0 ** -8, 1.0),                    # tie -> even (1.0)
        (1.0 + 2.0 ** -7, 1.0, 2.0 ** -8, 1.0 + 2.0 ** -6),  # tie -> even (up)
        (-1.0, 1.0, -(2.0 ** -8), -1.0),
        (3.0, -0.25, 4.0, 2.0),
    ]
    for xv, gv, av, ev in cases:
        y, yb = orc.gated_residual(_bf16([[xv]]), _bf16([[av]]), np.array([gv], dtype=np.float32))
        assert y[0, 0] == xv + gv * av
        assert yb[0, 0] == _bf16([ev]).view(torch.int16).numpy().view(np.uint16)[0]


def round_bf16_cases(orc) -> None:
    r = orc.round_bf16
    assert r(1.0 + 2.0 ** -8) == 1.0                                  # tie, even below
    assert r(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6                   # tie, even above
    assert r(1.0 + 2.0 ** -8 + 2.0 ** -40) == 1.0 + 2.0 ** -7           # just above the tie: up
    assert r(1.0 + 2.0 ** -8 - 2.0 ** -40) == 1.0                      # just below: down
    assert r(-(1.0 + 2.0 ** -8 + 2.0 ** -40)) == -(1.0 + 2.0 ** -7)
    assert r(2.0 ** -134) == 0.0                                        # half the subnormal step: even (0)
    assert r(1.5 * 2.0 ** -133) == 2.0 ** -132                          # tie between 1 and 2 steps: 2
    assert r(3.39e38) == 255.0 * 2.0 ** 120                             # largest finite bf16
    assert math.isinf(r(3.40e38))                                       # past the last half step
    assert r(0.0) == 0.0 and math.isnan(r(float("nan")))


# ------------------------------------------------------- windowed attention
def window_mask_numpy(n: int, t: int, c: int, w: int) -> np.ndarray:
    """The window written out independently of the oracle: frames of t tokens,
    chunks of c frames, chunk distance <= w, plus first/last frame anchors."""
    frames = n // t
    f = np.arange(n) // t
    ch = f // c
    allowed = np.abs(ch[:, None] - ch[None, :]) <= w
    anchor = (f == 0) | (f == frames - 1)
    return allowed | anchor[:, None] | anchor[None, :]


def window_brute_force(orc, n: int, t: int, c: int, w: int, seed: int) -> float:
    q = _rand_bf16((n, 2 * D), seed)
    k = _rand_bf16((n, 2 * D), seed + 1)
    v = _rand_bf16((n, 2 * D), seed + 2)
    scale = 1.0 / math.sqrt(D)
    mask = window_mask_numpy(n, t, c, w)
    worst = 0.0
    for h in range(2):
        s = scale * (_head(q, h) @ _head(k, h).T)
        s = np.where(mask, s, -np.inf)
        o_ref = scipy.special.softmax(s, axis=1) @ _head(v, h)
        lse_ref = scipy.special.logsumexp(s, axis=1)
        o, lse = orc.attn_rows_window(q, k, v, h, np.arange(n), scale, t, c, w)
        worst = max(worst, _rel(o, o_ref), _rel(lse, lse_ref))
    return worst


def window_structure(orc) -> None:
    n, t, c, w = 12 * 16, 16, 3, 1        # 12 frames of 16 tokens, chunks of 3 frames
    scale = 1.0 / math.sqrt(D)
    q = _rand_bf16((n, D), 71)
    k = _rand_bf16((n, D), 72)
    v = _rand_bf16((n, D), 73)
    rows = np.arange(n)
    o_win, l_win = orc.attn_rows_window(q, k, v, 0, rows, scale, t, c, w)
    o_den, l_den = orc.attn_rows(q, k, v, 0, rows, scale)
    # a window wider than the clip is dense attention
    o_all, l_all = orc.attn_rows_window(q, k, v, 0, rows, scale, t, c, 12)
    assert _rel(o_all, o_den) < 1e-13 and _rel(l_all, l_den) < 1e-13
    # queries in the first and last frame see every key
    anchor_rows = np.r_[0:t, n - t:n]
    assert np.array_equal(o_win[anchor_rows], o_den[anchor_rows])
    # a middle query differs from dense attention, and ignores keys outside its window
    i = 6 * t + 5                          # frame 6, chunk 2: sees chunks 1-3 (frames 3-11) and frame 0
    assert np.max(np.abs(o_win[i] - o_den[i])) > 1e-6
    hidden = np.r_[t:3 * t]                # frames 1-2 (chunk 0 minus the anchor frame 0)
    k2, v2 = k.clone(), v.clone()
    k2[hidden] = 7.0
    v2[hidden] = -3.0
    o2, _ = orc.attn_rows_window(q, k2, v2, 0, [i], scale, t, c, w)
    assert np.array_equal(o2[0], o_win[i])
    seen = np.r_[4 * t:4 * t + 3]           # frame 4 is inside the window
    k3 = k.clone()
    k3[seen] = 2.0
    o3, _ = orc.attn_rows_window(q, k3, v, 0, [i], scale, t, c, w)
    assert np.max(np.abs(o3[0] - o_win[i])) > 1e-6
    # the window is symmetric and matches the independent numpy statement
    m = window_mask_numpy(n, t, c, w)
    got = np.array([[orc.window_allowed(a, b, n, t, c, w) for b in range(0, n, 4)] for a in range(0, n, 4)])
    assert np.array_equal(got, m[::4, ::4]) and np.array_equal(m, m.T)
