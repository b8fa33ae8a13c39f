"""Pins for the fp64 Video Delta Attention oracle (oracle/delta.py): the
page's least-squares definition checked by autograd and by a generic
minimiser, the stability bound, closed forms and the readout indexing."""
import numpy as np
import pytest
import scipy.optimize
import torch

from oracle import delta as V


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def objective_torch(s, s_bar, k_hat, v, beta):
    """1/2 ||S - Sbar||_F^2 + 1/2 sum_u beta_u ||S k_u - v_u||^2, as printed."""
    r = s @ k_hat.T - v.T
    return 0.5 * ((s - s_bar) ** 2).sum() + 0.5 * (beta[None, :] * r ** 2).sum()


def test_update_is_the_argmin_autograd():
    d, t = 16, 40
    rng = np.random.default_rng(1)
    k_hat = V.l2_normalize(rng.standard_normal((t, d)))
    v = rng.standard_normal((t, d))
    beta = rng.uniform(0.0, 2.0, t)
    alpha = rng.uniform(0.2, 1.0, d)
    s_prev = rng.standard_normal((d, d))
    a, b = V.frame_stats(k_hat, v, beta)
    s_new = V.update(s_prev, alpha, a, b)
    s = torch.tensor(s_new, requires_grad=True)
    f = objective_torch(s, torch.tensor(s_prev * alpha[None, :]), torch.tensor(k_hat), torch.tensor(v),
                        torch.tensor(beta))
    f.backward()
    assert float(s.grad.abs().max()) < 1e-10


def test_update_matches_a_generic_minimiser():
    d, t = 4, 6
    rng = np.random.default_rng(2)
    k_hat = V.l2_normalize(rng.standard_normal((t, d)))
    v = rng.standard_normal((t, d))
    beta = rng.uniform(0.1, 1.5, t)
    alpha = rng.uniform(0.3, 1.0, d)
    s_prev = rng.standard_normal((d, d))
    s_bar = s_prev * alpha[None, :]

    def f(x):
        s = x.reshape(d, d)
        r = s @ k_hat.T - v.T
        return 0.5 * ((s - s_bar) ** 2).sum() + 0.5 * (beta[None, :] * r ** 2).sum()

    res = scipy.optimize.minimize(f, np.zeros(d * d), method="BFGS", options={"gtol": 1e-12})
    a, b = V.frame_stats(k_hat, v, beta)
    assert np.abs(res.x.reshape(d, d) - V.update(s_prev, alpha, a, b)).max() < 1e-6


def test_carried_state_never_grows():
    """The page's bound: ||Diag(alpha)(I + A)^{-1}|| <= 1, so with nothing
    written (B = 0) the state norm cannot grow from one frame to the next."""
    d, t = 32, 100
    rng = np.random.default_rng(3)
    for trial in range(20):
        k_hat = V.l2_normalize(rng.standard_normal((t, d)))
        beta = rng.uniform(0.0, 3.0, t)
        alpha = rng.uniform(0.0, 1.0, d)
        a, _ = V.frame_stats(k_hat, np.zeros((t, d)), beta)
        assert np.linalg.norm(np.diag(alpha) @ np.linalg.inv(np.eye(d) + a), 2) <= 1.0 + 1e-12
        s_prev = rng.standard_normal((d, d))
        s_new = V.update(s_prev, alpha, a, np.zeros((d, d)))
        assert np.linalg.norm(s_new, 2) <= np.linalg.norm(s_prev, 2) + 1e-12


def test_no_writes_pure_decay_and_seed_counted_once():
    d, tok, frames = 8, 5, 9
    n = tok * frames
    q, k, v = _rand((n, d), 4), _rand((n, d), 5), _rand((n, d), 6)
    s_t = _rand((d, d), 7)
    beta = np.zeros(n)
    # alpha = 1: every state is the seed S_T / 2, every readout is S_T q_hat
    rows = np.arange(n)
    out, fwd, rev = V.delta_attn_head(q, k, v, beta, np.ones((frames, d)), s_t, rows, tok, 2, 1)
    assert np.allclose(fwd, 0.5 * s_t) and np.allclose(rev, 0.5 * s_t)
    assert np.abs(out - V.l2_normalize(q) @ s_t.T).max() < 1e-12
    # alpha = 1/2: the forward state after frames 1..t is S_T/2 * 2^-t
    _, fwd, rev = V.delta_attn_head(q, k, v, beta, np.full((frames, d), 0.5), s_t, rows, tok, 2, 1)
    for t in range(frames - 1):
        assert np.abs(fwd[t] - 0.5 * s_t * 0.5 ** t).max() < 1e-12
    for t in range(1, frames):
        assert np.abs(rev[t] - 0.5 * s_t * 0.5 ** (frames - 1 - t)).max() < 1e-12


def test_strong_write_stores_the_value():
    d = 8
    rng = np.random.default_rng(8)
    k_hat = V.l2_normalize(rng.standard_normal((1, d)))
    v = rng.standard_normal((1, d))
    a, b = V.frame_stats(k_hat, v, np.array([1e9]))
    s = V.update(rng.standard_normal((d, d)), np.ones(d), a, b)
    assert np.abs(s @ k_hat[0] - v[0]).max() < 1e-6


def test_readout_uses_the_states_around_the_window():
    d, tok, frames, c, w = 4, 3, 16, 2, 1
    n = tok * frames
    q, k, v = _rand((n, d), 9), _rand((n, d), 10), _rand((n, d), 11)
    beta = np.abs(_rand(n, 12))
    alpha = np.random.default_rng(13).uniform(0.5, 1.0, (frames, d))
    fwd, rev = V.delta_states(q, k, v, beta, alpha, None, tok)
    q_hat = V.l2_normalize(q)
    for frame in (0, 3, 7, 15):
        i = frame * tok + 1
        ch = frame // c
        p, nx = (ch - w) * c - 1, (ch + w + 1) * c
        sf = fwd[p] if p >= 1 else np.zeros((d, d))
        sr = rev[nx] if nx <= frames - 2 else np.zeros((d, d))
        o = V.delta_readout(q, fwd, rev, [i], tok, c, w)
        assert np.abs(o[0] - (sf + sr) @ q_hat[i]).max() < 1e-12
    # the anchor frames write nothing: states skip frames 0 and F-1
    assert np.array_equal(fwd[0], np.zeros((d, d))) and np.array_equal(rev[frames - 1], np.zeros((d, d)))
    assert np.array_equal(fwd[frames - 1], fwd[frames - 2]) and np.array_equal(rev[0], rev[1])


def test_readout_sees_only_frames_outside_the_window():
    """The page: a frame reads a summary of the past before its softmax window
    and of the future after it (the window itself is the softmax branch's).
    With values zero everywhere except one written frame f, a query's readout
    is non-zero exactly when f lies outside its window -- before it (carried
    by the forward scan) or after it (by the reverse scan) -- and exactly zero
    when f lies inside it.  The window is taken from its own definition: the
    frames whose chunk is within window_chunks of the query's chunk."""
    d, tok, frames, c, w = 8, 3, 16, 2, 1
    n = tok * frames
    rng = np.random.default_rng(21)
    q, k = rng.standard_normal((n, d)), rng.standard_normal((n, d))
    beta = rng.uniform(0.5, 1.5, n)
    alpha = np.ones((frames, d))
    for f in range(1, frames - 1):  # the anchor frames 0 and F-1 are written by neither scan
        v = np.zeros((n, d))
        v[f * tok:(f + 1) * tok] = rng.standard_normal((tok, d))
        rows = np.arange(n)
        out, _, _ = V.delta_attn_head(q, k, v, beta, alpha, None, rows, tok, c, w)
        for i in rows:
            g = i // tok
            inside = abs(f // c - g // c) <= w
            mag = np.abs(out[i]).max()
            if inside:
                assert mag == 0.0, (f, g, mag)
            else:
                assert mag > 1e-6, (f, g, mag)


def test_queries_and_keys_enter_only_through_their_directions():
    """The branch L2-normalises q and k: scaling a token's q or k changes nothing."""
    d, tok, frames = 6, 4, 7
    n = tok * frames
    q, k, v = _rand((n, d), 14), _rand((n, d), 15), _rand((n, d), 16)
    beta = np.abs(_rand(n, 17))
    alpha = np.random.default_rng(18).uniform(0.5, 1.0, (frames, d))
    s_t = _rand((d, d), 19)
    rows = np.arange(n)
    base = V.delta_attn_head(q, k, v, beta, alpha, s_t, rows, tok, 2, 1)
    scale = np.exp(_rand((n, 1), 20))
    other = V.delta_attn_head(q * scale, k * scale[::-1], v, beta, alpha, s_t, rows, tok, 2, 1)
    for x, y in zip(base, other):
        assert np.abs(x - y).max() < 1e-10


# Plausible mistakes planted in copies of the oracle module; each must fail a pin.
MUTANTS = {
    "minus_a": ("np.eye(a.shape[0]) + a", "np.eye(a.shape[0]) - a"),
    "decay_rows": ("s_prev * alpha[None, :] + b", "s_prev * alpha[:, None] + b"),
    "no_transpose_solve": ("np.linalg.solve(np.eye(a.shape[0]) + a, rhs.T).T", "np.linalg.solve(np.eye(a.shape[0]) + a, rhs)"),
    "b_transposed": ("b = (v * beta[:, None]).T @ k_hat", "b = k_hat.T @ (v * beta[:, None])"),
    "full_seed": ("0.5 * np.asarray(text_state, dtype=np.float64)", "np.asarray(text_state, dtype=np.float64)"),
    "window_off_by_one": ("p = max((c - window_chunks) * chunk_frames - 1, 0)", "p = max((c - window_chunks) * chunk_frames, 0)"),
    "no_key_normalisation": ("k_hat = l2_normalize(k)", "k_hat = k"),
    "window_end_off_by_one": ("nx = min((c + window_chunks + 1) * chunk_frames, frames - 1)",
                              "nx = min((c + window_chunks + 1) * chunk_frames - 1, frames - 1)"),
}


def _mutant_module(name):
    import importlib.util
    import os
    import sys
    import tempfile
    src = open(V.__file__).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, name
    d = tempfile.mkdtemp()
    path = os.path.join(d, f"delta_{name}.py")
    open(path, "w").write(src.replace(old, new))
    spec = importlib.util.spec_from_file_location(f"delta_{name}", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_delta_mutant_is_caught(name, monkeypatch):
    mod = _mutant_module(name)
    import sys
    monkeypatch.setattr(sys.modules[__name__], "V", mod)
    checks = [test_update_is_the_argmin_autograd, test_update_matches_a_generic_minimiser,
              test_carried_state_never_grows, test_no_writes_pure_decay_and_seed_counted_once,
              test_strong_write_stores_the_value, test_readout_uses_the_states_around_the_window,
              test_readout_sees_only_frames_outside_the_window,
              test_queries_and_keys_enter_only_through_their_directions]
    failed = 0
    for fn in checks:
        try:
            fn()
        except (AssertionError, np.linalg.LinAlgError, ValueError):
            failed += 1
    assert failed >= 1, f"mutant {name} passed every pin"
