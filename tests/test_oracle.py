"""Pins for the fp64 oracle, independent of the oracle itself.

Each check is something the mathematics fixes without the oracle's own
formula: brute force on tiny inputs, closed forms, invariants, and library
routines on the CPU (torch float64 scaled_dot_product_attention and
layer_norm).  ``test_oracle_mutants.py`` plants plausible mistakes in copies of
the oracle and shows that these pins catch each one.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from tests import pins

D = 128


def rand_bf16(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g, dtype=torch.float32) * scale).to(torch.bfloat16)


# ---------------------------------------------------------------- attention
@pytest.mark.parametrize("n", [1, 2, 3, 17, 128, 129])
def test_attn_brute_force_tiny(n):
    assert pins.attn_brute_force(oracle, n=n, heads=2, seed=n) < 1e-12


@pytest.mark.parametrize("n,heads", [(257, 3), (1008, 2)])
def test_attn_matches_torch_sdpa_f64(n, heads):
    assert pins.attn_vs_sdpa(oracle, n=n, heads=heads, seed=7) < 1e-12


def test_attn_closed_forms():
    pins.attn_closed_forms(oracle)


def test_attn_invariants():
    pins.attn_invariants(oracle)


def test_attn_rows_are_probabilities():
    pins.attn_probability_rows(oracle)


def test_attn_large_scores_stay_finite():
    pins.attn_large_scores(oracle)


def test_attn_rejects_bad_rows():
    q = rand_bf16((4, D), 1)
    with pytest.raises(ValueError):
        oracle.attn_rows(q, q, q, 0, [4], 0.1)
    with pytest.raises(ValueError):
        oracle.attn_rows(q, q, q, 0, [-1], 0.1)


# ----------------------------------------------------------------- modulate
def test_modulate_vs_torch_layer_norm():
    assert pins.modulate_vs_layer_norm(oracle) < 1e-12


def test_modulate_closed_forms():
    pins.modulate_closed_forms(oracle)


# ----------------------------------------------------------- gated residual
def test_gated_residual_closed_forms():
    pins.gated_residual_closed_forms(oracle)


def test_round_bf16_ties_and_double_rounding():
    pins.round_bf16_cases(oracle)


def test_round_bf16_matches_torch_on_float32_values():
    g = torch.Generator().manual_seed(11)
    f = torch.randn(20000, generator=g, dtype=torch.float32) * torch.exp(torch.randn(20000, generator=g) * 8)
    ref = f.to(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.round_bf16(float(v)) for v in f.tolist()])
    assert np.array_equal(ref, got)


# ------------------------------------------------------- windowed attention
@pytest.mark.parametrize("n,t,c,w", [(10 * 8, 8, 2, 1), (7 * 30, 30, 3, 1), (5 * 13, 13, 5, 1), (9 * 4, 4, 1, 2)])
def test_window_brute_force(n, t, c, w):
    assert pins.window_brute_force(oracle, n, t, c, w, seed=n) < 1e-12


def test_window_structure():
    pins.window_structure(oracle)


def test_window_density_under_this_reading():
    """Video-only share of admitted (query, key) frame pairs at 42 and 102
    latent frames; the pages quote 42.1 % and 20.0 % for sequences that also
    hold text and audio tokens, which see and are seen by everything."""
    for frames, expect in ((42, 0.400), (102, 0.177)):
        got = sum(oracle.window_allowed(a, b, frames, 1) for a in range(frames) for b in range(frames)) / frames ** 2
        assert abs(got - expect) < 5e-4
