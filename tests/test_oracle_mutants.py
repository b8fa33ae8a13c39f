"""Plant plausible mistakes in copies of the oracle and check that the pins
catch every one.  Each mutant is a text edit of ``oracle/oracle.c`` compiled
on the CPU into a temporary directory; the real oracle is untouched."""
import os
import subprocess

import pytest

import oracle
from oracle import build as obuild
from tests import pins

MUTANTS = {
    "no_max_subtraction": ("s[t] = exp(s[t] - m);", "s[t] = exp(s[t]);"),
    "no_normalisation": ("o[c] /= l;", "o[c] /= 1.0;"),
    "scale_dropped": ("s[t] = j->scale * dot;", "s[t] = dot;"),
    "head_offset_dropped_in_q": ("j->Q[i * j->ld + (int64_t)j->h * D + c]", "j->Q[i * j->ld + c]"),
    "k_used_for_v": ("const double *v = j->Vd + t * D;", "const double *v = j->Kd + t * D;"),
    "lse_without_max": ("j->lse[r] = m + log(l);", "j->lse[r] = log(l);"),
    "unbiased_variance": ("var /= (double)C;", "var /= (double)(C - 1);"),
    "scale_not_one_plus": ("y[c] = n * (1.0 + (double)j->t1[c]) + (double)j->t0[c];",
                           "y[c] = n * ((double)j->t1[c]) + (double)j->t0[c];"),
    "shift_scale_swapped": ("y[c] = n * (1.0 + (double)j->t1[c]) + (double)j->t0[c];",
                            "y[c] = n * (1.0 + (double)j->t0[c]) + (double)j->t1[c];"),
    "eps_dropped": ("1.0 / sqrt(var + j->eps)", "1.0 / sqrt(var)"),
    "residual_sign": ("bf16_to_double(x[c]) + (double)j->t0[c] * bf16_to_double(a[c])",
                      "bf16_to_double(x[c]) - (double)j->t0[c] * bf16_to_double(a[c])"),
    "round_via_float": ("double r = nearbyint(ldexp(x, -q));", "double r = nearbyint(ldexp((double)(float)x, -q));"),
    "round_truncates": ("double r = nearbyint(ldexp(x, -q));", "double r = trunc(ldexp(x, -q));"),
    "window_no_anchor_rows": ("if (fi == 0 || fi == frames - 1) return 1;", ""),
    "window_no_anchor_keys": ("if (fj == 0 || fj == frames - 1) return 1;", ""),
    "window_off_by_one": ("return d <= W;", "return d < W;"),
    "window_chunks_of_tokens": ("int64_t d = fi / C - fj / C;", "int64_t d = i / C - j / C;"),
}


def _all_pins(orc):
    """Run every pin; return the names of the ones that fail."""
    checks = {
        "brute_force": lambda: pins.attn_brute_force(orc, n=129, heads=2, seed=3) < 1e-12,
        "brute_force_n1": lambda: pins.attn_brute_force(orc, n=1, heads=2, seed=4) < 1e-12,
        "sdpa": lambda: pins.attn_vs_sdpa(orc, n=200, heads=2, seed=5) < 1e-12,
        "closed_forms": lambda: pins.attn_closed_forms(orc) is None,
        "invariants": lambda: pins.attn_invariants(orc) is None,
        "probability_rows": lambda: pins.attn_probability_rows(orc) is None,
        "large_scores": lambda: pins.attn_large_scores(orc) is None,
        "layer_norm": lambda: pins.modulate_vs_layer_norm(orc) < 1e-12,
        "modulate_closed": lambda: pins.modulate_closed_forms(orc) is None,
        "residual_closed": lambda: pins.gated_residual_closed_forms(orc) is None,
        "rounding": lambda: pins.round_bf16_cases(orc) is None,
        "window_brute": lambda: pins.window_brute_force(orc, 7 * 30, 30, 3, 1, seed=5) < 1e-12,
        "window_structure": lambda: pins.window_structure(orc) is None,
    }
    failed = []
    for name, fn in checks.items():
        try:
            ok = fn()
        except (AssertionError, FloatingPointError, ValueError):
            ok = False
        if not ok:
            failed.append(name)
    return failed


def test_unmutated_oracle_passes_every_pin():
    assert _all_pins(oracle.default()) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    src = open(obuild.SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    mutated = tmp_path / "oracle_mutant.c"
    mutated.write_text(src.replace(old, new))  # every occurrence (dense and windowed paths)
    lib = tmp_path / "liboracle_mutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", str(mutated), "-o", str(lib), "-lm"],
                   check=True)
    failed = _all_pins(oracle.Oracle(str(lib)))
    assert failed, f"mutant {name} passed every pin"
