"""The oracle pins are sharp: each plausible slip, planted in a private copy of
the oracle source on the CPU, makes at least one pin fail.

Each mutation is a textual edit of ``oracle/kata_oracle.cpp`` compiled into a
temporary directory and swapped in for the real library while a battery of
pins from ``test_oracle_pins.py`` runs.  The real oracle is never modified.
"""
import ctypes
import os
import subprocess

import pytest

import oracle.kata_oracle as km
from oracle import build as obuild
import tests.test_oracle_pins as pins

MUTATIONS = {
    "drop_sqrt2": ("r2 * u[i] * u[j]", "u[i] * u[j]"),
    "halve_diagonal": ("(i == j) ? u[i] * u[i]", "(i == j) ? 0.5 * u[i] * u[i]"),
    "skip_normalise": ("u[i] = nrm > 0.0 ? x[i] / nrm : 0.0;", "u[i] = x[i];"),
    "strict_causality_plain": ("for (int s = 0; s <= t; ++s)", "for (int s = 0; s < t; ++s)"),
    "unsquared_score": ("double w = c * c;", "double w = c * (c > 0 ? 1.0 : -1.0);"),
    "unit_denominator": ("den += w;", "den += 1.0;"),
    "wrong_normaliser_state": ("z[a] += pk[a];\n            }\n            normalize(qt",
                               "z[a] += pk[a] * pk[a];\n            }\n            normalize(qt"),
    "inclusive_prefix": (
        "for (int64_t e = 0; e < w; ++e) out[c * w + e] = run[e];\n"
        "        for (int64_t e = 0; e < w; ++e) run[e] += x[c * w + e];",
        "for (int64_t e = 0; e < w; ++e) run[e] += x[c * w + e];\n"
        "        for (int64_t e = 0; e < w; ++e) out[c * w + e] = run[e];"),
    "tree_off_by_one": ("(c >= d ? cur[(c - d) * w + e] : 0.0)", "(c > d ? cur[(c - d) * w + e] : 0.0)"),
    "transposed_state_read": ("num[j] += pq[a] * P[c * ws + a * dv + j]",
                              "num[j] += pq[a] * P[c * ws + j * n + a]"),
    "strict_causality_chunk": ("for (int64_t s = t0; s <= t; ++s)", "for (int64_t s = t0; s < t; ++s)"),
    "shifted_value_column": (
        "normalize(kt, p, u.data());\n            lift(u.data(), p, pk.data());\n"
        "            for (int64_t a = 0; a < n; ++a) {\n"
        "                for (int j = 0; j < dv; ++j) S[a * dv + j] += pk[a] * vt[j];",
        "normalize(kt, p, u.data());\n            lift(u.data(), p, pk.data());\n"
        "            for (int64_t a = 0; a < n; ++a) {\n"
        "                for (int j = 0; j < dv; ++j) S[a * dv + j] += pk[a] * vt[(j + 1) % dv];"),
}


def _battery():
    """Pins that run in well under a second each."""
    yield lambda: pins.test_lift_golden_values()
    yield lambda: pins.test_lift_identities(16)
    yield lambda: pins.test_worked_examples()
    yield lambda: pins.test_single_token_returns_its_value()
    yield lambda: pins.test_identical_keys_give_prefix_mean()
    yield lambda: pins.test_orthonormal_keys_exact_recall()
    yield lambda: pins.test_weights_visible_nonnegative_convex_causal()
    yield lambda: pins.test_psnr_regular_simplex_welch_bound(3)
    yield lambda: pins.test_rotation_and_scale_invariance()
    yield lambda: pins.test_state_readout_identity()
    yield lambda: pins.test_scan_tree_equals_sequential(5)
    yield lambda: pins.test_split_call_with_carried_state(21)
    for case in pins.FORM_CASES[2:5]:
        yield lambda case=case: pins.test_quadratic_recurrent_chunked_agree(*case)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path, monkeypatch):
    old, new = MUTATIONS[name]
    src = open(obuild.SRC).read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    mutated = tmp_path / "mut.cpp"
    mutated.write_text(src.replace(old, new, 1))
    lib = tmp_path / "libmut.so"
    cmd = [c if c not in (obuild.SRC, obuild.LIB) else (str(mutated) if c == obuild.SRC else str(lib))
           for c in obuild.CMD]
    subprocess.run(cmd, check=True)
    monkeypatch.setattr(km, "_lib", km._bind(ctypes.CDLL(os.fspath(lib))))
    failures = 0
    for pin in _battery():
        try:
            pin()
        except AssertionError:
            failures += 1
    assert failures > 0, f"no pin caught the planted mistake {name}"


def test_unmutated_battery_passes():
    for pin in _battery():
        pin()
