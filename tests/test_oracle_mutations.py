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

# Slips in the block lifts (KATA-Sigma-g / KATA-M-g), caught by the block pins.
BLOCK_MUTATIONS = {
    "block_drop_sqrt2": ("psi[pidx(m, i, j)] = (i == j) ? sum : r2 * sum;",
                         "psi[pidx(m, i, j)] = (i == j) ? sum : sum;"),
    "block_sigma_without_cross_terms": ("if (family != 1 && a != b) continue;", "if (a != b) continue;"),
    "block_multi_with_cross_terms": ("if (family != 1 && a != b) continue;", "if (family == 0 && a != b) continue;"),
    "block_multi_wrong_block_start": ("lift(u + a * m, m, psi + a * packed_dim_i(m));",
                                      "lift(u + a, m, psi + a * packed_dim_i(m));"),
    "block_interleaved_blocks": ("sum += u[a * m + i] * u[a * m + j];", "sum += u[a + i * g] * u[a + j * g];"),
    "block_kernel_diagonal_pairs": ("dot(qu + a * m, ku + b * m, m)", "dot(qu + a * m, ku + a * m, m)"),
    "block_state_skips_normalise": ("normalize(k + (bh * T + t) * p, p, u.data());\n            lift_block(",
                                    "std::copy(k + (bh * T + t) * p, k + (bh * T + t) * p + p, u.begin());\n"
                                    "            lift_block("),
}


# Slips in the backward, caught by the backward pins.
BACKWARD_MUTATIONS = {
    "backward_drops_output_term": ("gw += G[j] * (vh[(int64_t)s * dv + j] - o[j]);",
                                   "gw += G[j] * vh[(int64_t)s * dv + j];"),
    "backward_missing_factor_two": ("const double gc = 2.0 * c * gw;", "const double gc = c * gw;"),
    "backward_skips_projection": ("for (int i = 0; i < p; ++i) gx[i] = (gu[i] - ug * u[i]) / nrm;",
                                  "for (int i = 0; i < p; ++i) gx[i] = gu[i] / nrm;"),
    "backward_unnormalised_value_weight": ("gv[(size_t)s * dv + j] += w / den * G[j];",
                                           "gv[(size_t)s * dv + j] += w * G[j];"),
    "backward_strict_causality": ("for (int s = 0; s <= t; ++s) {\n                const double c = dot(&qu[(size_t)t * p], "
                                  "&ku[(size_t)s * p], p);\n                const double w = c * c;",
                                  "for (int s = 0; s < t; ++s) {\n                const double c = dot(&qu[(size_t)t * p], "
                                  "&ku[(size_t)s * p], p);\n                const double w = c * c;"),
}


# Slips in the gated prefix, caught by the gated pins.
GATED_MUTATIONS = {
    "gated_decay_counts_own_gate": ("if (s < t) decay *= gh[s + 1];", "decay *= gh[s];"),
    "gated_gate_after_adding": ("S[a * dv + j] = gam * S[a * dv + j] + pk[a] * vt[j];",
                                "S[a * dv + j] = gam * (S[a * dv + j] + pk[a] * vt[j]);"),
    "gated_tree_wrong_carry": ("nx[c * w + e] = ca[c] * cx[(c - d) * w + e] + cx[c * w + e];",
                               "nx[c * w + e] = ca[c - d] * cx[(c - d) * w + e] + cx[c * w + e];"),
    "gated_readout_skips_first_gate": ("head_decay *= gh[t];", "head_decay *= 1.0;"),
    "gated_local_decay_off_by_one": ("for (int64_t r = s + 1; r < t1; ++r) decay *= gh[r];",
                                     "for (int64_t r = s; r < t1; ++r) decay *= gh[r];"),
}


def _gated_battery():
    import tests.test_oracle_gated_pins as gp
    yield lambda: gp.test_unit_gate_is_the_ungated_forward()
    yield lambda: gp.test_zero_gate_restarts_the_sequence(9)
    yield lambda: gp.test_constant_gate_identical_keys_is_the_moving_average()
    yield lambda: gp.test_gated_forms_agree(37, 8, 4, 1)
    yield lambda: gp.test_gated_scan_is_associative(7)
    yield lambda: gp.test_gated_split_call_with_carried_state(13)


def _backward_battery():
    import tests.test_oracle_backward_pins as bw
    yield lambda: bw.test_directional_derivatives(33, 5, 2)
    yield lambda: bw.test_gradients_are_orthogonal_to_q_and_k()
    yield lambda: bw.test_value_shift_and_value_gradient_sum()
    yield lambda: bw.test_single_token_and_zero_vectors()


def _block_battery():
    import tests.test_oracle_block_pins as bp
    yield lambda: bp.test_state_sizes_at_d64()
    yield lambda: bp.test_lifts_are_the_block_outer_products(12, 3)
    yield lambda: bp.test_inner_product_identities(12, 3)
    yield lambda: bp.test_g1_is_the_full_lift(4)
    yield lambda: bp.test_definition_and_lifted_recurrence_agree(bp.SIGMA, 12, 3, 9)
    yield lambda: bp.test_definition_and_lifted_recurrence_agree(bp.MULTI, 12, 4, 30)
    yield lambda: bp.test_sigma_with_scalar_blocks_is_the_running_mean()
    yield lambda: bp.test_disjoint_blocks_separate_the_families()
    yield lambda: bp.test_block_permutations()


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


ALL_MUTATIONS = {**MUTATIONS, **BLOCK_MUTATIONS, **BACKWARD_MUTATIONS, **GATED_MUTATIONS}


@pytest.mark.parametrize("name", sorted(MUTATIONS) + sorted(BLOCK_MUTATIONS) + sorted(BACKWARD_MUTATIONS)
                         + sorted(GATED_MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path, monkeypatch):
    old, new = ALL_MUTATIONS[name]
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
    battery = (_block_battery() if name in BLOCK_MUTATIONS
               else _backward_battery() if name in BACKWARD_MUTATIONS
               else _gated_battery() if name in GATED_MUTATIONS else _battery())
    for pin in battery:
        try:
            pin()
        except AssertionError:
            failures += 1
    assert failures > 0, f"no pin caught the planted mistake {name}"


def test_unmutated_battery_passes():
    for pin in _battery():
        pin()
    for pin in _block_battery():
        pin()
    for pin in _backward_battery():
        pin()
    for pin in _gated_battery():
        pin()
