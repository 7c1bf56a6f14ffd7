"""Planted mistakes: each plausible error in the oracle's definition must fail a pin.

A copy of the oracle source is edited on the CPU (only inside the sequential
recurrence, which is the definition the others are checked against), compiled
to a temporary library and run through the pins of test_oracle_pins.py. Every
mutant must be caught by at least one pin.
"""
import os

import pytest

import test_oracle_pins as pins
from oracle import oracle

SEQ_BEGIN = "int m3o_scan_seq("
SEQ_END = "int m3o_scan_rope("
BC_BEGIN = "int m3o_bc_norm("

MUTANTS = {
    "beta_term_not_rotated": [
        ("Gm[i] = hs[i] + beta_hat * Up[i];", "Gm[i] = hs[i];"),
        ("hs[i] = alpha * Gm[i] + gamma * U[i];",
         "hs[i] = alpha * (Gm[i] + beta_hat * Up[i]) + gamma * U[i];"),
    ],
    "rotation_clockwise": [
        ("Gm[(2 * k) * P + p] = c * g0 - s * g1;", "Gm[(2 * k) * P + p] = c * g0 + s * g1;"),
        ("Gm[(2 * k + 1) * P + p] = s * g0 + c * g1;",
         "Gm[(2 * k + 1) * P + p] = -s * g0 + c * g1;"),
    ],
    "rotation_not_orthogonal": [
        ("Gm[(2 * k + 1) * P + p] = s * g0 + c * g1;",
         "Gm[(2 * k + 1) * P + p] = -s * g0 - c * g1;"),
    ],
    "beta_uses_previous_lambda": [
        ("const double beta_hat = (1.0 - lm) * d;",
         "const double beta_hat = (1.0 - lam[IX_T(b, (t ? t - 1 : 0), h)]) * d;"),
    ],
    "beta_uses_previous_delta": [
        ("const double beta_hat = (1.0 - lm) * d;",
         "const double beta_hat = (1.0 - lm) * dt[IX_T(b, (t ? t - 1 : 0), h)];"),
    ],
    "gamma_dropped": [
        ("hs[i] = alpha * Gm[i] + gamma * U[i];", "hs[i] = alpha * Gm[i];"),
    ],
    "gamma_decayed": [
        ("hs[i] = alpha * Gm[i] + gamma * U[i];", "hs[i] = alpha * (Gm[i] + gamma * U[i]);"),
    ],
    "angle_without_delta": [
        ("const double phi = d * theta[IX_TH(b, t, g, k)];",
         "const double phi = theta[IX_TH(b, t, g, k)];"),
    ],
    "output_rank_transposed": [
        ("for (int64_t n = 0; n < N; ++n) acc += Ct[n * R + r] * hs[n * P + p];",
         "for (int64_t n = 0; n < N; ++n) acc += Ct[n * R + (R - 1 - r)] * hs[n * P + p];"),
    ],
    "c_bias_from_b": [
        ("Ct[n * R + r] = C[IX_BC(b, t, g, n, r)] + (C_bias ? C_bias[IX_BIAS(h, n, r)] : 0.0);",
         "Ct[n * R + r] = C[IX_BC(b, t, g, n, r)] + (C_bias ? B_bias[IX_BIAS(h, n, r)] : 0.0);"),
    ],
    "previous_input_not_kept": [
        ("memcpy(Up, U, sizeof(double) * (size_t)(N * P));", ""),
    ],
}

# Mistakes planted in BCNorm (the normalisation of B and C over N).
BC_MUTANTS = {
    "bc_norm_without_root": [
        ("const double inv = 1.0 / sqrt(ss / (double)N + eps);",
         "const double inv = 1.0 / (ss / (double)N + eps);"),
    ],
    "bc_norm_sum_not_mean": [
        ("const double inv = 1.0 / sqrt(ss / (double)N + eps);",
         "const double inv = 1.0 / sqrt(ss + eps);"),
    ],
    "bc_norm_over_ranks": [
        ("const double v = in[IX_BC(b, t, g, n, r)];", "const double v = in[IX_BC(b, t, g, n, 0)];"),
    ],
    "bc_norm_eps_outside_root": [
        ("const double inv = 1.0 / sqrt(ss / (double)N + eps);",
         "const double inv = 1.0 / (sqrt(ss / (double)N) + eps);"),
    ],
}


def _mutate(src, edits, begin=SEQ_BEGIN, end=SEQ_END):
    i0 = src.index(begin)
    i1 = src.index(end) if end else len(src)
    body = src[i0:i1]
    for old, new in edits:
        assert body.count(old) == 1, old
        body = body.replace(old, new)
    return src[:i0] + body + src[i1:]


def _run_pins(orc):
    checks = [
        lambda: pins.test_euler_reduction(orc),
        lambda: pins.test_convergence_order(orc, 0.5, 2.0),
        lambda: pins.test_convergence_order(orc, 1.0, 1.0),
        lambda: pins.test_geometric_series(orc),
        lambda: pins.test_rope_form_equals_explicit_rotation(orc),
        lambda: pins.test_parity_fixture(orc),
        lambda: pins.test_rotation_preserves_norm(orc),
        lambda: pins.test_chunked_equals_sequential(orc, 4, 3),
        lambda: pins.test_dense_mask_product_form(orc, True),
        lambda: pins.test_mimo_is_sum_of_siso(orc),
        lambda: pins.test_hand_two_tokens(orc),
    ]
    failed = 0
    for c in checks:
        try:
            c()
        except AssertionError:
            failed += 1
    return failed


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    src = _mutate(oracle.source_text(), MUTANTS[name])
    path = oracle.build_variant(src, os.path.join(str(tmp_path), "libmut_%s.so" % name))
    failed = _run_pins(oracle.Oracle(path))
    assert failed >= 1, "planted mistake %r passed every pin" % name


def _run_bc_pins(orc):
    failed = 0
    for c in (pins.test_bc_norm_hand_fixture, pins.test_bc_norm_invariants,
              pins.test_bc_norm_matches_the_input_recipe):
        try:
            c(orc)
        except AssertionError:
            failed += 1
    return failed


@pytest.mark.parametrize("name", sorted(BC_MUTANTS))
def test_bc_norm_mutant_is_caught(tmp_path, name):
    src = _mutate(oracle.source_text(), BC_MUTANTS[name], BC_BEGIN, None)
    path = oracle.build_variant(src, os.path.join(str(tmp_path), "libmut_%s.so" % name))
    assert _run_bc_pins(oracle.Oracle(path)) >= 1, "planted mistake %r passed every pin" % name


def test_unmutated_source_passes_every_pin(tmp_path):
    path = oracle.build_variant(oracle.source_text(), os.path.join(str(tmp_path), "libsame.so"))
    orc = oracle.Oracle(path)
    assert _run_pins(orc) == 0
    assert _run_bc_pins(orc) == 0
