"""Planted mistakes in a copy of the oracle must fail the pins.

Each mutant is a small change to ``oracle/tq_oracle.c`` of the kind a
hand-written implementation could plausibly contain (a wrong sign, index,
normalisation, rounding mode, clamp or nibble order).  The copy is compiled
on the CPU and swapped in; the pins of ``test_oracle_pins`` are then run and
at least one must fail.
"""
import multiprocessing as mp
import os

import pytest

import oracle
import test_oracle_pins as pins
import test_oracle_blocked as blocked_pins
import test_oracle_swiglu as swiglu_pins
import test_oracle_modnorm as modnorm_pins

MUTANTS = {
    "sign_of_hadamard": ("& 1) ? -1 : 1", "& 1) ? 1 : -1"),
    "hadamard_index": ("popcount_u32((uint32_t)(i & j))", "popcount_u32((uint32_t)(i | j))"),
    "norm_1_over_n": ("return sqrt(1.0 / (double)n);", "return 1.0 / (double)n;"),
    "no_norm": ("o[g0 + i] = c * s;", "o[g0 + i] = s;"),
    "perturbed_h_entry": ("(double)H[i * n + j] * v[j]",
                          "(double)H[i * n + j + (i == 1 && j == 2)] * v[j]"),
    "tail_uses_norm_of_256": ("const double c = or_hadamard_norm(n);",
                              "const double c = or_hadamard_norm(256);"),
    "tail_group_refused": ("if (rest == 128 || rest == 64 || rest == 32) return (int)rest;",
                           "if (rest == 64 || rest == 32) return (int)rest;"),
    "truncate_not_round": ("double q = nearbyint(v[k] / (double)s);",
                           "double q = trunc(v[k] / (double)s);"),
    "round_half_away": ("double q = nearbyint(v[k] / (double)s);",
                        "double q = round(v[k] / (double)s);"),
    # (dropping the clamp is an equivalent mutant: with s = fp32(amax/qmax),
    # |v'/s| <= qmax (1 + 2^-24) < qmax + 1/2, so the clamp never acts)
    "clamp_too_tight": ("if (q > qmax) q = qmax;", "if (q > qmax - 1) q = qmax - 1;"),
    "scale_over_qmax_plus_1": ("(float)(amax / (double)qmax);\n        scales[r] = s;",
                               "(float)(amax / (double)(qmax + 1));\n        scales[r] = s;"),
    "block_scale_over_qmax_plus_1": ("(float)(amax / (double)qmax);\n            scales[r * nb + b] = s;",
                                     "(float)(amax / (double)(qmax + 1));\n            scales[r * nb + b] = s;"),
    "nibble_order": ("(uint8_t)(lo | (hi << 4))", "(uint8_t)(hi | (lo << 4))"),
    "dropped_product_term": (
        "for (int64_t k = 0; k < K; ++k) s += (int64_t)x[k] * (int64_t)w[k];",
        "for (int64_t k = 1; k < K; ++k) s += (int64_t)x[k] * (int64_t)w[k];"),
    "wrong_scale_in_y": ("(double)a->sx[m] * (double)a->sw[n] * (double)s",
                         "(double)a->sx[m] * (double)s"),
    "a16_wrong_index": ("s += (double)w[k] * or_bf16_to_f64(x[k]);",
                        "s += (double)w[k] * or_bf16_to_f64(x[k ^ 1]);"),
    "bf16_truncates": ("nearbyint(ldexp(a, -q))", "floor(ldexp(a, -q))"),
    "silu_sigmoid_of_minus_g": ("g[i] / (1.0 + exp(-g[i])) * u[i]", "g[i] / (1.0 + exp(g[i])) * u[i]"),
    "swiglu_plain_sigmoid_gate": ("g[i] / (1.0 + exp(-g[i])) * u[i]", "1.0 / (1.0 + exp(-g[i])) * u[i]"),
    "swiglu_gate_and_up_swapped": ("g[i] / (1.0 + exp(-g[i])) * u[i]", "u[i] / (1.0 + exp(-u[i])) * g[i]"),
    "modnorm_unbiased_variance": ("    var /= (double)K;", "    var /= (double)(K - 1);"),
    "modnorm_eps_outside_sqrt": ("1.0 / sqrt(var + eps)", "1.0 / (sqrt(var) + eps)"),
    "modnorm_eps_dropped": ("1.0 / sqrt(var + eps)", "1.0 / sqrt(var)"),
    "modnorm_mean_not_subtracted": ("h[k] = (x[k] - mu) * rstd", "h[k] = x[k] * rstd"),
    "modnorm_scale_without_one": ("* (1.0 + scale[k]) + shift[k]", "* scale[k] + shift[k]"),
    "modnorm_shift_and_scale_swapped": ("* (1.0 + scale[k]) + shift[k]", "* (1.0 + shift[k]) + scale[k]"),
    "block_amax_over_half_block": ("for (int64_t k = 0; k < G; ++k) {\n                const double a",
                                   "for (int64_t k = 0; k < G / 2; ++k) {\n                const double a"),
    "block_scale_stored_in_next_slot": ("scales[r * nb + b] = s;", "scales[r * nb + (b + 1) % nb] = s;"),
    "block_amax_carried_over": ("            double amax = 0.0;\n            for (int64_t k = 0; k < G",
                                "            static double amax = 0.0;\n            for (int64_t k = 0; k < G"),
    "blocked_product_next_block_scale": ("y += (double)a->sw[n * nb + b] * part;",
                                         "y += (double)a->sw[n * nb + (b + 1) % nb] * part;"),
    "blocked_product_drops_last_block": ("for (int64_t b = 0; b < nb; ++b) {\n                double part",
                                         "for (int64_t b = 0; b + 1 < nb; ++b) {\n                double part"),
    "blocked_product_row_scale": ("y += (double)a->sw[n * nb + b] * part;",
                                  "y += (double)a->sw[n * nb] * part;"),
}

PIN_TESTS = [
    lambda: [pins.test_sylvester_matches_scipy(n) for n in (4, 256)],
    lambda: pins.test_normalised_h256_is_exactly_orthogonal(),
    lambda: [pins.test_tail_norms(n) for n in (32, 128)],
    lambda: pins.test_group_layout(),
    lambda: pins.test_rotation_of_unit_vectors_gives_columns(),
    lambda: pins.test_rotation_of_ones_is_16_e0(),
    lambda: pins.test_rotation_tail_group_uses_its_own_h(),
    lambda: pins.test_explicit_product_equals_butterfly_exactly(),
    lambda: pins.test_rotation_leaves_the_product_unchanged(256, 512),
    lambda: [pins.test_quantiser_error_bound_and_range(q) for q in (127, 7)],
    lambda: pins.test_quantiser_scale_is_fp32_of_fp64_ratio(),
    lambda: pins.test_quantiser_ties_to_even(),
    lambda: pins.test_hadamard_rows_closed_form(),
    lambda: pins.test_int4_pack_layout(),
    lambda: pins.test_a8_product_brute_force(),
    lambda: pins.test_a16_product_brute_force(),
    lambda: pins.test_bf16_rounding_matches_exact_nearest(),
    lambda: swiglu_pins.test_silu_odd_part_is_the_identity(),
    lambda: swiglu_pins.test_silu_special_values(),
    lambda: swiglu_pins.test_swiglu_is_linear_in_up(),
    lambda: modnorm_pins.test_worked_row(),
    lambda: modnorm_pins.test_moments_and_invariances(),
    lambda: modnorm_pins.test_modulation_special_values(),
    lambda: modnorm_pins.test_constant_row_gives_the_shift(),
    lambda: blocked_pins.test_block_quantiser_error_bound_range_and_scale(7, 32),
    lambda: blocked_pins.test_blocks_scale_independently(),
    lambda: blocked_pins.test_block_quantiser_ties_to_even_in_a_later_block(),
    lambda: blocked_pins.test_blocked_product_brute_force(),
]


def _failures():
    n = 0
    for pin in PIN_TESTS:
        try:
            pin()
        except (AssertionError, ValueError):
            n += 1
    return n


def _count_in_child(so, queue):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
    with oracle.using(so):
        queue.put(_failures())


def _failures_isolated(so, limit=120):
    """Pin failures of a build, run in a child process: a planted mistake
    that crashes or never returns counts as caught (returns None)."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    p = ctx.Process(target=_count_in_child, args=(so, q))
    p.start()
    p.join(limit)
    if p.is_alive():
        p.kill()
        p.join()
        return None
    return q.get() if p.exitcode == 0 and not q.empty() else None


def test_unmutated_copy_passes(tmp_path):
    so = oracle.compile_variant(oracle.source(), str(tmp_path), "clean")
    assert _failures_isolated(so) == 0


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = oracle.source()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    so = oracle.compile_variant(src.replace(old, new), str(tmp_path), name)
    n = _failures_isolated(so)
    assert n is None or n > 0, f"no pin caught the planted mistake {name}"
