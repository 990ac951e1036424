"""Plant plausible mistakes in a copy of the CPU oracle and check that the pins catch each.

Each mutant is one textual change to oracle/specdec_ref.c (a dropped term, a wrong sign,
a transposed operand, an off-by-one, a wrong tie rule ...). The copy is compiled into a
temporary directory; the committed oracle is never touched.
"""
import os
import shutil

import pytest

import oracle
import _pins

SRC_DIR = os.path.dirname(oracle.__file__)

MUTANTS = {
    "accept_le_instead_of_lt": ("if ((double)c->uniforms[t] < alpha)", "if ((double)c->uniforms[t] <= alpha)"),
    "residual_transposed": ("double r = c->p[i] - (double)c->q[d * (int64_t)c->V + i];",
                            "double r = (double)c->q[d * (int64_t)c->V + i] - c->p[i];"),
    "model_free_residual_keeps_draft": ("wi = (i == x) ? 0.0 : c->p[i];", "wi = c->p[i];"),
    "temperature_dropped": ("double e = (c->z[i] > -INFINITY) ? exp(c->z[i] / T - m) : 0.0;",
                            "double e = (c->z[i] > -INFINITY) ? exp(c->z[i] - m * T) : 0.0;"),
    "greedy_ties_to_highest_index": ("if (c->z[i] > bz) { bz = c->z[i]; best = i; }",
                                     "if (c->z[i] >= bz) { bz = c->z[i]; best = i; }"),
    "race_multiplies_noise": ("s = c->w[i] / (double)E[i];", "s = c->w[i] * (double)E[i];"),
    "ratio_inverted": ("return px / qx;", "return qx / px;"),
    "mask_bit_order_reversed": ("return (int)((word >> (i & 31)) & 1u);",
                                "return (int)((word >> (31 - (i & 31))) & 1u);"),
    "counters_I_D_swapped": ("c->counters[1] += (uint64_t)(k - g);", "c->counters[1] += (uint64_t)g;"),
    "accepted_counter_off_by_one": ("c->counters[3] += (uint64_t)a;", "c->counters[3] += (uint64_t)(a + 1);"),
    "bonus_is_argmax": ("for (int32_t i = 0; i < c->V; ++i) c->w[i] = c->p[i];\n            emitted = exponential_race(c, t, b);",
                        "double zz; emitted = greedy_token(c, &zz);"),
    "grammar_prefix_from_last_invalid": ("if (g == k && (!ok || !grammar_allows(c, row0 + j, x))) g = j;",
                                         "if (!ok || !grammar_allows(c, row0 + j, x)) g = j;"),
    "bonus_row_skipped": ("for (int32_t j = 0; j <= k; ++j) {\n        const int64_t t = row0 + j;",
                          "for (int32_t j = 0; j < k; ++j) {\n        const int64_t t = row0 + j;"),
    "softmax_not_normalised": ("for (int32_t i = 0; i < c->V; ++i) c->p[i] /= S;\n    *m_out = m;", "*m_out = m;"),
    "empty_row_not_flagged": ("if (live == 0) {", "if (live < 0) {"),
    "model_free_alpha_is_one": ("if (!qmode) return px;", "if (!qmode) return 1.0;"),
    "telemetry_accepted_through_stop_row": ("for (int32_t j = 0; j < a; ++j) tm[2 * 33 + j] += 1;",
                                            "for (int32_t j = 0; j <= a; ++j) tm[2 * 33 + j] += 1;"),
    "telemetry_eligible_counts_every_draft": ("for (int32_t j = 0; j < g; ++j) tm[1 * 33 + j] += 1;",
                                              "for (int32_t j = 0; j < k; ++j) tm[1 * 33 + j] += 1;"),
    "telemetry_histogram_of_k": ("tm[3 * 33 + a] += 1;", "tm[3 * 33 + k] += 1;"),
    "ngram_tail_matches_itself": ("for (int64_t start = 0; start < L - n; ++start) {",
                                  "for (int64_t start = 0; start <= L - n; ++start) {"),
    "ngram_latest_start": ("for (int64_t start = 0; start < L - n; ++start) {\n                int64_t i = 0;\n                while (i < n && h[start + i] == tail[i]) ++i;\n                if (i == n) { hit_n = (int32_t)n; hit_start = start; break; }",
                           "for (int64_t start = 0; start < L - n; ++start) {\n                int64_t i = 0;\n                while (i < n && h[start + i] == tail[i]) ++i;\n                if (i == n) { hit_n = (int32_t)n; hit_start = start; }"),
    "ngram_short_windows_first": ("for (int64_t n = n_hi; n >= min_n && hit_n == 0; --n) {",
                                  "for (int64_t n = min_n; n <= n_hi && hit_n == 0; ++n) {"),
    "filter_drops_boundary_group": ("if (!(c->z[i] >= zp) || c->z[i] == -INFINITY) c->p[i] = 0.0;",
                                    "if (!(c->z[i] > zp) || c->z[i] == -INFINITY) c->p[i] = 0.0;"),
    "top_p_mass_not_renormalised": ("above += gm / Mk;", "above += gm;"),
    "top_k_off_by_one": ("if (k > 0 && k < m) zk = a[k - 1].z;", "if (k > 0 && k < m) zk = a[k].z;"),
    "no_stop_at_rejection": ("        a = j;\n        emitted = exponential_race(c, t, b);\n        break;",
                             "        a = j;\n        emitted = exponential_race(c, t, b);\n        c->out_tokens[t] = emitted;\n        continue;"),
}


def _build_mutant(tmp_path, name):
    search, repl = MUTANTS[name]
    src = open(os.path.join(SRC_DIR, "specdec_ref.c")).read()
    assert src.count(search) == 1, f"mutant {name}: search text must occur exactly once"
    d = tmp_path / name
    d.mkdir()
    shutil.copy(os.path.join(SRC_DIR, "specdec_ref.h"), d / "specdec_ref.h")
    (d / "specdec_ref.c").write_text(src.replace(search, repl))
    return oracle.build(src=str(d / "specdec_ref.c"), out=str(d / "libmutant.so"))


# fast versions of the pins (the chi-square at 2e5 trials is still far past any of these mutants)
def _run_pins(lib):
    failures = []
    checks = [
        ("worked_counter_example", lambda: _pins.check_worked_counter_example(lib)),
        ("telemetry", lambda: _pins.check_telemetry(lib)),
        ("ngram", lambda: _pins.check_ngram_proposer(lib)),
        ("top_k_top_p", lambda: _pins.check_top_k_top_p(lib, n=100_000)),
        ("strict_accept_comparison", lambda: _pins.check_strict_accept_comparison(lib)),
        ("edge_cases", lambda: _pins.check_edge_cases(lib)),
        ("residual_excludes_draft", lambda: _pins.check_residual_excludes_draft(lib)),
        ("p_equals_q", lambda: _pins.check_p_equals_q_accepts_all(lib, B=100)),
        ("greedy_brute_force", lambda: _pins.check_greedy_brute_force(lib, cases=30)),
        ("grammar_invariants", lambda: _pins.check_grammar_invariants(lib)),
        ("softmax_library", lambda: _pins.check_softmax_matches_library(lib)),
        ("chi_square", lambda: _pins.check_chi_square(lib, n=200_000)),
    ]
    for name, fn in checks:
        try:
            fn()
        except Exception as e:  # noqa: BLE001 - any failure counts as caught
            failures.append(f"{name}: {type(e).__name__}")
    return failures


def test_unmutated_copy_passes(tmp_path):
    d = tmp_path / "clean"
    d.mkdir()
    shutil.copy(os.path.join(SRC_DIR, "specdec_ref.h"), d / "specdec_ref.h")
    shutil.copy(os.path.join(SRC_DIR, "specdec_ref.c"), d / "specdec_ref.c")
    lib = oracle.build(src=str(d / "specdec_ref.c"), out=str(d / "libclean.so"))
    assert _run_pins(lib) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    lib = _build_mutant(tmp_path, name)
    failures = _run_pins(lib)
    assert failures, f"mutant {name} passed every pin"
