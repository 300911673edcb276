"""Planted mistakes in the oracle must fail its pins.

Each case copies the oracle's C source, plants one plausible mistake (a flipped
comparison, a wrong sign, a dropped renormalisation, a wrong index...),
compiles the copy with gcc and runs the pin checks against it. The unmodified
source must pass every check; every mutant must fail at least one. Nothing here
touches a GPU.
"""
import os

import numpy as np
import pytest

import oracle
import test_oracle_filter as F
import test_oracle_philox as P
import test_oracle_det as DD
import test_oracle_margins as MM
import test_oracle_verify as VV

MUTATIONS = {
    "accept_test_flipped": ("if (u_acc < (float)ratio) {", "if (u_acc > (float)ratio) {"),
    "residual_sign": ("r[j] = p[j] - q[j] > 0.0 ? p[j] - q[j] : 0.0;",
                      "r[j] = q[j] - p[j] > 0.0 ? q[j] - p[j] : 0.0;"),
    "residual_dropped": ("last = draw_ascending(Zr > 0.0 ? r : p, V, u_draw, &mgd);",
                         "last = draw_ascending(p, V, u_draw, &mgd);"),
    "no_renormalise_after_top_p": ("p[t] = p[t] / Wkept;", "p[t] = p[t] / W;"),
    "temperature_multiplies": ("p[t] = exp(e[t].x / T - zmax);", "p[t] = exp(e[t].x * T - zmax);"),
    "tie_break_high_index": ("return (ea->j < eb->j) ? -1 : (ea->j > eb->j) ? 1 : 0;",
                             "return (ea->j > eb->j) ? -1 : (ea->j < eb->j) ? 1 : 0;"),
    "argmax_last_of_ties": ("if (x > best_x) {", "if (x >= best_x) {"),
    "top_p_le": ("if (!(before_f < top_p)) {", "if (!(before_f <= top_p)) {"),
    "top_k_off_by_one": ("const int k = (top_k <= 0 || top_k >= V) ? V : top_k;",
                         "const int k = (top_k <= 0 || top_k >= V) ? V : (top_k > 1 ? top_k - 1 : 1);"),
    "bonus_wrong_row": ("int np = filter_dense(Xb + (size_t)gamma * row_bytes",
                        "int np = filter_dense(Xb + (size_t)(gamma - 1) * row_bytes"),
    "philox_key_word": ("uint32_t y0 = (uint32_t)(prod_b >> 32) ^ x1 ^ k0;",
                        "uint32_t y0 = (uint32_t)(prod_b >> 32) ^ x1 ^ k1;"),
    "uniform_bits": ("*u_accept = (float)((double)(w[0] >> 8) / 16777216.0);",
                     "*u_accept = (float)((double)(w[0] >> 9) / 16777216.0);"),
    "greedy_wrong_position": ("while (n < gamma && d[n] == argmax[n]) {",
                              "while (n < gamma && d[n] == argmax[n > 0 ? n - 1 : 0]) {"),
    "det_residual_keeps_draft": ("r[j] = j == tok ? 0.0 : p[j];", "r[j] = p[j];"),
    "det_accept_uses_draw_uniform": (
        "oracle_uniforms(seed, (uint32_t)b, (uint32_t)i, 0u, &u_acc, &u_draw);\n      update_margin(&mg, (double)u_acc, p_d);",
        "oracle_uniforms(seed, (uint32_t)b, (uint32_t)i, 0u, &u_draw, &u_acc);\n      update_margin(&mg, (double)u_acc, p_d);"),
    "det_accept_slack": ("if (u_acc < (float)p_d) {", "if (u_acc < (float)p_d + 0.02f) {"),
    "cut_margin_into_accept": ("      int nq = filter_dense(Yb + (size_t)i * row_bytes, V, dtype, T, top_k, top_p, q, &mgc);",
                               "      int nq = filter_dense(Yb + (size_t)i * row_bytes, V, dtype, T, top_k, top_p, q, &mg);"),
    "margins_not_split": ("  if (margin_cut) {\n    margin_cut[b] = cut;", "  if (0) {\n    margin_cut[b] = cut;"),
}


def _pin_checks(curand_pin):
    return [
        ("philox_vs_curand", lambda: P.test_philox_matches_curand(curand_pin)),
        ("unfiltered_softmax", lambda: F.test_unfiltered_is_softmax(0.6)),
        ("top_k_support", lambda: F.test_top_k_support_and_ratios(3, True)),
        ("top_k_support_5", lambda: F.test_top_k_support_and_ratios(5, False)),
        ("top_p_prefix", lambda: F.test_top_p_is_minimal_prefix(0.8, 4)),
        ("top_p_exact_boundary", lambda: F.test_top_p_exact_boundary()),
        ("argmax_numpy", F.test_argmax_matches_numpy_first_max),
        ("greedy_decoding", lambda: VV.test_greedy_is_target_argmax_decoding("f32")),
        ("law_closed_form", lambda: VV.test_sampling_law_closed_form(*VV.LAW_CASES[1])),
        ("identical_draft", VV.test_identical_draft_is_always_accepted),
        ("uniforms_uniform", P.test_uniforms_are_uniform_and_independent),
        ("det_point_mass", lambda: DD.test_det_equals_general_rule_with_point_mass_drafts(20, 0.95)),
        ("det_law", lambda: DD.test_det_accept_length_and_token_laws(*DD.DET_LAW_CASES[3])),
        ("cut_margin", lambda: MM.test_cut_margin_closed_form(4, 0.6)),
        ("accept_margin", MM.test_accept_margin_alone_is_the_uniforms_gap),
    ]


def _run_all(checks):
    failed = []
    for name, fn in checks:
        try:
            fn()
        except Exception:   # an assertion, or a crash on the mutant's output
            failed.append(name)
    return failed


@pytest.fixture(scope="module")
def variant_dir(tmp_path_factory):
    return tmp_path_factory.mktemp("oracle_variants")


def _with_lib(lib, checks):
    saved = oracle._lib
    oracle._lib = lib
    try:
        return _run_all(checks)
    finally:
        oracle._lib = saved


def test_unmodified_oracle_passes_all_checks(variant_dir, curand_pin):
    src = oracle.source_text()
    lib = oracle.load_variant(oracle.compile_variant(src, str(variant_dir / "lib_clean.so")))
    assert _with_lib(lib, _pin_checks(curand_pin)) == []


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, variant_dir, curand_pin):
    old, new = MUTATIONS[name]
    src = oracle.source_text()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    path = str(variant_dir / f"lib_{name}.so")
    lib = oracle.load_variant(oracle.compile_variant(src.replace(old, new), path))
    failed = _with_lib(lib, _pin_checks(curand_pin))
    assert failed, f"planted mistake {name!r} passed every pin"
