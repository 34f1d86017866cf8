"""The pins catch plausible mistakes.  Each case plants one slip in a copy of
the oracle's C source (on the CPU), builds it, runs the pin suite against it,
and requires that at least one pin fails; the unmodified source passes them
all (test_oracle_pins.py)."""
import os
import subprocess

import pytest

import oracle

import test_oracle_pins as P

SRC = os.path.join(os.path.dirname(oracle.__file__), "moe_oracle.c")

MUTANTS = {
    "router bias dropped": ("if (b) s += (double)b[e];", ""),
    "softmax sign flipped": ("p[e] = exp(l[e] - mx);", "p[e] = exp(mx - l[e]);"),
    "ties go to the higher index": ("while (pos > 0 && l[order[pos - 1]] < l[e]) {",
                                    "while (pos > 0 && l[order[pos - 1]] <= l[e]) {"),
    "gates not renormalised": ("gate[t * k + j] = renorm ? p[order[j]] / chosen : p[order[j]];",
                               "gate[t * k + j] = p[order[j]];"),
    "slots granted token-major": ("""    for (int j = 0; j < k; ++j)
        for (int64_t t = 0; t < T; ++t) {
            int e = idx[t * k + j];""", """    for (int64_t t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) {
            int e = idx[t * k + j];"""),
    "capacity truncated instead of rounded": ("return (int64_t)llround(((double)T / (double)E) * cf);",
                                              "return (int64_t)(((double)T / (double)E) * cf);"),
    "capacity counts T*k tokens": ("return (int64_t)llround(((double)T / (double)E) * cf);",
                                   "return (int64_t)llround(((double)T * 2.0 / (double)E) * cf);"),
    "counts after drops": ("counts[e] = (int32_t)fill[e];", "counts[e] = (int32_t)(fill[e] < cap ? fill[e] : cap);"),
    "SwiGLU halves swapped": ("a[n] = act_silu(z[n]) * z[F + n];", "a[n] = act_silu(z[F + n]) * z[n];"),
    "GELU tanh approximation": ("return z * 0.5 * (1.0 + erf(z / sqrt(2.0)));",
                                "return z * 0.5 * (1.0 + tanh(0.7978845608028654 * (z + 0.044715 * z * z * z)));"),
    "dropped slots still contribute": ("if (pos[t * k + j] < 0) continue;", ""),
    "down projection transposed": ("elem(w2, wdt, w2e + (int64_t)o * F + n)", "elem(w2, wdt, w2e + (int64_t)n * d + o)"),
    "aux loss without the E factor": ("return alpha * (double)E * s;", "return alpha * s;"),
    "P_i not divided by T": ("((double)counts[e] / (double)T) * (prob_sum[e] / (double)T)",
                             "((double)counts[e] / (double)T) * prob_sum[e]"),
    "group score is the group's sum": ("if (l[e] > score[g]) score[g] = l[e];", "score[g] += l[e];"),
    "group ties go to the higher index": ("while (pos > 0 && score[gorder[pos - 1]] < score[g]) {",
                                          "while (pos > 0 && score[gorder[pos - 1]] <= score[g]) {"),
    "groups strided instead of contiguous": ("if (!allowed[e / gsz]) continue;",
                                             "if (!allowed[e % n_group]) continue;"),
    "one group too many kept": ("for (int r = 0; r < topk_group; ++r) allowed[gorder[r]] = 1;",
                                "for (int r = 0; r <= topk_group && r < n_group; ++r) allowed[gorder[r]] = 1;"),
    "log-sum-exp without the shift back": ("lse[t] = mx + log(z);", "lse[t] = log(z);"),
    "z-loss of lse, not lse squared": ("s += lse[t] * lse[t];", "s += lse[t];"),
}


def _pins():
    """(name, callable) for one representative call of every pin."""
    return [
        ("topk brute force", lambda: [P.test_topk_brute_force_with_exact_ties(E, k)
                                      for E, k in [(4, 2), (6, 4), (8, 2)]]),
        ("tie rule", P.test_topk_tie_goes_to_lower_index),
        ("zero router", P.test_zero_router_picks_first_k_with_uniform_gates),
        ("softmax vs library", P.test_softmax_against_library_and_two_expert_sigmoid),
        ("sums", P.test_prob_sum_is_T_and_gate_sums),
        ("capacity table", lambda: [P.test_capacity_table(*row) for row in P._capacity_rows()]),
        ("slot order", lambda: [P.test_slot_order_brute_force(*a) for a in [(30, 4, 2, 9), (25, 5, 3, 4)]]),
        ("zero-router slot order", P.test_zero_router_slot_order_first_choices_in_token_order),
        ("rank beats token", P.test_rank_beats_token_order),
        ("dense ffn", lambda: [P.test_dense_ffn_special_case_matches_torch(a) for a in ("gelu", "swiglu")]),
        ("dense mixture", P.test_dense_mixture_k_equals_E),
        ("single row", P.test_single_row_ffn_exposes_activation),
        ("identity", P.test_identity_experts_return_x),
        ("identity with drops", P.test_identity_experts_with_drops_scale_by_kept_gates),
        ("aux uniform", lambda: [P.test_aux_loss_uniform_router_is_alpha_k(c) for c in (None, 0)]),
        ("aux circulant", lambda: P.test_aux_loss_circulant_router_is_alpha_k(8, 2)),
        ("aux concentration", P.test_aux_loss_one_hot_concentration),
        ("grouped brute force", lambda: [P.test_grouped_topk_brute_force_with_exact_ties(*a)
                                         for a in [(6, 3, 1, 2), (8, 4, 2, 2), (8, 4, 3, 5)]]),
        ("grouped worked example", P.test_grouped_routing_worked_example),
        ("grouped first choice", P.test_grouped_routing_keeps_first_choice_and_stays_in_kept_groups),
        ("lse", P.test_logsumexp_against_library_and_closed_forms),
        ("z-loss", P.test_z_loss_closed_forms),
        ("post-drop aux", lambda: [P.test_post_drop_aux_loss_uniform_router(c) for c in (0, 3)]),
    ]


@pytest.mark.parametrize("name", list(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site of {name!r} not found exactly once"
    path = tmp_path / "moe_oracle_mutant.c"
    path.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                           str(path), "-o", str(lib), "-lm"])
    saved = oracle._lib
    oracle._lib = oracle.load(str(lib))
    caught = []
    try:
        for pin, fn in _pins():
            try:
                fn()
            except (AssertionError, ValueError, IndexError):
                caught.append(pin)
    finally:
        oracle._lib = saved
    assert caught, f"no pin caught the planted mistake {name!r}"


# ---------------------------------------------------------------- backward ---

import importlib.util  # noqa: E402

import test_oracle_backward as PB  # noqa: E402

BWD_SRC = os.path.join(os.path.dirname(oracle.__file__), "backward.py")

BWD_MUTANTS = {
    "gate left out of do": ("dO = g[:, None] * DY[ts]", "dO = DY[ts]"),
    "softmax backward without the mean term": ("dL = P * (dP - np.sum(P * dP, axis=1, keepdims=True))",
                                               "dL = P * dP"),
    "renormalisation backward without the coupling term": (
        "dP[t, sel] += (dgate[t] - np.dot(dgate[t], gate[t])) / S", "dP[t, sel] += dgate[t] / S"),
    "silu derivative taken as the sigmoid": ("dsilu = s * (1.0 + gate * (1.0 - s))", "dsilu = s"),
    "GELU derivative without the density term": ("return da * (cdf + z * pdf)", "return da * cdf"),
    "z-loss gradient without the factor 2": ("(2.0 * z_beta / T)", "(z_beta / T)"),
    "aux gradient without the 1/T of P_i": ("dP += aux_weight * alpha * E * f[None, :] / T",
                                            "dP += aux_weight * alpha * E * f[None, :]"),
    "expert input gradient dropped": ("np.add.at(dX, ts, dZ @ W1e)", "pass"),
    "w2 gradient from the ungated dy": ("dW2[e] = dO.T @ A", "dW2[e] = DY[ts].T @ A"),
    "router input gradient dropped": ("dX += dL @ Wr", "pass"),
}


def _bwd_pins():
    return [
        ("autograd", lambda: [PB.test_backward_matches_autograd(i) for i in range(len(PB.CFGS))]),
        ("finite differences", lambda: PB.test_backward_matches_finite_differences_of_the_c_forward(0)),
        ("identity", PB.test_identity_experts_pass_dy_through),
        ("uniform aux", PB.test_aux_loss_gradient_of_a_uniform_router),
    ]


@pytest.mark.parametrize("name", list(BWD_MUTANTS))
def test_backward_pins_catch_planted_mistake(name, tmp_path):
    old, new = BWD_MUTANTS[name]
    src = open(BWD_SRC).read()
    assert src.count(old) == 1, f"mutation site of {name!r} not found exactly once"
    path = tmp_path / "backward_mutant.py"
    path.write_text(src.replace(old, new))
    spec = importlib.util.spec_from_file_location("oracle.backward_mutant", str(path),
                                                  submodule_search_locations=None)
    mod = importlib.util.module_from_spec(spec)
    mod.__package__ = "oracle"
    spec.loader.exec_module(mod)
    saved = PB.B
    PB.B = mod
    caught = []
    try:
        for pin, fn in _bwd_pins():
            try:
                fn()
            except AssertionError:
                caught.append(pin)
    finally:
        PB.B = saved
    assert caught, f"no pin caught {name!r}"
