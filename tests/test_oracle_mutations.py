"""Planted mistakes in a copy of the oracle must trip at least one pin.

Each mutation edits the C source of a temporary copy of the oracle (a
dropped clamp, a swapped operand, an off-by-one row, a wrong tie-break, ...),
builds it with the same flags and runs the pins against it. This shows the
pins constrain every step of the oracle, not just that it runs. CPU only; the
real oracle is never modified.
"""

import os

import pytest

import oracle
import oracle_pins as P

MUTATIONS = {
    "residual_operands_swapped*": (
        "w = fmax(0.0, w - prob(Lq, dt, offq, v, T, Mq[m], Zq[m]));",
        "w = fmax(0.0, prob(Lq, dt, offq, v, T, Mq[m], Zq[m]) - w);"),
    "residual_clamp_dropped": (
        "w = fmax(0.0, w - prob(Lq, dt, offq, v, T, Mq[m], Zq[m]));",
        "w = w - prob(Lq, dt, offq, v, T, Mq[m], Zq[m]);"),
    "ratio_inverted": (
        "double r = q > 0.0 ? p / q : INFINITY;",
        "double r = p > 0.0 ? q / p : INFINITY;"),
    "temperature_dropped_from_Z": (
        "z += exp(elem(L, dt, off + (size_t)v) / T - m);",
        "z += exp(elem(L, dt, off + (size_t)v) - m);"),
    "last_rejection_instead_of_first": (
        "        m = k;\n        break;\n      }\n    }\n    accept_len[b] = m;\n    for (int k = 0; k < m; ++k) out[k] = x[(size_t)b * K + k];\n\n",
        "        m = k;\n      }\n    }\n    accept_len[b] = m;\n    for (int k = 0; k < m; ++k) out[k] = x[(size_t)b * K + k];\n\n"),
    "accept_with_le": ("if (!(u < r))", "if (!(u <= r))"),
    "cdf_with_ge": ("if (C > t)", "if (C >= t)"),
    "bonus_from_previous_row": (
        "size_t offp = ((size_t)b * (K + 1) + m) * (size_t)V;",
        "size_t offp = ((size_t)b * (K + 1) + (m == K ? K - 1 : m)) * (size_t)V;"),
    "px_with_draft_normaliser": (
        "xk, T, Mp[k], Zp[k]);", "xk, T, Mq[k], Zq[k]);"),
    "residual_not_normalised": ("double t = ur[b] * S,", "double t = ur[b],"),
    "greedy_tie_to_highest": ("else if (s > bv)", "else if (s >= bv)"),
    "greedy_emits_draft_at_m": ("out[m] = a[m];", "out[m] = m < K ? x[(size_t)b * K + m] : a[m];"),
    "tree_compares_own_argmax": (
        "if (nd == -1 || tk[nd] != a[row[t - 1]]) break;", "if (nd == -1 || tk[nd] != a[nd]) break;"),
    "tree_last_best_row": ("if (L > bestL) {", "if (L >= bestL) {"),
    "tree_bonus_from_parent": ("out[bestL] = a[row[bestL]];", "out[bestL] = a[row[bestL > 0 ? bestL - 1 : 0]];"),
    "tree_subtree_boundary": ("(row[1] <= n1 ? 1 : 2)", "(row[1] < n1 ? 1 : 2)"),
    "confidence_wrong_count": ("s2 = n2 > 0 ? s2 / n2 : -INFINITY;", "s2 = n2 > 0 ? s2 / n1 : -INFINITY;"),
    "confidence_root_included": ("for (int i = 1; i <= n1; ++i) s1 +=", "for (int i = 0; i <= n1; ++i) s1 +="),
    "kv_dest_off_by_one": ("memcpy(plane + (size_t)(b0 + t) * (size_t)ss", "memcpy(plane + (size_t)(b0 + t + 1) * (size_t)ss"),
    "kv_length_short": ("new_len[b] = b0 + L + 1;", "new_len[b] = b0 + L;"),
    "kv_last_row_kept": (
        "for (int t = 0; t <= L; ++t)\n        memcpy(plane", "for (int t = 0; t < L; ++t)\n        memcpy(plane"),
    "kv_first_plane_only": ("for (int p = 0; p < P; ++p) {", "for (int p = 0; p < 1; ++p) {"),
    "kv_batch_stride_ignored": ("(size_t)b * (size_t)sb) * (size_t)es", "(size_t)b * (size_t)ss) * (size_t)es"),
    "kv_repeated_node_allowed": ("if (pr[t] <= pr[t - 1]) ok = 0;", "if (pr[t] < pr[t - 1]) ok = 0;"),
    "entropy_sign": ("e[i] = log(Z) - y / Z;", "e[i] = log(Z) + y / Z;"),
    "entropy_temperature_dropped": ("double d = elem(Ld, dt, off + (size_t)v) / T - M;",
                                    "double d = elem(Ld, dt, off + (size_t)v) - M;"),
    "entropy_higher_wins": ("choice[b] = s2 < s1 ? 2 : 1;", "choice[b] = s2 > s1 ? 2 : 1;"),
    "entropy_root_included": ("for (int i = 1; i <= n1; ++i) s1 += e[i];", "for (int i = 0; i <= n1; ++i) s1 += e[i];"),
    "entropy_empty_tree_zero": ("s2 = n2 > 0 ? s2 / n2 : INFINITY;", "s2 = n2 > 0 ? s2 / n2 : 0.0;"),
    "warped_topk_off_by_one": ("if (top_k > 0 && top_k < V) tk = tmp[top_k - 1].s;",
                               "if (top_k > 0 && top_k < V) tk = tmp[top_k].s;"),
    "warped_topp_drops_crossing_token": ("if (!(cum < cut)) break;", "if (!(cum + g < cut)) break;"),
    "warped_topp_on_full_mass": ("const double target = top_p * Zk,", "const double target = top_p * Z,"),
    "warped_not_renormalised": ("? out[v] / Zw : 0.0;", "? out[v] / Z : 0.0;"),
    "warped_residual_unwarped_draft": (
        "if (residual) warped_row(Lq, dt, ((size_t)b * K + m) * (size_t)V, V, T, top_k, top_p, near_p, wq, tmp, &near);",
        "if (residual) warped_row(Lq, dt, ((size_t)b * K + m) * (size_t)V, V, T, 0, 1.0, near_p, wq, tmp, &near);"),
    "valid_accept_window_ignored": ("if (!(fmax(0.0, u[k] - win) < r[k])) return 0;", "if (!(u[k] < r[k])) return 0;"),
    "valid_reject_window_ignored": ("if (m < K && !(fmin(u[m] + win, kOneMinus) >= r[m])) return 0;",
                                    "if (m < K && !(u[m] >= r[m])) return 0;"),
    "valid_draw_interval_shifted": ("if (Cprev <= hi * S && C > lo * S) return 1;",
                                    "if (C <= hi * S && C > lo * S) return 1;"),
    "valid_prefix_unchecked": ("    if (out[k] != x[k]) return 0;", "    if (0) return 0;"),
    "valid_warped_no_alternative_cuts": ("nalt[sl] = nn ? 2 + nn : 1;", "nalt[sl] = 1;"),
    "valid_warped_keep_all_cut_missing": ("if (alt == 1) cut = target + band;", "if (alt == 1) cut = target;"),
    "valid_warped_gives_up_past_cap": ("    const int exhaustive = combos <= 4096;",
                                       "    if (combos > 4096) {\n      valid[b] = 0;\n      continue;\n    }\n"
                                       "    const int exhaustive = 1;"),
    "pflag_window_halved": ("pf += fmin(w / S, 2.0 * near);", "pf += fmin(w / S, near);"),
    "expand_ties_to_higher_node": ("if (x->f != y->f) return x->f < y->f ? -1 : 1;",
                                   "if (x->f != y->f) return x->f > y->f ? -1 : 1;"),
    "expand_cumulative_dropped": ("cand[n].s = logc[(size_t)b * F + f] + (", "cand[n].s = 0.0 + ("),
    "expand_temperature_dropped": ("+ (elem(Ld, dt, off + (size_t)v) / T - Mx - lz);",
                                   "+ (elem(Ld, dt, off + (size_t)v) - Mx - lz);"),
    "expand_unnormalised": ("+ (elem(Ld, dt, off + (size_t)v) / T - Mx - lz);",
                            "+ (elem(Ld, dt, off + (size_t)v) / T - Mx);"),
    "kv_in_place_from_last_row": (
        "      for (int t = 0; t <= L; ++t) {\n        int src = pr ? pr[t] : t;\n        memcpy(tmp + (size_t)t * rowb,",
        "      for (int t = L; t >= 0; --t) {\n        int src = pr ? pr[t] : t;\n"
        "        memmove(plane + (size_t)(b0 + t) * (size_t)ss * (size_t)es,"
        " plane + (size_t)(b0 + src) * (size_t)ss * (size_t)es, rowb);\n        memcpy(tmp + (size_t)t * rowb,"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(oracle._SRC).read()
    assert old in src, f"mutation anchor for {name} no longer in oracle.c"
    mutated = tmp_path / "oracle_mut.c"
    # a trailing "*" in the name applies the edit to every occurrence
    mutated.write_text(src.replace(old, new) if name.endswith("*") else src.replace(old, new, 1))
    lib = oracle.load(oracle.build(str(mutated), str(tmp_path / "liboracle_mut.so"), force=True))
    caught = []
    for pin_name, pin in P.ALL_PINS:
        try:
            pin(lib)
        except AssertionError:
            caught.append(pin_name)
            break
    assert caught, f"no pin caught mutation {name}"
