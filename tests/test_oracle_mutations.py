"""Plant plausible mistakes in the oracle (CPU only) and check a pin catches each.

A pin set that passes a broken oracle proves nothing; each mutant below is a
mistake someone could make while writing the oracle from the pages."""
from dataclasses import replace

import numpy as np
import pytest

from oracle import moe_oracle as orc
from tests import oracle_pins as pins

_real_route = orc.route
_real_swiglu = orc.swiglu_ffn
_real_experts_forward = orc.experts_forward
_real_permutation = orc.permutation
_real_combine = orc.combine
_real_balance = orc.balance_update
_real_e4m3 = orc.e4m3_round
_real_quant = orc.quantize_fp8_blocks


def _route_ties_high(logits, bias, cfg):
    # evaluate on reversed expert ids: equal scores now go to the higher index
    rb = None if bias is None else bias[::-1].copy()
    r = _real_route(logits[:, ::-1].copy(), rb, cfg)
    r.idx = cfg.E - 1 - r.idx
    return r


def _route_biased_gates(logits, bias, cfg):
    r = _real_route(logits, bias, cfg)
    rows = np.arange(r.idx.shape[0])[:, None]
    g = r.sel32.astype(np.float64)[rows, r.idx]
    if cfg.norm_topk:
        g = g / g.sum(1, keepdims=True)
    r.gates = g * cfg.routed_scaling_factor
    return r


def _route_no_renorm(logits, bias, cfg):
    return _real_route(logits, bias, replace(cfg, norm_topk=False))


def _route_softmax_over_selected(logits, bias, cfg):
    r = _real_route(logits, bias, cfg)
    rows = np.arange(r.idx.shape[0])[:, None]
    sel = np.asarray(logits)[rows, r.idx]
    e = np.exp(sel - sel.max(1, keepdims=True))
    r.gates = e / e.sum(1, keepdims=True) * cfg.routed_scaling_factor
    return r


def _route_strided_groups(logits, bias, cfg):
    # groups taken as e % n_group instead of contiguous blocks
    E, G = cfg.E, cfg.n_group
    perm = np.arange(E).reshape(E // G, G).T.ravel()
    rb = None if bias is None else bias[perm].copy()
    r = _real_route(np.asarray(logits)[:, perm], rb, cfg)
    r.idx = perm[r.idx]
    return r


def _group_score_sum_all(sel32, cfg):
    T, E = sel32.shape
    return sel32.reshape(T, cfg.n_group, E // cfg.n_group).sum(axis=2).astype(np.float32)


def _swiglu_swapped(u, w1, w3, w2):
    return _real_swiglu(u, w3, w1, w2)


def _swiglu_no_gate(u, w1, w3, w2):
    u = np.asarray(u, np.float64)
    return (orc.silu(u @ np.asarray(w1).T)) @ np.asarray(w2).T


def _experts_no_shared(x, idx, gates, expert, shared, E):
    return _real_experts_forward(x, idx, gates, expert, None, E)


def _experts_with_residual(x, idx, gates, expert, shared, E):
    return _real_experts_forward(x, idx, gates, expert, shared, E) + np.asarray(x, np.float64)


def _permutation_reversed(idx, E):
    counts, offsets, row2tok, tok2row = _real_permutation(idx, E)
    row2tok = row2tok.copy()
    for e in range(E):
        a, b = offsets[e], offsets[e + 1]
        row2tok[a:b] = row2tok[a:b][::-1]
    return counts, offsets, row2tok, tok2row


def _combine_slot_swap(y_rows, y_shared, tok2row, gates):
    return _real_combine(y_rows, y_shared, tok2row, gates[:, ::-1])


def _balance_wrong_direction(counts, bias32, gamma):
    return _real_balance(counts, bias32, -gamma)


def _balance_biased_std(counts, bias32, gamma):
    nb, st = _real_balance(counts, bias32, gamma)
    E = len(counts)
    st = st.copy()
    st[0] *= ((E - 1) / E) ** 0.5
    return nb, st


def _balance_mean_counts_as_over(counts, bias32, gamma):
    # an expert exactly at the mean treated as overloaded
    c = np.asarray(counts, np.int64)
    nb, st = _real_balance(counts, bias32, gamma)
    at_mean = c * c.size == c.sum()
    nb = nb.copy()
    nb[at_mean] = (np.asarray(bias32, np.float32)[at_mean] - np.float32(gamma)).astype(np.float32)
    return nb, st


def _e4m3_ties_away(v):
    # round half away from zero instead of to even
    v = np.asarray(v, np.float64)
    a = np.abs(v)
    _, x = np.frexp(np.where(a > 0, a, 1.0))
    step = np.ldexp(1.0, (np.maximum(x - 1, -6) - 3).astype(np.int64))
    return np.copysign(np.minimum(np.floor(a / step + 0.5) * step, 448.0), v)


def _quant_scale_from_127(w):
    # the listing's integer range taken literally: scale = 2^ceil(log2(amax / 127))
    w = np.asarray(w, np.float64)
    rows, cols = w.shape
    b = w.reshape(rows, cols // 64, 64)
    amax = np.abs(b).max(2)
    e = np.where(amax > 0, np.ceil(np.log2(np.where(amax > 0, amax, 1.0) / 127.0)), 0.0)
    s = np.exp2(e)
    return orc.e4m3_round(b / s[..., None]).reshape(rows, cols), s


def _silu_grad_sigma_only(z):
    return 1.0 / (1.0 + np.exp(-z))


def _swiglu_backward_w1_w3_swapped(u, w1, w3, w2, dy):
    return _ORIG_SWIGLU_BACKWARD(u, w3, w1, w2, dy)


def _gate_backward_no_renorm_term(dg, s, idx, cfg):
    import dataclasses
    return _ORIG_GATE_BACKWARD(dg, s, idx, dataclasses.replace(cfg, norm_topk=False)) if cfg.norm_topk else \
        _ORIG_GATE_BACKWARD(dg, s, idx, cfg)


def _gate_backward_softmax_diag(dg, s, idx, cfg):
    import dataclasses
    if cfg.score_fn != "softmax":
        return _ORIG_GATE_BACKWARD(dg, s, idx, cfg)
    # sigmoid-style diagonal Jacobian applied to softmax affinities
    return _ORIG_GATE_BACKWARD(dg, s, idx, dataclasses.replace(cfg, score_fn="sigmoid"))


def _swiglu_backward_dw2_from_gate(u, w1, w3, w2, dy):
    du, g1, g3, g2 = _ORIG_SWIGLU_BACKWARD(u, w1, w3, w2, dy)
    # dW2 from silu(W1 u) alone (the up projection dropped)
    a = np.asarray(u, np.float64) @ np.asarray(w1, np.float64).T
    return du, g1, g3, np.asarray(dy, np.float64).T @ orc.silu(a)


def _expert_backward_ungated(x, dout, idx, gates, e, w1e, w3e, w2e):
    # the expert's rows back-propagate dout itself, not g * dout
    return _ORIG_EXPERT_BACKWARD(x, dout, idx, np.ones_like(np.asarray(gates, np.float64)), e, w1e, w3e, w2e)


def _expert_backward_dg_unsummed(x, dout, idx, gates, e, w1e, w3e, w2e):
    tok, slot, dg, du, g1, g3, g2 = _ORIG_EXPERT_BACKWARD(x, dout, idx, gates, e, w1e, w3e, w2e)
    # dL/dg from the first output column only instead of <dout_t, y_t>
    y = orc.swiglu_ffn(np.asarray(x, np.float64)[tok], w1e, w3e, w2e)
    return tok, slot, np.asarray(dout, np.float64)[tok, 0] * y[:, 0], du, g1, g3, g2


def _valid_selection_variant(old_threshold=False, group_tol_sign=1.0, require_groups=True, expert_tol_sign=1.0):
    """is_valid_selection with one planted mistake (flags name it)."""
    from itertools import combinations

    def valid(idx_row, sel32_row, cfg):
        sel = np.asarray(sel32_row, np.float64)
        picked = np.asarray(list(idx_row), np.int64)
        if len(set(picked.tolist())) != cfg.k:
            return False
        tol = orc.NEAR_TIE_REL * np.abs(sel).max()
        if cfg.topk_method == "group_limited_greedy":
            gsize = cfg.E // cfg.n_group
            g = orc._group_scores64(sel[None, :], cfg)[0]
            need = set((picked // gsize).tolist())
            if old_threshold:
                # groups judged against the topk_group-th best group, padded with the best others
                if len(need) > cfg.topk_group:
                    return False
                thresh = np.sort(g)[::-1][cfg.topk_group - 1]
                if any(g[x] < thresh - tol for x in need):
                    return False
                kept = set(need)
                for gg in np.argsort(-g, kind="stable"):
                    if len(kept) >= cfg.topk_group:
                        break
                    kept.add(int(gg))
                cands = [np.array([(e // gsize) in kept for e in range(cfg.E)])]
            else:
                cands = []
                for K in combinations(range(cfg.n_group), cfg.topk_group):
                    if require_groups and not need <= set(K):
                        continue
                    in_k = np.zeros(cfg.n_group, bool)
                    in_k[list(K)] = True
                    if (~in_k).any() and g[~in_k].max() > g[in_k].min() + group_tol_sign * tol:
                        continue
                    cands.append(np.repeat(in_k, gsize))
        else:
            cands = [np.ones(cfg.E, bool)]
        worst = sel[picked].min()
        for elig in cands:
            others = np.where(elig, sel, -np.inf)
            others[picked] = -np.inf
            if others.max() <= worst + expert_tol_sign * tol:
                return True
        return False
    return valid


_valid_old_threshold_rule = _valid_selection_variant(old_threshold=True)
_valid_old_threshold_rule.__name__ = "_valid_old_threshold_rule"
_valid_group_tol_reversed = _valid_selection_variant(group_tol_sign=-1.0)
_valid_group_tol_reversed.__name__ = "_valid_group_tol_reversed"
_valid_groups_not_required = _valid_selection_variant(require_groups=False)
_valid_groups_not_required.__name__ = "_valid_groups_not_required"
_valid_expert_tol_reversed = _valid_selection_variant(expert_tol_sign=-1.0)
_valid_expert_tol_reversed.__name__ = "_valid_expert_tol_reversed"


def _near_ties_variant(group_offset=0, absolute=False, group_gap=True):
    def near(sel64, elig, cfg):
        T, E = sel64.shape
        scale = 1.0 if absolute else np.abs(sel64).max(axis=1)
        out = np.zeros(T, bool)
        if cfg.k < E:
            e64 = np.where(elig, sel64, -np.inf)
            desc = -np.sort(-e64, axis=1)
            gap = np.where(elig.sum(axis=1) > cfg.k, desc[:, cfg.k - 1] - desc[:, cfg.k], np.inf)
            out |= gap < orc.NEAR_TIE_REL * scale
        if group_gap and cfg.topk_method == "group_limited_greedy" and cfg.topk_group < cfg.n_group:
            g64 = -np.sort(-orc._group_scores64(sel64, cfg), axis=1)
            j = min(cfg.topk_group - 1 + group_offset, cfg.n_group - 2)
            out |= g64[:, j] - g64[:, j + 1] < orc.NEAR_TIE_REL * scale
        return out
    return near


_near_group_gap_off_by_one = _near_ties_variant(group_offset=1)
_near_group_gap_off_by_one.__name__ = "_near_group_gap_off_by_one"
_near_absolute_tolerance = _near_ties_variant(absolute=True)
_near_absolute_tolerance.__name__ = "_near_absolute_tolerance"
_near_no_group_gap = _near_ties_variant(group_gap=False)
_near_no_group_gap.__name__ = "_near_no_group_gap"


def _rel_err_mean(got, ref):
    ref, got = np.asarray(ref, np.float64), np.asarray(got, np.float64)
    return float(np.mean(np.abs(got - ref))) / float(np.sqrt(np.mean(ref * ref)))


def _rel_err_over_max_ref(got, ref):
    ref, got = np.asarray(ref, np.float64), np.asarray(got, np.float64)
    return float(np.max(np.abs(got - ref))) / float(np.max(np.abs(ref)))


def _rel_err_over_mean_abs(got, ref):
    ref, got = np.asarray(ref, np.float64), np.asarray(got, np.float64)
    return float(np.max(np.abs(got - ref))) / float(np.mean(np.abs(ref)))


def _rel_err_no_sqrt(got, ref):
    ref, got = np.asarray(ref, np.float64), np.asarray(got, np.float64)
    return float(np.max(np.abs(got - ref))) / float(np.mean(ref * ref))


_ORIG_SWIGLU_BACKWARD = orc.swiglu_backward
_ORIG_GATE_BACKWARD = orc.gate_backward
_ORIG_EXPERT_BACKWARD = orc.expert_backward


MUTANTS = [
    ("route", _route_ties_high, pins.pin_brute_force_selection),
    ("route", _route_biased_gates, pins.pin_bias_only_steers_selection),
    ("route", _route_no_renorm, pins.pin_invariants),
    ("route", _route_softmax_over_selected, pins.pin_top1),
    ("route", _route_strided_groups, pins.pin_brute_force_selection),
    ("_group_scores32", _group_score_sum_all, pins.pin_brute_force_selection),
    ("swiglu_ffn", _swiglu_swapped, pins.pin_single_expert),
    ("swiglu_ffn", _swiglu_no_gate, pins.pin_dense_einsum),
    ("experts_forward", _experts_no_shared, pins.pin_zero_gates_give_shared),
    ("experts_forward", _experts_with_residual, pins.pin_zero_gates_give_shared),
    ("permutation", _permutation_reversed, pins.pin_permutation),
    ("combine", _combine_slot_swap, pins.pin_combine),
    ("balance_update", _balance_wrong_direction, pins.pin_balance_update),
    ("balance_update", _balance_biased_std, pins.pin_balance_update),
    ("balance_update", _balance_mean_counts_as_over, pins.pin_balance_update),
    ("e4m3_round", _e4m3_ties_away, pins.pin_fp8_quantization),
    ("quantize_fp8_blocks", _quant_scale_from_127, pins.pin_fp8_quantization),
    ("silu_grad", _silu_grad_sigma_only, pins.pin_backward_finite_differences),
    ("swiglu_backward", _swiglu_backward_w1_w3_swapped, pins.pin_backward_finite_differences),
    ("gate_backward", _gate_backward_no_renorm_term, pins.pin_backward_finite_differences),
    ("gate_backward", _gate_backward_softmax_diag, pins.pin_backward_finite_differences),
    ("swiglu_backward", _swiglu_backward_dw2_from_gate, pins.pin_backward_homogeneity),
    ("expert_backward", _expert_backward_ungated, pins.pin_backward_finite_differences),
    ("expert_backward", _expert_backward_dg_unsummed, pins.pin_backward_finite_differences),
    ("gate_backward", _gate_backward_no_renorm_term, pins.pin_backward_homogeneity),
    ("is_valid_selection", _valid_old_threshold_rule, pins.pin_valid_selection_brute_force),
    ("is_valid_selection", _valid_group_tol_reversed, pins.pin_valid_selection_brute_force),
    ("is_valid_selection", _valid_groups_not_required, pins.pin_valid_selection_brute_force),
    ("is_valid_selection", _valid_expert_tol_reversed, pins.pin_valid_selection_brute_force),
    ("near_ties", _near_group_gap_off_by_one, pins.pin_group_near_tie_gap),
    ("near_ties", _near_absolute_tolerance, pins.pin_group_near_tie_gap),
    ("near_ties", _near_no_group_gap, pins.pin_group_near_tie_gap),
    ("relative_error", _rel_err_mean, pins.pin_relative_error),
    ("relative_error", _rel_err_over_max_ref, pins.pin_relative_error),
    ("relative_error", _rel_err_over_mean_abs, pins.pin_relative_error),
    ("relative_error", _rel_err_no_sqrt, pins.pin_relative_error),
]


@pytest.mark.parametrize("attr,mutant,pin", MUTANTS, ids=[m[1].__name__ for m in MUTANTS])
def test_pin_catches_mutant(monkeypatch, attr, mutant, pin):
    monkeypatch.setattr(orc, attr, mutant)
    with pytest.raises(AssertionError):
        pin()
