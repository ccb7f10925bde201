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


_ORIG_SWIGLU_BACKWARD = orc.swiglu_backward
_ORIG_GATE_BACKWARD = orc.gate_backward


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
    ("gate_backward", _gate_backward_no_renorm_term, pins.pin_backward_homogeneity),
]


@pytest.mark.parametrize("attr,mutant,pin", MUTANTS, ids=[m[1].__name__ for m in MUTANTS])
def test_pin_catches_mutant(monkeypatch, attr, mutant, pin):
    monkeypatch.setattr(orc, attr, mutant)
    with pytest.raises(AssertionError):
        pin()
