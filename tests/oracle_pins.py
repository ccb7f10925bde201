"""Checks that pin the fp64 oracle to facts outside itself.

Every check raises AssertionError when the oracle disagrees with:
  * brute-force enumeration of expert subsets and group subsets on tiny inputs,
    with exact rational sums (Fractions) of the float32 decision values;
  * invariants the method guarantees (k largest affinities, kept groups,
    sum of counts, renormalised gate sum, zero gates -> shared FFN only);
  * special cases that reduce to textbook forms written here with torch:
    E=1/k=1 -> plain SwiGLU sum, k=E -> the dense einsum gate fusion of the
    intelliparadigm.com page (section 3.3.3), k=1 -> the Top-1 MoE of the
    Tencent Cloud page, greedy == torch.topk on float64 scores;
  * symmetries: expert relabelling, token independence, linearity in W2;
  * the balancing step (bias +/- gamma, load statistics) against hand-worked
    counts, closed forms and exact rational rounding bounds;
  * the FP8 block quantisation against torch's float8_e4m3fn conversion, the
    minimality of the power-of-two scale, the e4m3 error bound and exactness
    in bf16.

The independent pieces (softmax via scipy, SwiGLU via torch.nn.functional)
never call the oracle's own helpers.  ``tests/test_oracle_mutations.py``
plants plausible mistakes in the oracle and checks that these pins catch them.
"""
from dataclasses import replace
from fractions import Fraction
from itertools import combinations
import math

import numpy as np
import scipy.special
import torch
import torch.nn.functional as F

from oracle import moe_oracle as orc


# ------------------------------------------------------------------ helpers

def _rng(seed):
    return np.random.default_rng(seed)


def independent_sel32(logits, score_fn, bias):
    if score_fn == "softmax":
        s = scipy.special.softmax(logits, axis=1)
    else:
        s = scipy.special.expit(logits)
    s32 = s.astype(np.float32)
    if bias is not None:
        s32 = (s32 + bias.astype(np.float32)[None, :]).astype(np.float32)
    return s, s32


def torch_swiglu(x, w1, w3, w2):
    x, w1, w3, w2 = (torch.as_tensor(a, dtype=torch.float64) for a in (x, w1, w3, w2))
    return (F.silu(x @ w1.T) * (x @ w3.T)) @ w2.T


def _brute_group_score(vals32, score, m):
    if score == "max":
        return Fraction(float(max(vals32)))
    best = max(sum(Fraction(float(v)) for v in c) for c in combinations(vals32, m))
    return Fraction(float(np.float32(float(best))))   # the float32 rounding of the exact best sum


def brute_force_choice(sel_row, cfg):
    """Best k-subset (max exact sum, then lexicographically smallest) inside the
    best topk_group-subset of groups (same rule)."""
    E = sel_row.size
    if cfg.topk_method == "group_limited_greedy":
        gs = E // cfg.n_group
        gsc = [_brute_group_score(sel_row[g * gs:(g + 1) * gs], cfg.group_score, cfg.group_top)
               for g in range(cfg.n_group)]
        best = None
        for c in combinations(range(cfg.n_group), cfg.topk_group):
            key = (sum(gsc[g] for g in c), tuple(-g for g in c))
            if best is None or key > best[0]:
                best = (key, c)
        elig = [e for e in range(E) if (e // gs) in best[1]]
    else:
        elig = list(range(E))
    best = None
    for c in combinations(elig, cfg.k):
        key = (sum(Fraction(float(sel_row[e])) for e in c), tuple(-e for e in c))
        if best is None or key > best[0]:
            best = (key, c)
    return set(best[1])


def small_layer(seed, T, d, E, I, k, n_shared, **cfgkw):
    r = _rng(seed)
    cfg = orc.OracleConfig(T=T, d=d, E=E, I=I, k=k, n_shared=n_shared, **cfgkw)
    x = r.standard_normal((T, d))
    wg = r.uniform(-1, 1, (E, d)) / np.sqrt(d)
    w1 = r.uniform(-1, 1, (E, I, d)) / np.sqrt(d)
    w3 = r.uniform(-1, 1, (E, I, d)) / np.sqrt(d)
    w2 = r.uniform(-1, 1, (E, d, I)) / np.sqrt(I)
    Is = max(1, n_shared) * I
    shared = (r.uniform(-1, 1, (Is, d)) / np.sqrt(d), r.uniform(-1, 1, (Is, d)) / np.sqrt(d),
              r.uniform(-1, 1, (d, Is)) / np.sqrt(Is)) if n_shared > 0 else None
    return cfg, x, wg, (w1, w3, w2), shared


SELECTION_CASES = [
    dict(E=8, k=2, score_fn="softmax", topk_method="greedy"),
    dict(E=12, k=4, score_fn="softmax", topk_method="greedy"),
    dict(E=16, k=3, score_fn="sigmoid", topk_method="greedy", bias=True),
    dict(E=8, k=2, score_fn="softmax", topk_method="group_limited_greedy", n_group=4, topk_group=2,
         group_score="max"),
    dict(E=16, k=4, score_fn="sigmoid", topk_method="group_limited_greedy", n_group=4, topk_group=2,
         group_score="sum_top", group_top=2, bias=True),
    dict(E=12, k=3, score_fn="softmax", topk_method="group_limited_greedy", n_group=2, topk_group=1,
         group_score="max"),
    dict(E=16, k=1, score_fn="sigmoid", topk_method="group_limited_greedy", n_group=2, topk_group=1,
         group_score="sum_top", group_top=2, bias=True),
]


# --------------------------------------------------------------------- pins

def pin_brute_force_selection(o=orc, tokens=24):
    for ci, case in enumerate(SELECTION_CASES):
        case = dict(case)
        use_bias = case.pop("bias", False)
        E = case["E"]
        cfg = orc.OracleConfig(T=tokens, d=1, I=1, n_shared=0, **case)
        r = _rng(100 + ci)
        # coarse logits make exact float32 ties common, exercising the tie rule
        logits = r.integers(-3, 4, size=(tokens, E)).astype(np.float64) * 0.5
        logits[: tokens // 2] += r.standard_normal((tokens // 2, E))
        bias = (r.integers(-2, 3, size=E) * 0.05).astype(np.float32) if use_bias else None
        s, sel32 = independent_sel32(logits, cfg.score_fn, bias)
        got = o.route(logits, bias, cfg)
        for t in range(tokens):
            want = brute_force_choice(sel32[t], cfg)
            assert set(got.idx[t].tolist()) == want, (ci, t, got.idx[t], sorted(want))
            keys = [(-float(sel32[t, e]), e) for e in got.idx[t]]
            assert keys == sorted(keys), ("order", ci, t, got.idx[t])


def pin_greedy_is_torch_topk(o=orc):
    r = _rng(7)
    for E, k, fn in [(12, 4, "softmax"), (64, 6, "softmax"), (256, 8, "sigmoid")]:
        logits = r.standard_normal((50, E))
        cfg = orc.OracleConfig(T=50, d=1, E=E, I=1, k=k, n_shared=0, score_fn=fn)
        s = torch.softmax(torch.tensor(logits), dim=1) if fn == "softmax" else torch.sigmoid(torch.tensor(logits))
        want = torch.topk(s, k, dim=1).indices.numpy()
        got = o.route(logits, None, cfg).idx
        for t in range(50):
            assert set(got[t].tolist()) == set(want[t].tolist()), (E, t)


def pin_invariants(o=orc):
    r = _rng(11)
    T = 40
    for case in [dict(E=12, k=4, score_fn="softmax"),
                 dict(E=32, k=6, score_fn="softmax", topk_method="group_limited_greedy", n_group=8,
                      topk_group=3, group_score="max", routed_scaling_factor=16.0),
                 dict(E=32, k=8, score_fn="sigmoid", topk_method="group_limited_greedy", n_group=8,
                      topk_group=4, group_score="sum_top", group_top=2, norm_topk=True,
                      routed_scaling_factor=2.5, bias=True)]:
        case = dict(case)
        use_bias = case.pop("bias", False)
        E, k = case["E"], case["k"]
        cfg = orc.OracleConfig(T=T, d=1, I=1, n_shared=0, **case)
        logits = r.standard_normal((T, E))
        bias = (r.standard_normal(E) * 0.1).astype(np.float32) if use_bias else None
        s, sel32 = independent_sel32(logits, cfg.score_fn, bias)
        got = o.route(logits, bias, cfg)
        # counts
        assert int(got.counts.sum()) == T * k
        assert np.array_equal(got.counts, np.bincount(got.idx.ravel(), minlength=E))
        # distinct experts per token
        assert all(len(set(row.tolist())) == k for row in got.idx)
        if cfg.topk_method == "group_limited_greedy":
            gsz = E // cfg.n_group
            st = torch.tensor(sel32.astype(np.float64)).view(T, cfg.n_group, gsz)
            gsc = st.max(-1).values if cfg.group_score == "max" else st.topk(cfg.group_top, -1).values.sum(-1)
            best = torch.topk(gsc, cfg.topk_group, dim=1).indices.numpy()
            for t in range(T):
                assert set((got.idx[t] // gsz).tolist()) <= set(best[t].tolist()), t
        elif bias is None:
            for t in range(T):
                assert np.allclose(np.sort(s[t, got.idx[t]]), np.sort(s[t])[-k:], rtol=0, atol=0)
        g = got.gates
        scale = cfg.routed_scaling_factor
        if cfg.norm_topk:
            assert np.allclose(g.sum(1), scale, rtol=1e-12, atol=0)
        else:
            assert (g <= scale * (1 + 1e-12)).all() and (g.sum(1) <= scale * (1 + 1e-12)).all()
        assert (g > 0).all()


def pin_bias_only_steers_selection(o=orc):
    """With a bias that does not change the chosen set, gates are unchanged."""
    r = _rng(12)
    T, E = 60, 32
    cfg = orc.OracleConfig(T=T, d=1, E=E, I=1, k=8, n_shared=0, score_fn="sigmoid",
                           topk_method="group_limited_greedy", n_group=8, topk_group=4,
                           group_score="sum_top", group_top=2, norm_topk=True, routed_scaling_factor=2.5)
    logits = r.standard_normal((T, E))
    bias = (r.standard_normal(E) * 0.02).astype(np.float32)
    a = o.route(logits, None, cfg)
    b = o.route(logits, bias, cfg)
    same = 0
    for t in range(T):
        if set(a.idx[t].tolist()) == set(b.idx[t].tolist()):
            same += 1
            ga = dict(zip(a.idx[t].tolist(), a.gates[t].tolist()))
            gb = dict(zip(b.idx[t].tolist(), b.gates[t].tolist()))
            for e in ga:
                assert abs(ga[e] - gb[e]) <= 1e-12 * abs(ga[e]), (t, e)
    assert same > T // 4


def pin_zero_gates_give_shared(o=orc):
    cfg, x, wg, (w1, w3, w2), shared = small_layer(3, 20, 16, 12, 8, 4, 2)
    cfg = replace(cfg, routed_scaling_factor=0.0)
    out, _ = o.moe_forward(x, wg, None, orc.stacked_experts(w1, w3, w2), shared, cfg)
    want = torch_swiglu(x, *shared).numpy()
    assert np.allclose(out, want, rtol=1e-12, atol=1e-14)


def pin_group1_is_greedy(o=orc):
    r = _rng(13)
    logits = r.standard_normal((30, 16))
    a = o.route(logits, None, orc.OracleConfig(T=30, d=1, E=16, I=1, k=4, n_shared=0))
    b = o.route(logits, None, orc.OracleConfig(T=30, d=1, E=16, I=1, k=4, n_shared=0,
                                               topk_method="group_limited_greedy", n_group=1, topk_group=1))
    assert np.array_equal(a.idx, b.idx) and np.allclose(a.gates, b.gates, rtol=0, atol=0)


def pin_single_expert(o=orc):
    cfg, x, wg, (w1, w3, w2), shared = small_layer(4, 10, 12, 1, 6, 1, 2)
    out, r = o.moe_forward(x, wg, None, orc.stacked_experts(w1, w3, w2), shared, cfg)
    want = (torch_swiglu(x, w1[0], w3[0], w2[0]) + torch_swiglu(x, *shared)).numpy()
    assert np.allclose(out, want, rtol=1e-12, atol=1e-13)


def pin_dense_einsum(o=orc):
    """k = E with softmax and scale 1: the dense gate fusion einsum('ted,te->td')."""
    cfg, x, wg, (w1, w3, w2), shared = small_layer(5, 12, 10, 6, 7, 6, 1)
    out, _ = o.moe_forward(x, wg, None, orc.stacked_experts(w1, w3, w2), shared, cfg)
    xt = torch.tensor(x)
    p = torch.softmax(xt @ torch.tensor(wg).T, dim=-1)
    ys = torch.stack([torch_swiglu(x, w1[e], w3[e], w2[e]) for e in range(6)], dim=1)   # [T,E,d]
    want = torch.einsum("ted,te->td", ys, p) + torch_swiglu(x, *shared)
    assert np.allclose(out, want.numpy(), rtol=1e-11, atol=1e-13)


def pin_top1(o=orc):
    """k = 1: out = p_max * E_argmax(x) (+ shared), the Top-1 gated MoE."""
    cfg, x, wg, (w1, w3, w2), shared = small_layer(6, 16, 8, 5, 4, 1, 1)
    out, _ = o.moe_forward(x, wg, None, orc.stacked_experts(w1, w3, w2), shared, cfg)
    xt = torch.tensor(x)
    p = torch.softmax(xt @ torch.tensor(wg).T, dim=-1)
    top_p, top_i = p.max(dim=-1)
    want = torch_swiglu(x, *shared).clone()
    for t in range(x.shape[0]):
        e = int(top_i[t])
        want[t] += top_p[t] * torch_swiglu(x[t:t + 1], w1[e], w3[e], w2[e])[0]
    assert np.allclose(out, want.numpy(), rtol=1e-12, atol=1e-13)


def pin_permutation(o=orc):
    r = _rng(14)
    T, E, k = 37, 9, 3
    idx = np.stack([r.choice(E, k, replace=False) for _ in range(T)])
    counts, offsets, row2tok, tok2row = o.permutation(idx, E)
    flat = idx.ravel()
    order = np.argsort(flat, kind="stable")        # sorted by expert, stable in (t, j)
    assert np.array_equal(row2tok, order // k)
    assert np.array_equal(counts, np.bincount(flat, minlength=E))
    assert offsets[0] == 0 and np.array_equal(np.diff(offsets), counts)
    inv = np.empty_like(order)
    inv[order] = np.arange(order.size)
    assert np.array_equal(tok2row.ravel(), inv)


def pin_symmetries(o=orc):
    cfg, x, wg, (w1, w3, w2), shared = small_layer(8, 24, 16, 8, 12, 3, 1,
                                                    score_fn="sigmoid", norm_topk=True,
                                                    routed_scaling_factor=2.5,
                                                    topk_method="group_limited_greedy", n_group=2,
                                                    topk_group=1, group_score="sum_top", group_top=2)
    bias = (_rng(9).standard_normal(8) * 0.1).astype(np.float32)
    out, r = o.moe_forward(x, wg, bias, orc.stacked_experts(w1, w3, w2), shared, cfg)
    # relabel experts inside each group (groups keep their members)
    perm = np.array([3, 1, 0, 2, 6, 7, 5, 4])
    out2, r2 = o.moe_forward(x, wg[perm], bias[perm], orc.stacked_experts(w1[perm], w3[perm], w2[perm]),
                             shared, cfg)
    assert np.allclose(out, out2, rtol=1e-12, atol=1e-13)
    for t in range(cfg.T):
        assert set(perm[r2.idx[t]].tolist()) == set(r.idx[t].tolist())   # new id e' is old id perm[e']
    # token independence
    sub = np.array([5, 0, 17, 3])
    out3, _ = o.moe_forward(x[sub], wg, bias, orc.stacked_experts(w1, w3, w2), shared, replace(cfg, T=4))
    assert np.allclose(out3, out[sub], rtol=1e-12, atol=1e-13)
    # linear in W2 and W2_s together
    out4, _ = o.moe_forward(x, wg, bias, orc.stacked_experts(w1, w3, 2.0 * w2),
                            (shared[0], shared[1], 2.0 * shared[2]), cfg)
    assert np.allclose(out4, 2.0 * out, rtol=1e-12, atol=1e-13)


def pin_combine(o=orc):
    """Rows in (token, slot) order: combine is the listing's
    (y.view(T,k,d) * w[..., None]).sum(1) + shared, written here with torch."""
    r = _rng(15)
    T, k, d = 11, 3, 5
    y = r.standard_normal((T * k, d))
    ys = r.standard_normal((T, d))
    g = r.uniform(0, 1, (T, k))
    tok2row = np.arange(T * k).reshape(T, k)
    want = (torch.tensor(y).view(T, k, d) * torch.tensor(g)[..., None]).sum(1) + torch.tensor(ys)
    assert np.allclose(o.combine(y, ys, tok2row, g), want.numpy(), rtol=1e-13, atol=1e-14)
    # any row order: permuting the stored rows together with tok2row changes nothing
    perm = r.permutation(T * k)
    inv = np.argsort(perm)
    assert np.allclose(o.combine(y[perm], ys, inv[tok2row], g), want.numpy(), rtol=1e-13, atol=1e-14)


def pin_balance_update(o=orc):
    """V3 page section 1.2: overloaded experts lose gamma, underloaded ones
    gain gamma, an expert at the mean keeps its bias; the Tencent Cloud
    listing's load = counts / sum and its (unbiased) std."""
    g = np.float32(0.001)
    # hand-worked: counts 3,1,2,2 (mean 2): signs -,+,0,0; loads .375,.125,.25,.25,
    # squared deviations 2 * (1/8)^2 = 1/32 over E-1 = 3 -> std = sqrt(1/96)
    b0 = np.array([0.0, 0.0, 0.5, -0.25], np.float32)
    nb, st = o.balance_update([3, 1, 2, 2], b0, g)
    assert nb.dtype == np.float32
    assert nb[2] == b0[2] and nb[3] == b0[3]
    assert nb[0] < b0[0] and nb[1] > b0[1]
    assert abs(st[0] - (1.0 / 96.0) ** 0.5) < 1e-15 and st[1] == 1.5 and st[2] == 0.5
    # uniform load: nothing moves, std 0, max = min = mean
    nb, st = o.balance_update([7] * 16, np.linspace(-1, 1, 16).astype(np.float32), g)
    assert np.array_equal(nb, np.linspace(-1, 1, 16).astype(np.float32))
    assert st[0] == 0.0 and st[1] == 1.0 and st[2] == 1.0
    # two experts a > b: std of (a, b)/(a+b) is |a-b| / (a+b) / sqrt(2)
    nb, st = o.balance_update([9, 3], np.zeros(2, np.float32), g)
    assert abs(st[0] - 6 / 12 / 2 ** 0.5) < 1e-15
    assert nb[0] == -g and nb[1] == g
    # random counts: each moved bias is b +/- gamma correctly rounded to float32
    r = _rng(21)
    for _ in range(20):
        E = int(r.integers(2, 257))
        c = r.integers(0, 50, E)
        b = (r.standard_normal(E) * 0.1).astype(np.float32)
        nb, st = o.balance_update(c, b, g)
        tot = int(c.sum())
        for e in range(E):
            want = Fraction(float(b[e]))
            if c[e] * E > tot:
                want -= Fraction(float(g))
            elif c[e] * E < tot:
                want += Fraction(float(g))
            else:
                assert nb[e] == b[e]
                continue
            got = Fraction(float(nb[e]))
            ulp = Fraction(float(np.spacing(np.float32(abs(float(nb[e]))))))
            assert abs(got - want) <= ulp / 2
        if tot:
            assert abs(st[1] - c.max() * E / tot) < 1e-12 and abs(st[2] - c.min() * E / tot) < 1e-12


def pin_fp8_quantization(o=orc):
    """intelliparadigm.com section 4: blocks of 64 values, one scale per block;
    e4m3 values (torch's float8_e4m3fn cast rounds to nearest even)."""
    r = _rng(31)
    # e4m3 rounding of values inside the format's range agrees with torch's cast
    v = np.concatenate([r.uniform(-448, 448, 4000), r.uniform(-1, 1, 4000), r.uniform(-2 ** -6, 2 ** -6, 4000),
                        np.array([0.0, 448.0, -448.0, 240.0, 232.0, 1.0625, 1.1875, 2 ** -10, 3 * 2 ** -10])])
    want = torch.tensor(v).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(o.e4m3_round(v), want)
    # blocks: bf16-valued weights of very different magnitudes, one zero block
    w = (r.standard_normal((6, 256)) * np.exp2(r.integers(-12, 4, (6, 1)))).astype(np.float32)
    w = torch.tensor(w).to(torch.bfloat16).double().numpy()
    w[2, 64:128] = 0.0
    q, s = o.quantize_fp8_blocks(w)
    assert q.shape == w.shape and s.shape == (6, 4)
    amax = np.abs(w.reshape(6, 4, 64)).max(2)
    nz = amax > 0
    # smallest power of two that brings the block inside +-448
    assert np.all(np.log2(s) == np.round(np.log2(s)))
    assert np.all(amax[nz] <= 448 * s[nz]) and np.all(amax[nz] > 224 * s[nz])
    assert s[2, 1] == 1.0 and np.all(q[2, 64:128] == 0)
    # every q is an e4m3 value, and the dequantized weight is a bf16 number
    assert np.array_equal(torch.tensor(q).to(torch.float8_e4m3fn).to(torch.float64).numpy(), q)
    wd = o.dequantize_fp8_blocks(q, s)
    assert np.array_equal(torch.tensor(wd).to(torch.bfloat16).double().numpy(), wd)
    # error: at most half an e4m3 spacing of the value's binade (3 mantissa bits)
    sc = np.repeat(s, 64, axis=1)
    a = np.abs(w) / sc
    _, x = np.frexp(np.where(a > 0, a, 1.0))
    half_step = np.ldexp(1.0, np.maximum(x - 1, -6) - 4) * sc
    assert np.all(np.abs(wd - w) <= half_step)
    # values already of the form e4m3 * 2^k come back unchanged
    exact = np.tile(np.array([448.0, -1.0, 0.125, 3.5] * 16), (1, 1)) * 2.0 ** -5
    assert np.array_equal(o.fp8_dequantized(exact), exact)


def _fd_case(seed, score_fn):
    """A small layer with well separated routing decisions."""
    g = _rng(seed)
    if score_fn == "softmax":
        cfg = orc.OracleConfig(T=6, d=10, E=6, I=5, k=2, n_shared=2, score_fn="softmax",
                               topk_method="greedy", routed_scaling_factor=1.0)
        bias = None
    else:
        cfg = orc.OracleConfig(T=6, d=10, E=8, I=5, k=3, n_shared=1, score_fn="sigmoid",
                               topk_method="group_limited_greedy", n_group=4, topk_group=2,
                               group_score="sum_top", group_top=2, norm_topk=True, routed_scaling_factor=2.5)
        bias = g.normal(0, 0.1, cfg.E).astype(np.float32)
    T, d, E, I, Is = cfg.T, cfg.d, cfg.E, cfg.I, cfg.n_shared * cfg.I
    p = {"x": g.normal(0, 1, (T, d)), "wg": g.normal(0, 0.5, (E, d)),
         "w1": g.normal(0, 0.4, (E, I, d)), "w3": g.normal(0, 0.4, (E, I, d)), "w2": g.normal(0, 0.4, (E, d, I)),
         "ws1": g.normal(0, 0.4, (Is, d)), "ws3": g.normal(0, 0.4, (Is, d)), "ws2": g.normal(0, 0.4, (d, Is))}
    dout = g.normal(0, 1, (T, d))
    return cfg, bias, p, dout


def _fd_loss(o, cfg, bias, p, dout):
    out, r = o.moe_forward(p["x"], p["wg"], bias, o.stacked_experts(p["w1"], p["w3"], p["w2"]),
                           (p["ws1"], p["ws3"], p["ws2"]), cfg)
    return float(np.sum(dout * out)), r.idx


def pin_backward_finite_differences(o=orc):
    """The oracle's gradients against central differences of the oracle's own
    fp64 forward, in random directions, for every parameter (softmax greedy
    router without renormalisation; sigmoid group-limited router with bias,
    renormalisation and scaling).  The routing decisions must not change within
    the step (checked)."""
    h = 1e-6
    for seed, score_fn in ((11, "softmax"), (12, "sigmoid")):
        cfg, bias, p, dout = _fd_case(seed, score_fn)
        grads = o.moe_backward(p["x"], p["wg"], bias, p["w1"], p["w3"], p["w2"], (p["ws1"], p["ws3"], p["ws2"]),
                               dout, cfg)
        _, idx0 = _fd_loss(o, cfg, bias, p, dout)
        g = _rng(seed + 100)
        for name, gname in (("x", "dx"), ("wg", "dwg"), ("w1", "dw1"), ("w3", "dw3"), ("w2", "dw2"),
                            ("ws1", "dws1"), ("ws3", "dws3"), ("ws2", "dws2")):
            v = g.normal(0, 1, p[name].shape)
            plus = dict(p, **{name: p[name] + h * v})
            minus = dict(p, **{name: p[name] - h * v})
            lp, ip = _fd_loss(o, cfg, bias, plus, dout)
            lm, im = _fd_loss(o, cfg, bias, minus, dout)
            assert np.array_equal(ip, idx0) and np.array_equal(im, idx0), (name, "routing changed")
            fd = (lp - lm) / (2 * h)
            an = float(np.sum(grads[gname] * v))
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (score_fn, name, fd, an)


def pin_backward_homogeneity(o=orc):
    """Exact identities of the gradient (Euler's theorem for homogeneous
    functions): the output is linear in (W2, Ws2) jointly and in (W3, Ws3)
    jointly, so sum <dW, W> over each pair equals <dout, out>; gradients are
    linear in dout; with k = 1 and renormalisation the gate is the constant
    routed_scaling_factor, so the router's gradient (dW_g) vanishes."""
    for seed, score_fn in ((21, "softmax"), (22, "sigmoid")):
        cfg, bias, p, dout = _fd_case(seed, score_fn)
        shared = (p["ws1"], p["ws3"], p["ws2"])
        gr = o.moe_backward(p["x"], p["wg"], bias, p["w1"], p["w3"], p["w2"], shared, dout, cfg)
        loss, _ = _fd_loss(o, cfg, bias, p, dout)
        e2 = float(np.sum(gr["dw2"] * p["w2"]) + np.sum(gr["dws2"] * p["ws2"]))
        e3 = float(np.sum(gr["dw3"] * p["w3"]) + np.sum(gr["dws3"] * p["ws3"]))
        assert abs(e2 - loss) <= 1e-10 * max(1.0, abs(loss)), (score_fn, e2, loss)
        assert abs(e3 - loss) <= 1e-10 * max(1.0, abs(loss)), (score_fn, e3, loss)
        g2 = o.moe_backward(p["x"], p["wg"], bias, p["w1"], p["w3"], p["w2"], shared, 2.0 * dout, cfg)
        for key in ("dx", "dwg", "dw1", "dw3", "dw2", "dws1", "dws3", "dws2"):
            assert np.allclose(g2[key], 2.0 * gr[key], rtol=1e-12, atol=1e-12), key
    import dataclasses
    cfg, bias, p, dout = _fd_case(23, "sigmoid")
    cfg1 = dataclasses.replace(cfg, k=1, topk_method="greedy", n_group=1, topk_group=1, norm_topk=True)
    g1 = o.moe_backward(p["x"], p["wg"], None, p["w1"], p["w3"], p["w2"], (p["ws1"], p["ws3"], p["ws2"]), dout,
                        cfg1)
    assert np.abs(g1["dwg"]).max() <= 1e-12 * max(1.0, np.abs(g1["dw1"]).max()), np.abs(g1["dwg"]).max()


# ------------------------------------------------- acceptance functions

def _perturbed_top(values, chosen, m, tol):
    """Whether the index set `chosen` (m of them) is a top-m set by sum, under
    some tie-break, after every chosen value is raised by tol/2 and every other
    value lowered by tol/2 (exact rationals throughout)."""
    v = [Fraction(x) + (tol / 2 if i in chosen else -tol / 2) for i, x in enumerate(values)]
    best = max(sum(v[i] for i in c) for c in combinations(range(len(v)), m))
    return sum(v[i] for i in chosen) == best


def brute_force_valid_sets(sel_row, cfg, tol):
    """Every k-subset of experts that the exact routing rule picks once the
    group scores and the expert scores are each moved by at most tol/2 (the
    two independently): a set K of topk_group groups that is a top set of the
    perturbed group scores, then k experts of K that are a top set of the
    perturbed expert scores.  Enumerates every K and every subset."""
    E = sel_row.size
    vals = [Fraction(float(v)) for v in sel_row]
    if cfg.topk_method == "group_limited_greedy":
        gs = E // cfg.n_group
        gscore = []
        for g in range(cfg.n_group):
            members = sorted(vals[g * gs:(g + 1) * gs], reverse=True)
            gscore.append(members[0] if cfg.group_score == "max" else sum(members[:cfg.group_top]))
        eligible_sets = [[e for e in range(E) if e // gs in K]
                         for K in combinations(range(cfg.n_group), cfg.topk_group)
                         if _perturbed_top(gscore, set(K), cfg.topk_group, tol)]
    else:
        gscore = []
        eligible_sets = [list(range(E))]
    valid = set()
    for elig in eligible_sets:
        ev = [vals[e] for e in elig]
        for S in combinations(range(len(elig)), cfg.k):
            if _perturbed_top(ev, set(S), cfg.k, tol):
                valid.add(frozenset(elig[i] for i in S))
    return valid, gscore


def _clear_of_boundary(vals, tol):
    """No two values differ by tol to within 2 % (so float rounding of tol
    cannot change a decision the test relies on)."""
    for a, b in combinations(vals, 2):
        if abs(abs(a - b) - tol) < tol / 50:
            return False
    return True


VALID_CASES = [
    dict(E=8, k=2, topk_method="group_limited_greedy", n_group=4, topk_group=2, group_score="max"),
    dict(E=8, k=3, topk_method="group_limited_greedy", n_group=4, topk_group=2, group_score="sum_top",
         group_top=2),
    dict(E=12, k=3, topk_method="group_limited_greedy", n_group=4, topk_group=2, group_score="max"),
    dict(E=12, k=2, topk_method="group_limited_greedy", n_group=4, topk_group=3, group_score="sum_top",
         group_top=2),
    dict(E=8, k=3, topk_method="greedy"),
]


def pin_valid_selection_brute_force(o=orc, tokens=40):
    """is_valid_selection (the acceptance of the other side's choice on a
    near-tie token) against brute-force enumeration: on tokens whose scores
    crowd within a few tolerances of each other, every k-subset of experts is
    accepted exactly when some perturbation of the scores by at most half the
    tolerance makes the exact rule pick it."""
    u = orc.NEAR_TIE_REL                      # tolerance per unit of the token's largest |score| (1.0 here)
    deficits = np.array([0.0, 0.0, 0.3, 0.7, 1.6, 2.5, 4.0, 40.0]) * u
    n_multi = 0
    for ci, case in enumerate(VALID_CASES):
        cfg = orc.OracleConfig(T=1, d=1, I=1, n_shared=0, score_fn="sigmoid", **case)
        r = _rng(300 + ci)
        kept_tokens = 0
        for _ in range(tokens * 4):
            base = r.choice([0.9, 0.8, 0.5], size=cfg.E, p=[0.5, 0.3, 0.2])
            sel = (base - r.choice(deficits, size=cfg.E)).astype(np.float32)
            sel[r.integers(cfg.E)] = np.float32(1.0)          # the token's largest |score|
            tol = Fraction(float(np.float64(orc.NEAR_TIE_REL) * float(np.abs(sel).max())))
            valid, gscore = brute_force_valid_sets(sel, cfg, tol)
            if not (_clear_of_boundary([Fraction(float(v)) for v in sel], tol)
                    and _clear_of_boundary(gscore, tol)):
                continue
            kept_tokens += 1
            n_multi += len(valid) > 1
            for S in combinations(range(cfg.E), cfg.k):
                got = o.is_valid_selection(list(S), sel, cfg)
                assert got == (frozenset(S) in valid), (ci, S, sel.tolist(), sorted(map(sorted, valid)))
            if kept_tokens == tokens:
                break
        assert kept_tokens == tokens, (ci, kept_tokens)
    assert n_multi >= 20, n_multi     # the cases do exercise several valid choices per token


def _route_with_scores(o, sel_rows, cfg, shift=0.0):
    """route() on sigmoid logits that reproduce the given selection scores
    (before a constant selection bias `shift`)."""
    p = np.asarray(sel_rows, np.float64)
    logits = np.log(p / (1.0 - p))
    bias = np.full(cfg.E, shift, np.float32) if shift else None
    return o.route(logits, bias, cfg)


def pin_group_near_tie_gap(o=orc):
    """The group near-tie flag of route(): a token whose topk_group-th and
    (topk_group+1)-th group scores differ by half the tolerance is a near tie,
    by twice the tolerance it is not; gaps between other ranks of groups do
    not count; the tolerance is relative to the token's largest |score|."""
    for score, top in (("max", 1), ("sum_top", 2)):
        cfg = orc.OracleConfig(T=4, d=1, E=8, I=1, k=2, n_shared=0, score_fn="sigmoid",
                               topk_method="group_limited_greedy", n_group=4, topk_group=2, group_score=score,
                               group_top=top)
        for shift in (0.0, 9.0):
            scale = 0.9 + shift
            tol = orc.NEAR_TIE_REL * scale

            def tok(g0, g1, g2, g3):
                # the first expert of each group carries the group's score, the second a low 0.1
                return [g0, 0.1, g1, 0.1, g2, 0.1, g3, 0.1]
            rows = [tok(0.9, 0.8, 0.8 - 0.5 * tol, 0.5),     # 2nd vs 3rd group: half the tolerance
                    tok(0.9, 0.8, 0.8 - 2.0 * tol, 0.5),     # 2nd vs 3rd group: twice the tolerance
                    tok(0.9, 0.9 - 0.5 * tol, 0.6, 0.5),     # 1st vs 2nd group close: no effect
                    tok(0.9, 0.8, 0.6, 0.6 - 0.5 * tol)]     # 3rd vs 4th group close: no effect
            r = _route_with_scores(o, rows, cfg, shift)
            assert r.near_tie.tolist() == [True, False, False, False], (score, shift, r.near_tie.tolist())
            # the kept groups are the first two in every row, so the expert gap (0.8 -> 0.1) is wide
            assert [sorted(i.tolist()) for i in r.idx] == [[0, 2]] * 4, r.idx


def pin_relative_error(o=orc):
    """relative_error = max |got - ref| / RMS(ref) over every element, on
    hand-worked arrays (the RMS is not the mean or the largest |ref|)."""
    ref = np.array([[3.0, 4.0]])
    assert abs(o.relative_error(np.array([[3.5, 3.0]]), ref) - 1.0 / math.sqrt(12.5)) <= 1e-15
    ref = np.array([1.0, -1.0, 1.0, 7.0])                       # RMS sqrt(13), mean |ref| 2.5, max |ref| 7
    got = ref + np.array([0.0, 0.5, 0.0, -0.25])
    assert abs(o.relative_error(got, ref) - 0.5 / math.sqrt(13.0)) <= 1e-15
    ref = np.array([[1.0, 2.0], [3.0, 4.0]])                    # RMS sqrt(7.5)
    got = np.array([[1.0, 2.0], [3.0, 2.5]])
    assert abs(o.relative_error(got, ref) - 1.5 / math.sqrt(7.5)) <= 1e-15
    assert o.relative_error(ref, ref) == 0.0


ALL_PINS = [pin_backward_finite_differences, pin_backward_homogeneity, pin_brute_force_selection, pin_greedy_is_torch_topk, pin_invariants,
            pin_bias_only_steers_selection, pin_zero_gates_give_shared, pin_group1_is_greedy,
            pin_single_expert, pin_dense_einsum, pin_top1, pin_permutation, pin_symmetries, pin_combine,
            pin_balance_update, pin_fp8_quantization, pin_valid_selection_brute_force,
            pin_group_near_tie_gap, pin_relative_error]
