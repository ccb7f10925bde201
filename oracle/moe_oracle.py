"""Plain fp64 CPU oracle of the DeepSeekMoE layer forward.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import or run
this module.  The product path (the CUDA library and its Python binding) never
calls it and shares no code with it: not a helper, not a table, not a constant.

What it computes (one token u_t at a time, all in float64 unless stated):

  1. logits  l_e = <u_t, W_g[e]>                      (gate linear layer, no bias)
  2. affinity s_e = softmax(l)_e over all E experts, or sigmoid(l_e)
  3. selection score  sigma_e = s_e + b_e            (b only steers selection)
  4. group-limited selection: contiguous groups of E/n_group experts, a group
     score (max, or sum of the top-m sigma in the group), keep the topk_group
     best groups, all other experts are ineligible
  5. top-k of sigma among the eligible experts, ties -> lower index
  6. gates g_j = s_{idx_j} (unbiased), optionally divided by their sum, times
     routed_scaling_factor
  7. out_t = sum_j g_j * FFN_{idx_j}(u_t) + FFN_shared(u_t), FFN = SwiGLU,
     no residual term.
  8. after a step (training-time load balancing): the selection bias of
     every expert moves by gamma toward balance, and the load statistics.
  9. FP8 expert weights: each run of 64 consecutive weights along a row is
     stored as FP8 e4m3 values times one power-of-two scale; the layer then
     computes steps 1-7 with the dequantized weights.
 10. backward (training): the gradient of <dout, out> with respect to x, W_g
     and every expert weight, by the chain rule through steps 7, 6 and 2 with
     the expert choice of step 5 held fixed (a choice is piecewise constant in
     the inputs; the selection bias carries no gradient).

Sources (page title, section):
  * "DeepSeek-V2" walkthrough (xingfushuangcheng.com): the DeepSeekMoE output
    definition for token t, the ``MoEGate`` listing (fp32 linear gate, softmax
    over all experts, greedy / group_limited_greedy, group score = max) and the
    ``MoE`` listing (repeat per top-k slot, per-expert FFN, gate-weighted sum
    plus the shared experts as one SwiGLU of hidden n_shared * I).
  * "DeepSeek大模型架构解析：MLA注意力与MoE创新设计" (intelliparadigm.com),
    section 3.3.1: SwiGLU = w2(silu(w1 x) * w3 x) with bias-free linears.
  * "【多模态大模型面经】 DeepSeek专题： DeepSeekMOE + MLA" (Tencent Cloud),
    router formula: p = softmax(W_gate x), y = sum over TopK(p) of p_i E_i(x).
  * "【Deepseek基础篇】--v3基本架构" (nxbn.cn), section 1.2: a per-expert bias is
    added to the affinity only to pick the top-K, gate values come from the
    unbiased affinity; node-limited routing picks nodes by the sum of the
    highest affinities on each node; no token is dropped; after each step the
    bias of an overloaded expert is lowered by the bias update speed gamma and
    that of an underloaded expert raised by gamma.
  * Tencent Cloud page, the balance-loss listing: load = per-expert counts of
    the top-k choices normalised to sum 1, and its standard deviation.
  * intelliparadigm.com page, section 4 (FP8 quantisation): weights quantised
    block by block (a block of 64 consecutive values, its own scale from the
    block's largest magnitude), experts quantised independently, GEMM inputs
    dequantised before the multiplication, accumulation in higher precision.

Readings where the pages are silent or garbled:
  * Decision precision.  The ``MoEGate`` listing holds logits and scores in
    float32 and takes ``topk`` on them.  The oracle therefore computes the
    affinities exactly (float64), rounds them once to float32, adds the float32
    bias in float32, and makes every comparison (group choice, top-k) on those
    float32 values.  Equal float32 values go to the lower index.
  * Group score "sum_top" (V3 node-limited routing, count garbled on the page):
    the sum of the top-m selection scores of the group, summed in float32 in
    descending order.  m = k / topk_group in the V3-shaped workloads.
  * Experts outside the kept groups are excluded outright (not zero-filled), so
    a negative biased score can never pull in an expert from a dropped group.
  * Overloaded / underloaded (step 8): more / fewer assignments than the mean
    T*k/E, decided exactly on integers; an expert at exactly the mean keeps its
    bias.  The bias is float32 and moves by one float32 addition.  The load
    standard deviation is the unbiased one (the listing's torch .std()).
  * FP8 weights (step 9): the section's listing rounds to an integer range
    (+-127) although it is titled FP8; here the values are FP8 e4m3 (largest
    finite 448, round to nearest even) and each block's scale is the smallest
    power of two with max|w| <= 448 * scale, so a dequantized weight is exactly
    a bf16 number.
  * A token is a near tie when the k-th and (k+1)-th eligible selection scores
    (or the topk_group-th and next group scores) differ by less than 1e-5 times
    the largest |score| of that token; its expert set may legitimately differ
    between two correct implementations.
"""
from __future__ import annotations

from dataclasses import dataclass
from itertools import combinations
from typing import Callable, Optional, Sequence, Tuple

import numpy as np

NEAR_TIE_REL = 1e-5


@dataclass
class OracleConfig:
    """Plain layer hyper-parameters, named as in the ``MoEGate`` / ``MoE`` listings."""

    T: int
    d: int
    E: int                      # n_routed_experts
    I: int                      # routed expert hidden size
    k: int                      # num_experts_per_tok
    n_shared: int               # shared experts, fused as one SwiGLU of hidden n_shared*I
    score_fn: str = "softmax"   # "softmax" | "sigmoid"
    topk_method: str = "greedy"  # "greedy" | "group_limited_greedy"
    n_group: int = 1
    topk_group: int = 1
    group_score: str = "max"    # "max" | "sum_top"
    group_top: int = 1          # m for "sum_top"
    norm_topk: bool = False
    routed_scaling_factor: float = 1.0


@dataclass
class Routing:
    idx: np.ndarray        # [T,k] int64, ordered by selection score desc, then index asc
    gates: np.ndarray      # [T,k] float64
    scores: np.ndarray     # [T,E] float64 affinities s
    sel32: np.ndarray      # [T,E] float32 selection scores (decision values)
    near_tie: np.ndarray   # [T] bool
    counts: np.ndarray     # [E] int64


# --------------------------------------------------------------------- router

def gate_logits(x: np.ndarray, wg: np.ndarray) -> np.ndarray:
    """l = x W_g^T in float64 (``MoEGate.forward``: ``F.linear`` without bias)."""
    return np.asarray(x, np.float64) @ np.asarray(wg, np.float64).T


def affinities(logits: np.ndarray, score_fn: str) -> np.ndarray:
    """Token-to-expert affinity s (``MoEGate.forward`` softmax over all experts;
    the V3 page's sigmoid affinity)."""
    logits = np.asarray(logits, np.float64)
    if score_fn == "softmax":
        z = logits - logits.max(axis=1, keepdims=True)
        ez = np.exp(z)
        return ez / ez.sum(axis=1, keepdims=True)
    if score_fn == "sigmoid":
        return 1.0 / (1.0 + np.exp(-logits))
    raise ValueError(score_fn)


def selection_scores32(s: np.ndarray, bias: Optional[np.ndarray]) -> np.ndarray:
    """sigma = s + b, held in float32 as the gate listing holds its scores."""
    s32 = np.asarray(s, np.float64).astype(np.float32)
    if bias is None:
        return s32
    return (s32 + np.asarray(bias, np.float32)[None, :]).astype(np.float32)


def _group_scores32(sel32: np.ndarray, cfg: OracleConfig) -> np.ndarray:
    T, E = sel32.shape
    grp = sel32.reshape(T, cfg.n_group, E // cfg.n_group)
    if cfg.group_score == "max":
        return grp.max(axis=2)
    if cfg.group_score == "sum_top":
        desc = -np.sort(-grp, axis=2)          # descending within each group
        acc = desc[:, :, 0].astype(np.float32)
        for m in range(1, cfg.group_top):
            acc = (acc + desc[:, :, m]).astype(np.float32)
        return acc
    raise ValueError(cfg.group_score)


def _group_scores64(sel64: np.ndarray, cfg: OracleConfig) -> np.ndarray:
    T, E = sel64.shape
    grp = sel64.reshape(T, cfg.n_group, E // cfg.n_group)
    if cfg.group_score == "max":
        return grp.max(axis=2)
    desc = -np.sort(-grp, axis=2)
    return desc[:, :, : cfg.group_top].sum(axis=2)


def eligible_mask(sel32: np.ndarray, cfg: OracleConfig) -> Tuple[np.ndarray, np.ndarray]:
    """Experts a token may pick, and the kept-group matrix [T, n_group].

    greedy: every expert.  group_limited_greedy (``MoEGate`` listing; the V3
    page's node-limited routing): keep the topk_group groups with the largest
    group score, ties -> lower group index."""
    T, E = sel32.shape
    if cfg.topk_method == "greedy":
        return np.ones((T, E), bool), np.ones((T, 1), bool)
    if cfg.topk_method != "group_limited_greedy":
        raise ValueError(cfg.topk_method)
    gs = _group_scores32(sel32, cfg)
    order = np.argsort(-gs, axis=1, kind="stable")   # stable: equal -> lower index first
    kept = np.zeros_like(gs, dtype=bool)
    rows = np.arange(T)[:, None]
    kept[rows, order[:, : cfg.topk_group]] = True
    return np.repeat(kept, E // cfg.n_group, axis=1), kept


def route(logits: np.ndarray, bias: Optional[np.ndarray], cfg: OracleConfig) -> Routing:
    """Router of one batch: affinities, (group-limited) top-k, gate values."""
    s = affinities(logits, cfg.score_fn)
    T, E = s.shape
    sel32 = selection_scores32(s, bias)
    elig, kept = eligible_mask(sel32, cfg)
    key = np.where(elig, sel32.astype(np.float64), -np.inf)
    order = np.argsort(-key, axis=1, kind="stable")
    idx = order[:, : cfg.k].astype(np.int64)

    g = gate_values(s, idx, cfg)

    # near ties, judged on exact float64 selection scores
    sel64 = s + (0.0 if bias is None else np.asarray(bias, np.float64)[None, :])
    near = near_ties(sel64, elig, cfg)
    counts = np.bincount(idx.ravel(), minlength=E).astype(np.int64)
    return Routing(idx=idx, gates=g, scores=s, sel32=sel32, near_tie=near, counts=counts)


def gate_values(s: np.ndarray, idx: np.ndarray, cfg: OracleConfig) -> np.ndarray:
    """Gate values [T,k] of a choice idx: the unbiased affinities of the chosen
    experts (V3 page, section 1.2), divided by their sum when norm_topk, times
    routed_scaling_factor."""
    rows = np.arange(idx.shape[0])[:, None]
    g = np.asarray(s, np.float64)[rows, idx]
    if cfg.norm_topk:
        g = g / g.sum(axis=1, keepdims=True)
    return g * float(cfg.routed_scaling_factor)


def near_ties(sel64: np.ndarray, elig: np.ndarray, cfg: OracleConfig) -> np.ndarray:
    """[T] bool: tokens whose choice two correct implementations may make
    differently.  With tol = NEAR_TIE_REL times the token's largest |score|
    (exact float64 selection scores sel64), a token is a near tie when its k-th
    and (k+1)-th eligible scores differ by less than tol, or, for group-limited
    routing that drops groups, its topk_group-th and (topk_group+1)-th largest
    group scores do."""
    T, E = sel64.shape
    scale = np.abs(sel64).max(axis=1)
    near = np.zeros(T, bool)
    n_elig = elig.sum(axis=1)
    if cfg.k < E:
        e64 = np.where(elig, sel64, -np.inf)
        desc = -np.sort(-e64, axis=1)
        has_next = n_elig > cfg.k
        gap = np.where(has_next, desc[:, cfg.k - 1] - desc[:, cfg.k], np.inf)
        near |= gap < NEAR_TIE_REL * scale
    if cfg.topk_method == "group_limited_greedy" and cfg.topk_group < cfg.n_group:
        g64 = -np.sort(-_group_scores64(sel64, cfg), axis=1)
        ggap = g64[:, cfg.topk_group - 1] - g64[:, cfg.topk_group]
        near |= ggap < NEAR_TIE_REL * scale
    return near


def route_tokens(x, wg, bias, cfg: OracleConfig) -> Routing:
    return route(gate_logits(x, wg), bias, cfg)


# ---------------------------------------------------------------- permutation

def permutation(idx: np.ndarray, E: int):
    """Expert-contiguous order of the T*k (token, slot) assignments.

    Rows of expert e are its assignments in increasing token order (each token
    picks an expert at most once), experts in increasing id; this is the
    per-expert gather of the ``MoE`` listing made explicit.
    Returns counts[E], offsets[E+1], row2tok[R], tok2row[T,k]."""
    idx = np.asarray(idx)
    T, k = idx.shape
    counts = np.zeros(E, np.int64)
    for e in idx.ravel():
        counts[e] += 1
    offsets = np.zeros(E + 1, np.int64)
    offsets[1:] = np.cumsum(counts)
    nxt = offsets[:-1].copy()
    row2tok = np.zeros(T * k, np.int64)
    tok2row = np.zeros((T, k), np.int64)
    # counting sort: visiting assignments in (token, slot) order keeps each
    # expert's rows in increasing token order
    for t in range(T):
        for j in range(k):
            e = idx[t, j]
            r = nxt[e]
            nxt[e] += 1
            row2tok[r] = t
            tok2row[t, j] = r
    return counts, offsets, row2tok, tok2row


# -------------------------------------------------------------------- experts

def silu(z: np.ndarray) -> np.ndarray:
    return z / (1.0 + np.exp(-z))


def swiglu_ffn(u: np.ndarray, w1: np.ndarray, w3: np.ndarray, w2: np.ndarray) -> np.ndarray:
    """FFN(u) = W2 (silu(W1 u) * (W3 u)); nn.Linear layouts W1,W3 [h,d], W2 [d,h]
    (intelliparadigm.com page, section 3.3.1)."""
    u = np.asarray(u, np.float64)
    a = u @ np.asarray(w1, np.float64).T
    b = u @ np.asarray(w3, np.float64).T
    return (silu(a) * b) @ np.asarray(w2, np.float64).T


ExpertFn = Callable[[int], Tuple[np.ndarray, np.ndarray, np.ndarray]]


def experts_forward(x: np.ndarray, idx: np.ndarray, gates: np.ndarray,
                    expert: ExpertFn, shared: Optional[Tuple[np.ndarray, np.ndarray, np.ndarray]],
                    E: int) -> np.ndarray:
    """out_t = sum_j g_{t,j} FFN_{idx[t,j]}(x_t) + FFN_shared(x_t) (``MoE`` listing).

    ``expert(e)`` returns expert e's (W1, W3, W2); only experts some token
    picked are requested.  No residual term is added."""
    x = np.asarray(x, np.float64)
    T, d = x.shape
    out = np.zeros((T, d), np.float64)
    for e in range(E):
        tok, slot = np.nonzero(idx == e)
        if tok.size == 0:
            continue
        w1, w3, w2 = expert(e)
        y = swiglu_ffn(x[tok], w1, w3, w2)
        np.add.at(out, tok, gates[tok, slot][:, None] * y)
    if shared is not None:
        out += swiglu_ffn(x, *shared)
    return out


def combine(y_rows: np.ndarray, y_shared: Optional[np.ndarray], tok2row: np.ndarray,
            gates: np.ndarray) -> np.ndarray:
    """out_t = sum_j g_{t,j} * y_rows[tok2row[t,j]] + y_shared[t]: the ``MoE``
    listing's gate-weighted sum over the k slots of a token plus the shared
    experts, with the slot rows stored in expert-contiguous order."""
    y_rows = np.asarray(y_rows, np.float64)
    T, k = tok2row.shape
    out = np.zeros((T, y_rows.shape[1]), np.float64)
    for j in range(k):
        out += np.asarray(gates, np.float64)[:, j:j + 1] * y_rows[tok2row[:, j]]
    if y_shared is not None:
        out += np.asarray(y_shared, np.float64)
    return out


def moe_forward(x, wg, bias, expert: ExpertFn, shared, cfg: OracleConfig,
                idx_override: Optional[np.ndarray] = None):
    """Whole layer for the tokens in ``x``.  ``idx_override`` re-evaluates the
    layer with another (equally valid) expert choice, used for near-tie tokens.
    Returns (out [T,d] float64, Routing)."""
    r = route_tokens(x, wg, bias, cfg)
    idx, gates = r.idx, r.gates
    if idx_override is not None:
        idx = np.asarray(idx_override, np.int64)
        gates = gate_values(r.scores, idx, cfg)
    out = experts_forward(x, idx, gates, expert, shared, cfg.E)
    return out, Routing(idx=idx, gates=gates, scores=r.scores, sel32=r.sel32,
                        near_tie=r.near_tie, counts=np.bincount(idx.ravel(), minlength=cfg.E))


def stacked_experts(w1: np.ndarray, w3: np.ndarray, w2: np.ndarray) -> ExpertFn:
    """Expert accessor over stacked [E,I,d],[E,I,d],[E,d,I] arrays."""
    return lambda e: (w1[e], w3[e], w2[e])


def relative_error(got: np.ndarray, ref: np.ndarray) -> float:
    """max |got - ref| / RMS(ref), the acceptance measure for layer outputs."""
    ref = np.asarray(ref, np.float64)
    got = np.asarray(got, np.float64)
    rms = float(np.sqrt(np.mean(ref * ref)))
    return float(np.max(np.abs(got - ref))) / max(rms, 1e-300)


def is_valid_selection(idx_row: Sequence[int], sel32_row: np.ndarray, cfg: OracleConfig) -> bool:
    """True when ``idx_row`` is a correct top-k choice up to the near-tie
    tolerance tol (NEAR_TIE_REL times the token's largest |score|).  Used to
    accept the other side's choice on near-tie tokens.

    The choice is valid when some set K of kept groups (every expert's group
    for greedy routing; topk_group groups otherwise) satisfies all of:
      (a) K holds the group of every picked expert;
      (b) no group outside K has a group score above the lowest group score
          in K by more than tol (K is a top-topk_group set up to tol);
      (c) no expert of K left unpicked has a selection score above the
          lowest picked score by more than tol (the k experts are a top-k
          set of K's experts up to tol).
    The k experts must be distinct.  Every K is tried (at most C(8, 4) = 70)."""
    sel = np.asarray(sel32_row, np.float64)
    picked = np.asarray(list(idx_row), np.int64)
    if len(set(picked.tolist())) != cfg.k:
        return False
    tol = NEAR_TIE_REL * np.abs(sel).max()
    if cfg.topk_method == "group_limited_greedy":
        gsize = cfg.E // cfg.n_group
        g = _group_scores64(sel[None, :], cfg)[0]
        need = set((picked // gsize).tolist())
        candidates = []
        for K in combinations(range(cfg.n_group), cfg.topk_group):
            if not need <= set(K):                                   # (a)
                continue
            in_k = np.zeros(cfg.n_group, bool)
            in_k[list(K)] = True
            if (~in_k).any() and g[~in_k].max() > g[in_k].min() + tol:   # (b)
                continue
            candidates.append(np.repeat(in_k, gsize))
    else:
        candidates = [np.ones(cfg.E, bool)]
    worst_picked = sel[picked].min()
    for elig in candidates:
        others = np.where(elig, sel, -np.inf)
        others[picked] = -np.inf
        if others.max() <= worst_picked + tol:                        # (c)
            return True
    return False


# ------------------------------------------------------------ load balancing

def balance_update(counts, bias32, gamma: float):
    """Step 8: the bias after one auxiliary-loss-free balancing step and the
    load statistics.

    "v3基本架构" page, section 1.2: at the end of a step an overloaded expert's
    bias is lowered by gamma and an underloaded expert's bias raised by gamma.
    Tencent Cloud balance-loss listing: load = counts / sum(counts) and its
    standard deviation.

    Returns (new bias as float32 [E], stats float64 [3]) with stats =
    (unbiased std of the load fractions, max count / mean count,
    min count / mean count)."""
    c = np.asarray(counts, dtype=np.int64)
    E = c.size
    total = int(c.sum())
    b = np.asarray(bias32, dtype=np.float32)
    g = np.float32(gamma)
    new = b.copy()
    for e in range(E):
        if c[e] * E > total:        # took more than the mean T*k/E
            new[e] = np.float32(b[e] - g)
        elif c[e] * E < total:      # took fewer
            new[e] = np.float32(b[e] + g)
    stats = np.zeros(3)
    if total > 0:
        load = c.astype(np.float64) / total
        if E > 1:
            stats[0] = np.sqrt(((load - load.mean()) ** 2).sum() / (E - 1))
        mean = total / E
        stats[1] = c.max() / mean
        stats[2] = c.min() / mean
    return new, stats


# --------------------------------------------------------- FP8 expert weights

E4M3_MAX = 448.0
FP8_BLOCK = 64


def e4m3_round(v: np.ndarray) -> np.ndarray:
    """Nearest FP8 e4m3 value of each float64 (ties to even mantissa), for
    |v| <= 448.  e4m3: sign, 4 exponent bits (bias 7), 3 mantissa bits; normal
    values from 2^-6 up, subnormals are multiples of 2^-9."""
    v = np.asarray(v, np.float64)
    a = np.abs(v)
    _, x = np.frexp(np.where(a > 0, a, 1.0))       # a = f * 2^x, f in [0.5, 1)
    e = np.maximum(x - 1, -6)                       # binade 2^e <= a < 2^(e+1), clamped to the subnormal step
    step = np.ldexp(1.0, (e - 3).astype(np.int64))  # spacing of e4m3 values in that binade
    q = np.round(a / step) * step                   # a / step is exact; np.round ties to even
    return np.copysign(np.minimum(q, E4M3_MAX), v)


def quantize_fp8_blocks(w: np.ndarray):
    """Step 9: w [rows, cols] (cols a multiple of 64) -> (q, scale): q [rows, cols]
    the e4m3 values, scale [rows, cols/64] the blocks' powers of two, with
    w ~= q * scale.  The scale is the smallest power of two with
    max|w| <= 448 * scale over the block (1 for an all-zero block)."""
    w = np.asarray(w, np.float64)
    rows, cols = w.shape
    blocks = w.reshape(rows, cols // FP8_BLOCK, FP8_BLOCK)
    amax = np.abs(blocks).max(axis=2)
    f, x = np.frexp(amax)                           # amax = f * 2^x
    # amax <= 448 * 2^e  <=>  f * 2^x <= 1.75 * 2^(8 + e)
    e = np.where(f <= 0.875, x - 9, x - 8)
    e = np.where(amax == 0, 0, e).astype(np.int64)
    scale = np.ldexp(1.0, e)
    q = e4m3_round(blocks / scale[..., None])
    return q.reshape(rows, cols), scale


def dequantize_fp8_blocks(q: np.ndarray, scale: np.ndarray) -> np.ndarray:
    rows, cols = q.shape
    return (np.asarray(q, np.float64).reshape(rows, cols // FP8_BLOCK, FP8_BLOCK)
            * np.asarray(scale, np.float64)[..., None]).reshape(rows, cols)


def fp8_dequantized(w: np.ndarray) -> np.ndarray:
    """The weights the FP8 layer computes with (step 9)."""
    q, s = quantize_fp8_blocks(w)
    return dequantize_fp8_blocks(q, s)


# ------------------------------------------------------------------- backward

def silu_grad(z: np.ndarray) -> np.ndarray:
    """d silu / dz = sigma(z) * (1 + z * (1 - sigma(z)))."""
    sg = 1.0 / (1.0 + np.exp(-z))
    return sg * (1.0 + z * (1.0 - sg))


def swiglu_backward(u: np.ndarray, w1, w3, w2, dy: np.ndarray):
    """Gradients of y = W2 (silu(W1 u) * (W3 u)) for rows u [n,d] and upstream
    dy [n,d]: returns (du [n,d], dW1 [h,d], dW3 [h,d], dW2 [d,h])."""
    u = np.asarray(u, np.float64)
    w1 = np.asarray(w1, np.float64)
    w3 = np.asarray(w3, np.float64)
    w2 = np.asarray(w2, np.float64)
    dy = np.asarray(dy, np.float64)
    a = u @ w1.T
    b = u @ w3.T
    h = silu(a) * b
    dw2 = dy.T @ h
    dh = dy @ w2
    da = dh * b * silu_grad(a)
    db = dh * silu(a)
    du = da @ w1 + db @ w3
    return du, da.T @ u, db.T @ u, dw2


def gate_backward(dg: np.ndarray, s: np.ndarray, idx: np.ndarray, cfg: OracleConfig) -> np.ndarray:
    """d L / d logits [T,E] from d L / d g [T,k]: through step 6 (g = c * raw /
    sum(raw) or c * raw, raw = s at the chosen experts) and step 2 (sigmoid, or
    softmax over all E experts)."""
    dg = np.asarray(dg, np.float64)
    s = np.asarray(s, np.float64)
    T, k = dg.shape
    rows = np.arange(T)[:, None]
    raw = s[rows, idx]
    c = float(cfg.routed_scaling_factor)
    if cfg.norm_topk:
        ssum = raw.sum(axis=1, keepdims=True)
        draw = c * (dg / ssum - np.sum(dg * raw, axis=1, keepdims=True) / (ssum * ssum))
    else:
        draw = c * dg
    ds = np.zeros_like(s)
    np.add.at(ds, (np.repeat(np.arange(T), k), np.asarray(idx).ravel()), draw.ravel())
    if cfg.score_fn == "sigmoid":
        return ds * s * (1.0 - s)
    return s * (ds - np.sum(ds * s, axis=1, keepdims=True))


def expert_backward(x, dout, idx, gates, e: int, w1e, w3e, w2e):
    """Expert e's share of the gradient of L = <dout, out> (step 10): its rows
    are the (token, slot) pairs with idx[t,j] = e, whose outputs enter out_t
    with weight g_{t,j}.  Returns (tokens, slots, dL/dg for those slots, the
    rows' dL/dx [n,d], dW1 [h,d], dW3 [h,d], dW2 [d,h])."""
    x = np.asarray(x, np.float64)
    dout = np.asarray(dout, np.float64)
    tok, slot = np.nonzero(np.asarray(idx) == e)
    y = swiglu_ffn(x[tok], w1e, w3e, w2e)                # expert output rows
    dg = np.sum(dout[tok] * y, axis=1)                   # d L / d g_{t,j}
    dy = np.asarray(gates, np.float64)[tok, slot][:, None] * dout[tok]
    du, g1, g3, g2 = swiglu_backward(x[tok], w1e, w3e, w2e, dy)
    return tok, slot, dg, du, g1, g3, g2


def moe_backward(x, wg, bias, w1, w3, w2, shared, dout, cfg: OracleConfig,
                 idx_override: Optional[np.ndarray] = None, weight_grads: bool = True):
    """Gradient of L = <dout, out> for the layer of ``moe_forward`` (step 10).

    w1, w3 [E,I,d] and w2 [E,d,I] are the routed experts (anything that
    yields expert e's matrix as w[e]), ``shared`` the shared expert's
    (W1, W3, W2) or None.  Returns a dict with dx [T,d], dwg [E,d], dw1, dw3,
    dw2 (stacked like the weights; None when ``weight_grads`` is False) and
    dws1, dws3, dws2, plus the Routing used."""
    x = np.asarray(x, np.float64)
    wg = np.asarray(wg, np.float64)
    dout = np.asarray(dout, np.float64)
    T, d = x.shape
    E, k = cfg.E, cfg.k
    logits = gate_logits(x, wg)
    r = route(logits, bias, cfg)
    idx = r.idx if idx_override is None else np.asarray(idx_override, np.int64)
    s = r.scores
    gates = gate_values(s, idx, cfg)

    dx = np.zeros((T, d), np.float64)
    dw1 = np.zeros(np.shape(w1), np.float64) if weight_grads else None
    dw3 = np.zeros(np.shape(w3), np.float64) if weight_grads else None
    dw2 = np.zeros(np.shape(w2), np.float64) if weight_grads else None
    dg = np.zeros((T, k), np.float64)
    for e in range(E):
        if not (idx == e).any():
            continue
        tok, slot, dg_e, du, g1, g3, g2 = expert_backward(x, dout, idx, gates, e, w1[e], w3[e], w2[e])
        dg[tok, slot] = dg_e
        np.add.at(dx, tok, du)
        if weight_grads:
            dw1[e] += g1
            dw3[e] += g3
            dw2[e] += g2
    out = {"dw1": dw1, "dw3": dw3, "dw2": dw2, "dws1": None, "dws3": None, "dws2": None}
    if shared is not None:
        du, g1, g3, g2 = swiglu_backward(x, *shared, dout)
        dx += du
        out.update(dws1=g1, dws3=g3, dws2=g2)

    dl = gate_backward(dg, s, idx, cfg)
    dx += dl @ wg
    out.update(dx=dx, dwg=dl.T @ x, routing=r)
    return out

