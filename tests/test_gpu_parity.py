"""Parity of the CUDA library (through the C ABI) with the fp64 CPU oracle.

Every input comes from the seeded generator; the oracle sees byte-identical
copies.  Acceptance (layer spec): expert indices set-exact on every token that
is not a near tie (near-tie tokens are counted and their GPU choice must be a
valid top-k); gate values within 1e-5 relative; counts / offsets / row order
bit-exact; outputs max|GPU - oracle| / RMS(oracle) <= 2e-2 (bf16) or 1e-4
(fp32).  Small cases span several tiles with ragged tails and are checked on
every token; the full-size workloads run in the benchmark's launch
configuration and are checked on all routing decisions and on sampled
output rows."""
import dataclasses

import numpy as np
import pytest
import torch

from mixture_experts_layer_85_b300 import _lib, inputs
from mixture_experts_layer_85_b300.layer import MoELayer
from oracle import moe_oracle as orc
from tests._cfg import expert_accessor, f64, oracle_cfg, output_error

pytestmark = pytest.mark.gpu

TOL = {"bf16": 2e-2, "f32": 1e-4}
GATE_RTOL = 1e-5

W = inputs.WORKLOADS
SMALL = {
    # softmax greedy, fp32 gate weight split over three bf16 MMAs (T >= 1024)
    "v2lite_small_t1037": inputs.small_workload(W["v2lite_t4096"], name="v2lite_small_t1037", T=1037, d=384,
                                                E=16, I=256, k=6, n_shared=2),
    # softmax group-limited (max), scale 16, SIMT gate
    "v2_small_t515": inputs.small_workload(W["v2_t8192"], name="v2_small_t515", T=515, d=256, E=32, I=128,
                                           n_group=8, topk_group=3),
    # sigmoid + bias, group-limited sum of top-2, renormalised, scale 2.5
    "v3_small_t333": inputs.small_workload(W["v3_prefill_t16384"], name="v3_small_t333", T=333, d=512, E=64,
                                           I=256, n_group=8, topk_group=4),
    # tensor-core gate path with bf16 gate weights, ragged last tile
    "v3_small_t1100": inputs.small_workload(W["v3_prefill_t16384"], name="v3_small_t1100", T=1100, d=512,
                                            E=64, I=128, n_group=8, topk_group=4),
    # d not a multiple of 128: zero-padded weight stages and row tiles that end inside a pair tile
    "v3_small_d320_t97": inputs.small_workload(W["v3_prefill_t16384"], name="v3_small_d320_t97", T=97, d=320, E=32,
                                               I=128, n_group=8, topk_group=4),
    # decode-sized batches
    "v3_small_t1": inputs.small_workload(W["v3_prefill_t16384"], name="v3_small_t1", T=1, d=512, E=64, I=256,
                                         n_group=8, topk_group=4),
    "v3_small_t3": inputs.small_workload(W["v3_prefill_t16384"], name="v3_small_t3", T=3, d=512, E=64, I=256,
                                         n_group=8, topk_group=4),
    # no shared expert: the expert kernel's shared classes are absent
    "v2lite_small_t77_noshared": inputs.small_workload(W["v2lite_t4096"], name="v2lite_small_t77_noshared", T=77,
                                                       d=256, E=16, I=256, k=6, n_shared=0),
}


def _np(t):
    return t.detach().cpu().numpy()


def oracle_route(li, wl):
    bias = None if li.bias is None else _np(li.bias.float())
    return orc.route(orc.gate_logits(f64(li.x), f64(li.wg)), bias, oracle_cfg(wl))


def check_routing(gidx, gw, r, wl):
    """Returns (near-tie tokens, near-tie tokens whose choice differs)."""
    cfg = oracle_cfg(wl)
    gidx = np.asarray(gidx, np.int64)
    same = (np.sort(gidx, 1) == np.sort(r.idx, 1)).all(1)
    near = r.near_tie
    bad = ~same & ~near
    assert not bad.any(), f"expert sets differ on {int(bad.sum())} non-tie tokens, e.g. {np.nonzero(bad)[0][:5]}"
    differ = ~same & near
    for t in np.nonzero(differ)[0]:
        assert orc.is_valid_selection(gidx[t], r.sel32[t], cfg), t
    # gate values, matched per expert, on tokens with the same set
    og = np.take_along_axis(r.gates, np.argsort(r.idx, 1), 1)
    gg = np.take_along_axis(np.asarray(gw, np.float64), np.argsort(gidx, 1), 1)
    rel = np.abs(gg - og) / np.maximum(np.abs(og), 1e-30)
    assert rel[same].max(initial=0.0) <= GATE_RTOL, rel[same].max()
    # reported order: selection score descending (up to the tie tolerance)
    rows = np.arange(gidx.shape[0])[:, None]
    s_ord = r.sel32.astype(np.float64)[rows, gidx]
    tol = orc.NEAR_TIE_REL * np.abs(r.sel32).max(1, keepdims=True)
    assert (np.diff(s_ord, axis=1) <= tol).all()
    return int(near.sum()), int(differ.sum())


def check_counts(gcounts, gidx, r, wl, n_differ):
    gcounts = np.asarray(gcounts, np.int64)
    assert gcounts.sum() == wl.T * wl.k
    assert np.array_equal(gcounts, np.bincount(np.asarray(gidx).ravel(), minlength=wl.E))
    assert np.abs(gcounts - r.counts).sum() <= 2 * wl.k * n_differ


def shared_of(li):
    return None if li.wl.n_shared == 0 else (f64(li.ws1), f64(li.ws3), f64(li.ws2))


def run_layer(wl, li):
    layer = MoELayer(wl, li, "cuda")
    T, k, E = wl.T, wl.k, wl.E
    idx = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    counts = torch.empty((E,), dtype=torch.int32, device="cuda")
    out = layer.forward(li.x, idx=idx, w=w, counts=counts)
    code, word = layer.device_status()
    assert code == _lib.MOE_OK, (_lib.moe_status_string(code), word)
    return layer, out, idx, w, counts


def check_layer(wl, li, out, idx, w, counts, sample=None):
    """Routing of every token, counts, and the outputs of `sample` (all tokens
    when None) against the oracle.  A near-tie token whose GPU choice differs
    from the oracle's (a valid choice, checked in check_routing) is compared
    with the oracle evaluated on the GPU's choice."""
    r = oracle_route(li, wl)
    cfg = oracle_cfg(wl)
    gidx, gw = _np(idx), _np(w)
    n_near, n_differ = check_routing(gidx, gw, r, wl)
    check_counts(_np(counts), gidx, r, wl, n_differ)
    toks = np.arange(wl.T) if sample is None else sample
    use = r.idx[toks].copy()
    differ = ~(np.sort(gidx[toks], 1) == np.sort(use, 1)).all(1)
    use[differ] = gidx[toks][differ]
    gates = orc.gate_values(r.scores[toks], use, cfg)
    want = orc.experts_forward(f64(li.x)[toks], use, gates, expert_accessor(li.w1, li.w3, li.w2), shared_of(li),
                               wl.E)
    err = output_error(f64(out)[toks], want, wl.out_dtype)
    assert err <= TOL[wl.act_dtype], err
    return {"near_tie": n_near, "near_tie_differ": n_differ, "err": err, "checked_tokens": int(toks.size),
            "checked_on_gpu_choice": int(differ.sum())}


def full_size_sample(wl):
    """Tokens whose outputs a full-size test compares: every token of a decode
    batch (T <= 512), 2048 seeded tokens of the V3 prefill layer, 1024 of the
    V2-shaped ones."""
    if wl.T <= 512:
        return None
    n = 2048 if wl.d >= 7168 else 1024
    return np.sort(np.random.default_rng(7).choice(wl.T, n, replace=False))


# ----------------------------------------------------------------- full layer

def test_tiny_fp32_layer():
    wl = W["tiny_fp32_t128"]
    li = inputs.make_inputs(wl, "cuda")
    _, out, idx, w, counts = run_layer(wl, li)
    info = check_layer(wl, li, out, idx, w, counts)
    assert info["err"] <= 1e-4


@pytest.mark.parametrize("name", list(SMALL))
def test_small_bf16_layer(name):
    wl = SMALL[name]
    li = inputs.make_inputs(wl, "cuda")
    _, out, idx, w, counts = run_layer(wl, li)
    check_layer(wl, li, out, idx, w, counts)


FULL = ["v2lite_t4096", "v2_t8192", "v3_prefill_t16384", "v3_decode_t1", "v3_decode_t8", "v3_decode_t64",
        "v3_decode_t512"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_layer(name):
    """Full workload in the benchmark's launch configuration: every routing
    decision against the oracle, sampled output rows against the oracle."""
    wl = W[name]
    li = inputs.make_inputs(wl, "cuda")
    _, out, idx, w, counts = run_layer(wl, li)
    info = check_layer(wl, li, out, idx, w, counts, sample=full_size_sample(wl))
    print(name, info)
    del li, out
    torch.cuda.empty_cache()


def test_stacked_calls_on_one_stream():
    """Layers stacked on one stream and one workspace with no synchronisation:
    each call's bf16 output is the next call's input.  Every output matches the
    oracle evaluated on the GPU's input of that call (a call must not start
    reading x, or overwrite the hidden rows, while the previous call runs)."""
    for T in (40, 1100):
        wl = inputs.small_workload(W["v3_prefill_t16384"], name=f"v3_stack_t{T}", T=T, d=512, E=64, I=256,
                                   n_group=8, topk_group=4, out_dtype="bf16")
        li = inputs.make_inputs(wl, "cuda")
        layer = MoELayer(wl, li, "cuda")
        xs, routes = [li.x], []
        for _ in range(3):
            idx = torch.empty((T, wl.k), dtype=torch.int32, device="cuda")
            w = torch.empty((T, wl.k), dtype=torch.float32, device="cuda")
            counts = torch.empty((wl.E,), dtype=torch.int32, device="cuda")
            xs.append(layer.forward(xs[-1], idx=idx, w=w, counts=counts))
            routes.append((idx, w, counts))
        code, word = layer.device_status()
        assert code == _lib.MOE_OK, (_lib.moe_status_string(code), word)
        for i, (idx, w, counts) in enumerate(routes):
            li_i = dataclasses.replace(li, x=xs[i])
            check_layer(wl, li_i, xs[i + 1], idx, w, counts)


def _twin_router(wl, twins):
    """Router inputs with bit-identical selection scores: every expert 2i+1 a
    copy of expert 2i (twins='experts'), or every group 2j+1 a copy of group 2j
    (twins='groups'), gate weight rows and bias entries alike."""
    wg, bias = inputs.make_router(wl)
    wg = wg.clone()
    bias = None if bias is None else bias.clone()
    if twins == "experts":
        src, dst = torch.arange(0, wl.E, 2), torch.arange(1, wl.E, 2)
    else:
        gs = wl.E // wl.n_group
        grp = torch.arange(wl.E).view(wl.n_group, gs)
        src, dst = grp[0::2].reshape(-1), grp[1::2].reshape(-1)
    wg[dst] = wg[src]
    if bias is not None:
        bias[dst] = bias[src]
    return wg, bias


TIE_CASES = {
    # k odd over expert twins: the k-th pick is always one expert of a tied pair
    "greedy_softmax_expert_twins": (dict(base="v2lite_t4096", T=700, d=256, E=64, I=128, k=5), "experts"),
    # topk_group odd over group twins: the last kept group is always one of a tied pair
    "group_max_group_twins": (dict(base="v2_t8192", T=700, d=256, E=64, I=128, k=6, n_group=8, topk_group=3),
                              "groups"),
    "group_sum_top2_bias_group_twins": (dict(base="v3_prefill_t16384", T=700, d=256, E=64, I=128, k=8,
                                             n_group=8, topk_group=3), "groups"),
    "group_sum_top2_bias_expert_twins": (dict(base="v3_prefill_t16384", T=700, d=256, E=64, I=128, k=7,
                                              n_group=8, topk_group=4), "experts"),
}


@pytest.mark.parametrize("name", list(TIE_CASES))
def test_exact_ties_go_to_the_lower_index(name):
    """Exact ties in the selection scores (and in the group scores) go to the
    lower expert (group) index, bit for bit: no near-tie excusal applies to a
    tie of identical fp32 values."""
    kw, twins = TIE_CASES[name]
    kw = dict(kw)
    wl = inputs.small_workload(W[kw.pop("base")], name=name, **kw)
    cfg = _lib.make_config(wl)
    x = inputs.make_tokens(wl)
    wg, bias = _twin_router(wl, twins)
    ws = torch.empty(_lib.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    idx = torch.empty((wl.T, wl.k), dtype=torch.int32, device="cuda")
    w = torch.empty((wl.T, wl.k), dtype=torch.float32, device="cuda")
    _lib.moe_gate_topk(cfg, x.cuda(), wg.cuda(), None if bias is None else bias.cuda(), idx, w, ws)
    assert _lib.moe_get_device_status(ws)[0] == _lib.MOE_OK
    r = orc.route(orc.gate_logits(f64(x), f64(wg)), None if bias is None else bias.numpy(), oracle_cfg(wl))
    gidx = _np(idx).astype(np.int64)
    sel = r.sel32
    # the twins' fp32 selection scores are identical on the oracle's side
    if twins == "experts":
        assert np.array_equal(sel[:, 0::2], sel[:, 1::2])
    exact_ties = 0
    for t in range(wl.T):
        assert set(gidx[t].tolist()) == set(r.idx[t].tolist()), (t, sorted(gidx[t]), sorted(r.idx[t]))
        if twins == "experts":
            picked = set(gidx[t].tolist())
            for e in range(0, wl.E, 2):
                if (e in picked) != (e + 1 in picked):
                    assert e in picked, (t, e)          # the lower twin wins
                    exact_ties += 1
    if twins == "experts":
        # k odd and every eligible set made of whole pairs: every token splits one pair
        assert exact_ties == wl.T
    og = np.take_along_axis(r.gates, np.argsort(r.idx, 1), 1)
    gg = np.take_along_axis(_np(w).astype(np.float64), np.argsort(gidx, 1), 1)
    assert (np.abs(gg - og) <= GATE_RTOL * np.abs(og)).all()


def test_forward_equals_staged_calls():
    """moe_forward == gate_topk -> permute -> grouped_swiglu -> combine, bit for bit."""
    wl = SMALL["v3_small_t333"]
    li = inputs.make_inputs(wl, "cuda")
    layer = MoELayer(wl, li, "cuda")
    out = layer.forward(li.x)
    o = layer.forward_staged(li.x)
    torch.cuda.synchronize()
    assert torch.equal(out, o["out"])


@pytest.mark.parametrize("name", ["v3_small_t3", "v3_small_t333"])
def test_fp8_forward_equals_staged_calls(name):
    """FP8 weights through the staged calls: moe_grouped_swiglu converts the
    caller's bf16 x_perm to the f16 rows the FP8 expert kernels take (the
    GEMV at T=3, the tensor-core kernel at T=333), and the outputs
    equal moe_forward's bit for bit."""
    wl = _fp8_copy(SMALL[name])
    li = inputs.make_inputs(wl, "cuda")
    layer = MoELayer(wl, li, "cuda")
    out = layer.forward(li.x)
    assert layer.device_status()[0] == _lib.MOE_OK
    o = layer.forward_staged(li.x)
    torch.cuda.synchronize()
    assert layer.device_status()[0] == _lib.MOE_OK
    assert torch.equal(out, o["out"])


def test_deterministic_across_runs():
    wl = SMALL["v2_small_t515"]
    li = inputs.make_inputs(wl, "cuda")
    layer = MoELayer(wl, li, "cuda")
    a = layer.forward(li.x).clone()
    b = layer.forward(li.x)
    assert torch.equal(a, b)


# ------------------------------------------------------------ stage by stage

@pytest.mark.parametrize("name", ["v2lite_t4096", "v2_t8192", "v3_prefill_t16384"])
def test_gate_topk_full_size(name):
    wl = W[name]
    li_x = inputs.make_tokens(wl)
    wg, bias = inputs.make_router(wl)
    cfg = _lib.make_config(wl)
    ws = torch.empty(_lib.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    idx = torch.empty((wl.T, wl.k), dtype=torch.int32, device="cuda")
    w = torch.empty((wl.T, wl.k), dtype=torch.float32, device="cuda")
    _lib.moe_gate_topk(cfg, li_x.cuda(), wg.cuda(), None if bias is None else bias.cuda(), idx, w, ws)
    assert _lib.moe_get_device_status(ws)[0] == _lib.MOE_OK
    r = orc.route(orc.gate_logits(f64(li_x), f64(wg)), None if bias is None else bias.numpy(), oracle_cfg(wl))
    n_near, n_differ = check_routing(_np(idx), _np(w), r, wl)
    print(name, {"near_tie_tokens": n_near, "near_tie_differ": n_differ})


@pytest.mark.parametrize("T,E,k,one_hot", [(1, 256, 8, None), (5, 12, 4, None), (17, 160, 6, 0),
                                           (32, 256, 8, None), (33, 256, 8, None), (128, 64, 6, None),
                                           (129, 64, 6, None), (4133, 256, 8, None), (300, 16, 1, 3),
                                           (777, 160, 6, 0)])
def test_permute_bit_exact(T, E, k, one_hot):
    wl = inputs.small_workload(W["v2lite_t4096"], name="perm", T=T, d=128, E=E, I=128, k=k)
    cfg = _lib.make_config(wl)
    idx = inputs.random_idx(T, E, k, seed=T + E, one_hot_expert=one_hot)
    x = inputs.random_rows(T, wl.d, seed=T)
    ws = torch.empty(_lib.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    dev = {n: torch.empty(s, dtype=torch.int32, device="cuda") for n, s in
           [("counts", (E,)), ("offsets", (E + 1,)), ("row2tok", (T * k,)), ("tok2row", (T, k))]}
    x_perm = torch.empty((T * k, wl.d), dtype=torch.bfloat16, device="cuda")
    _lib.moe_permute(cfg, x.cuda(), idx.cuda(), dev["counts"], dev["offsets"], dev["row2tok"], dev["tok2row"],
                     x_perm, ws)
    assert _lib.moe_get_device_status(ws)[0] == _lib.MOE_OK
    counts, offsets, row2tok, tok2row = orc.permutation(idx.numpy(), E)
    assert np.array_equal(_np(dev["counts"]), counts)
    assert np.array_equal(_np(dev["offsets"]), offsets)
    assert np.array_equal(_np(dev["row2tok"]), row2tok)
    assert np.array_equal(_np(dev["tok2row"]), tok2row)
    assert torch.equal(x_perm.cpu(), x[torch.from_numpy(row2tok)])


@pytest.mark.parametrize("T", [3, 100, 5000])
def test_permute_flags_out_of_range_expert(T):
    """An expert index outside [0, E) sets MOE_ERR_DEVICE_BOUNDS; that slot gets
    row -1 and no row, and the valid slots still form a dispatch of their own
    (one row each, grouped by expert in token order)."""
    E, k = 64, 6
    wl = inputs.small_workload(W["v2lite_t4096"], name="perm_bad", T=T, d=128, E=E, I=128, k=k)
    cfg = _lib.make_config(wl)
    idx = inputs.random_idx(T, E, k, seed=T, one_hot_expert=None)
    bad = [(0, 2, E), (T - 1, k - 1, -1)]
    for t, j, e in bad:
        idx[t, j] = e
    x = inputs.random_rows(T, wl.d, seed=T)
    ws = torch.empty(_lib.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    dev = {n: torch.full(s, -7, dtype=torch.int32, device="cuda") for n, s in
           [("counts", (E,)), ("offsets", (E + 1,)), ("row2tok", (T * k,)), ("tok2row", (T, k))]}
    x_perm = torch.zeros((T * k, wl.d), dtype=torch.bfloat16, device="cuda")
    _lib.moe_permute(cfg, x.cuda(), idx.cuda(), dev["counts"], dev["offsets"], dev["row2tok"], dev["tok2row"],
                     x_perm, ws)
    assert _lib.moe_get_device_status(ws)[0] == _lib.MOE_ERR_DEVICE_BOUNDS
    ix = idx.numpy()
    ok = (ix >= 0) & (ix < E)
    tok2row = _np(dev["tok2row"])
    assert (tok2row[~ok] == -1).all()
    assert np.array_equal(_np(dev["counts"]), np.bincount(ix[ok], minlength=E))
    n_rows = int(ok.sum())
    assert _np(dev["offsets"])[E] == n_rows
    rows = tok2row[ok]
    assert np.array_equal(np.sort(rows), np.arange(n_rows))
    row2tok = _np(dev["row2tok"])
    tt = np.nonzero(ok)[0]
    assert np.array_equal(row2tok[rows], tt)
    # grouped by expert, token order within an expert
    order = np.lexsort((tt, ix[ok]))
    assert np.array_equal(rows[order], np.arange(n_rows))
    assert torch.equal(x_perm.cpu()[torch.from_numpy(rows).long()], x[torch.from_numpy(tt)])


@pytest.mark.parametrize("name,seed", [("v3_small_t333", 1), ("v2lite_small_t1037", 2), ("v3_small_t1", 3)])
def test_grouped_swiglu_rows(name, seed):
    """Experts on seeded rows with seeded group sizes (empty experts, one big)."""
    wl = SMALL[name]
    cfg = _lib.make_config(wl)
    R = wl.T * wl.k
    counts = inputs.random_counts(wl.E, R, seed)
    offsets = torch.zeros(wl.E + 1, dtype=torch.int32)
    offsets[1:] = torch.cumsum(counts, 0)
    x_perm = inputs.random_rows(R, wl.d, seed)
    x = inputs.random_rows(wl.T, wl.d, seed + 100)
    w1, w3, w2, ws1, ws3, ws2 = inputs.make_experts(wl, "cuda")
    packed = torch.empty(_lib.moe_packed_size(cfg), dtype=torch.uint8, device="cuda")
    _lib.moe_prepack_experts(cfg, w1, w3, w2, ws1, ws3, ws2, packed)
    ws = torch.empty(_lib.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    y = torch.empty((R, wl.d), dtype=torch.float32, device="cuda")
    ys = torch.empty((wl.T, wl.d), dtype=torch.float32, device="cuda")
    _lib.moe_grouped_swiglu(cfg, x_perm.cuda(), offsets.cuda(), x.cuda(), packed, y, ys, ws)
    assert _lib.moe_get_device_status(ws)[0] == _lib.MOE_OK
    want = np.zeros((R, wl.d))
    xp = f64(x_perm)
    for e in range(wl.E):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if b > a:
            want[a:b] = orc.swiglu_ffn(xp[a:b], f64(w1[e]), f64(w3[e]), f64(w2[e]))
    assert orc.relative_error(f64(y), want) <= TOL["bf16"]
    want_s = orc.swiglu_ffn(f64(x), f64(ws1), f64(ws3), f64(ws2))
    assert orc.relative_error(f64(ys), want_s) <= TOL["bf16"]


@pytest.mark.parametrize("dtype,out_dtype", [("bf16", "f32"), ("bf16", "bf16"), ("f32", "f32")])
def test_combine(dtype, out_dtype):
    T, k, d = 301, 6, 256
    wl = inputs.small_workload(W["v2lite_t4096"], name="comb", T=T, d=d, E=16, I=128, k=k, act_dtype=dtype,
                               out_dtype=out_dtype)
    cfg = _lib.make_config(wl)
    y = inputs.random_rows(T * k, d, 11, torch.float32)      # expert outputs are fp32
    ys = inputs.random_rows(T, d, 12, torch.float32)
    g = inputs.random_gates(T, k, 13)
    tok2row = torch.randperm(T * k, generator=torch.Generator().manual_seed(14)).view(T, k).to(torch.int32)
    ws = torch.empty(_lib.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    out = torch.empty((T, d), dtype=inputs.torch_dtype(out_dtype), device="cuda")
    _lib.moe_combine(cfg, y.cuda(), ys.cuda(), tok2row.cuda(), g.cuda(), out, ws)
    assert _lib.moe_get_device_status(ws)[0] == _lib.MOE_OK
    want = orc.combine(f64(y), f64(ys), tok2row.numpy().astype(np.int64), g.double().numpy())
    assert orc.relative_error(f64(out), want) <= TOL[out_dtype]


def test_out_of_range_expert_is_flagged_not_faulted():
    """An idx entry outside [0,E) is skipped by the permutation and reported
    through the status word; the context stays usable."""
    T, E, k = 64, 16, 2
    wl = inputs.small_workload(W["v2lite_t4096"], name="bad", T=T, d=128, E=E, I=128, k=k)
    cfg = _lib.make_config(wl)
    idx = inputs.random_idx(T, E, k, seed=5)
    idx[7, 1] = E + 3
    ws = torch.empty(_lib.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    row2tok = torch.full((T * k,), -1, dtype=torch.int32, device="cuda")
    bufs = [torch.zeros(s, dtype=torch.int32, device="cuda") for s in [(E,), (E + 1,), (T, k)]]
    x_perm = torch.zeros((T * k, wl.d), dtype=torch.bfloat16, device="cuda")
    _lib.moe_permute(cfg, inputs.random_rows(T, wl.d, 1).cuda(), idx.cuda(), bufs[0], bufs[1], row2tok, bufs[2],
                     x_perm, ws)
    code, word = _lib.moe_get_device_status(ws)
    assert code == _lib.MOE_ERR_DEVICE_BOUNDS and word != 0
    assert int(bufs[0].sum()) == T * k - 1
    # the context is still fine
    torch.cuda.synchronize()
    assert float(torch.ones(4, device="cuda").sum()) == 4.0


# ------------------------------------------------------------ load balancing

@pytest.mark.parametrize("case", ["forward_counts", "synthetic"])
def test_balance_update(case):
    """moe_balance_update == the oracle's balancing step: the float32 bias bit
    for bit, the load statistics within 1e-6 relative."""
    gamma = 0.001
    if case == "forward_counts":
        wl = SMALL["v3_small_t333"]
        li = inputs.make_inputs(wl, "cuda")
        _, _, _, _, counts = run_layer(wl, li)
        bias0 = li.bias.float().clone()
    else:
        wl = inputs.small_workload(W["v3_prefill_t16384"], name="bal", T=96, d=512, E=64, I=128)
        c = torch.randint(0, 30, (wl.E,), generator=torch.Generator().manual_seed(3), dtype=torch.int32)
        c[5] = int(c.sum() - c[5]) // (wl.E - 1)          # some experts at or near the mean
        tot = int(c.sum())
        c[7] = tot // wl.E if tot % wl.E == 0 else c[7]
        counts = c.cuda()
        bias0 = (torch.randn(wl.E, generator=torch.Generator().manual_seed(4)) * 0.1).float().cuda()
    cfg = _lib.make_config(wl)
    bias = bias0.clone()
    stats = torch.zeros(4, dtype=torch.float32, device="cuda")
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    _lib.moe_balance_update(cfg, counts, bias, gamma, stats, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    want_b, want_s = orc.balance_update(_np(counts), _np(bias0), gamma)
    assert np.array_equal(_np(bias), want_b)
    got_s = _np(stats)[:3].astype(np.float64)
    assert np.allclose(got_s, want_s, rtol=1e-6, atol=1e-9), (got_s, want_s)


# ------------------------------------------------------------ FP8 expert weights

def _fp8_copy(wl):
    return inputs.small_workload(wl, name=wl.name + "_fp8", expert_w_dtype="fp8")


FP8_STAGE = 128 * 128 + 2 * 128 * 4   # one stage image: 128 x 128 e4m3 values, then int32 scale exponents [2][128]


def _fp8_tiled_bytes(rows, cols):
    return (rows // 128 + 1) * (cols // 128) * FP8_STAGE


def _decode_fp8_tiles(packed, off, rows, cols):
    """e4m3 values [rows, cols] and scales [rows, cols / 64] (float64) of one
    matrix stored as stage images: 128-row tiles of cols / 128 stages, each a
    128-byte-swizzled 128 x 128 byte image (16-byte chunk c of row r at chunk
    position c ^ (r % 8)) followed by its scale exponents [2][128] (int32, the
    scale is 2^e); one zero tile follows the last row."""
    nst, tiles = cols // 128, rows // 128 + 1
    blob = packed[off: off + tiles * nst * FP8_STAGE].view(tiles, nst, FP8_STAGE)
    img = blob[:, :, :128 * 128].reshape(tiles, nst, 128, 8, 16)
    r = torch.arange(128, device=blob.device)
    pos = torch.arange(8, device=blob.device)[None, :] ^ (r[:, None] % 8)          # [128 rows, 8 logical chunks]
    logical = img[:, :, r[:, None], pos, :]                                            # [tiles, nst, 128, 8, 16]
    q = logical.permute(0, 2, 1, 3, 4).reshape(tiles * 128, cols).contiguous()
    sc = blob[:, :, 128 * 128:].contiguous().view(torch.int32).view(tiles, nst, 2, 128)
    sc = sc.permute(0, 3, 1, 2).reshape(tiles * 128, cols // 64)
    assert int(q[rows:].count_nonzero()) == 0 and int(sc[rows:].count_nonzero()) == 0   # the zero tile
    qf = q[:rows].view(torch.float8_e4m3fn).to(torch.float64).cpu().numpy()
    return qf, np.ldexp(1.0, sc[:rows].cpu().numpy().astype(np.int64))


def test_fp8_prepack_matches_oracle_quantization():
    """moe_prepack_experts with FP8 weights: e4m3 bytes and block scales of every
    matrix bit for bit equal to the oracle's block quantisation, decoded from
    the stage-image layout the expert GEMM streams."""
    wl = _fp8_copy(SMALL["v3_small_t333"])
    cfg = _lib.make_config(wl)
    w1, w3, w2, ws1, ws3, ws2 = inputs.make_experts(wl, "cuda")
    packed = torch.empty(_lib.moe_packed_size(cfg), dtype=torch.uint8, device="cuda")
    _lib.moe_prepack_experts(cfg, w1, w3, w2, ws1, ws3, ws2, packed)
    torch.cuda.synchronize()
    E, I, d, Is = wl.E, wl.I, wl.d, wl.I_s
    al = lambda v: (v + 255) // 256 * 256
    o_w13 = 0
    o_w2 = al(o_w13 + _fp8_tiled_bytes(E * 2 * I, d))
    o_w13s = al(o_w2 + _fp8_tiled_bytes(E * d, I))
    o_w2s = al(o_w13s + _fp8_tiled_bytes(2 * Is, d))
    o_eref = al(o_w2s + _fp8_tiled_bytes(d, Is))
    assert al(o_eref + (E + 1) * 3 * 4) == packed.numel()
    eref = packed[o_eref: o_eref + (E + 1) * 3 * 4].view(torch.int32).view(E + 1, 3).cpu().numpy()
    q, s = _decode_fp8_tiles(packed, o_w2, E * d, I)
    wq, ws = orc.quantize_fp8_blocks(f64(w2).reshape(E * d, I))
    assert np.array_equal(q, wq) and np.array_equal(s, ws)
    # reference exponents: the largest block exponent of each matrix
    assert np.array_equal(eref[:E, 2], np.log2(ws).reshape(E, -1).max(1))
    q, s = _decode_fp8_tiles(packed, o_w2s, d, Is)
    wq, ws = orc.quantize_fp8_blocks(f64(ws2))
    assert np.array_equal(q, wq) and np.array_equal(s, ws)
    assert eref[E, 2] == np.log2(ws).max()
    # W13: rows in the 16-row interleave (16 W1 rows, then the 16 W3 rows of the same units)
    q, s = _decode_fp8_tiles(packed, o_w13, E * 2 * I, d)
    w13 = torch.stack([w1, w3], 1).view(E, 2, I // 16, 16, d).transpose(1, 2).reshape(E * 2 * I, d)
    wq, ws = orc.quantize_fp8_blocks(f64(w13))
    assert np.array_equal(q, wq) and np.array_equal(s, ws)
    for m, w in ((0, w1), (1, w3)):
        _, ws_m = orc.quantize_fp8_blocks(f64(w).reshape(E * I, d))
        assert np.array_equal(eref[:E, m], np.log2(ws_m).reshape(E, -1).max(1))
        _, ws_s = orc.quantize_fp8_blocks(f64((ws1, ws3)[m]))
        assert eref[E, m] == np.log2(ws_s).max()


def test_fp8_layer_flags_activations_beyond_f16():
    """An FP8 layer takes its token rows as f16: an input value beyond the f16
    range is reported (MOE_ERR_DEVICE_RANGE), while the bf16 layer takes it."""
    base = SMALL["v3_small_t333"]
    for wl, want in ((_fp8_copy(base), _lib.MOE_ERR_DEVICE_RANGE), (base, _lib.MOE_OK)):
        li = inputs.make_inputs(wl, "cuda")
        x = li.x.clone()
        x[17, 5] = 1.0e5
        layer = MoELayer(wl, li, "cuda")
        layer.forward(x)
        code, word = layer.device_status()
        assert code == want, (wl.name, _lib.moe_status_string(code), word)
        layer.forward(li.x)
        assert layer.device_status()[0] == _lib.MOE_OK


def _dq(t):
    """FP8 block dequantisation of one matrix (what the FP8 layer computes with)."""
    return orc.fp8_dequantized(f64(t))


def _dequantized_accessor(li):
    """Per-expert dequantised float64 weights, made lazily one expert at a time
    (a full-size layer's weights would not fit in host memory as float64)."""
    cache = {}

    def get(e):
        if e not in cache:
            cache.clear()
            cache[e] = (_dq(li.w1[e]), _dq(li.w3[e]), _dq(li.w2[e]))
        return cache[e]
    return get


def _dequantized_shared(li):
    if li.wl.n_shared == 0:
        return None
    return _dq(li.ws1), _dq(li.ws3), _dq(li.ws2)


# FP8 decode-sized cases whose tiles have an odd number of 128-deep stages (d = I = 384)
FP8_ODD = {
    "v3_odd_t5": inputs.small_workload(W["v3_prefill_t16384"], name="v3_odd_t5", T=5, d=384, E=64, I=384,
                                       n_group=8, topk_group=4),
    "v3_odd_t9": inputs.small_workload(W["v3_prefill_t16384"], name="v3_odd_t9", T=9, d=384, E=64, I=384,
                                       n_group=8, topk_group=4),
    "v3_odd_t72": inputs.small_workload(W["v3_prefill_t16384"], name="v3_odd_t72", T=72, d=384, E=64, I=384,
                                        n_group=8, topk_group=4),
    # the GEMV's largest batch with the decode layers' skewed bias: 512 rows
    # over 64 experts (8 on average) and the shared expert's 64, in items of 8
    "v3_gemv_t64_zipf": inputs.small_workload(W["v3_prefill_t16384"], name="v3_gemv_t64_zipf", T=64, d=384,
                                              E=64, I=384, n_group=8, topk_group=4, bias="zipf"),
    "v3_odd_t40": inputs.small_workload(W["v3_prefill_t16384"], name="v3_odd_t40", T=40, d=384, E=64, I=384,
                                        n_group=8, topk_group=4),
    # batches of at most 64 tokens take the FP8 GEMV (warp-level MMAs, 8 token
    # rows per item): one item per group, and one without a shared expert
    "v3_gemv_t8": inputs.small_workload(W["v3_prefill_t16384"], name="v3_gemv_t8", T=8, d=384, E=64, I=384,
                                        n_group=8, topk_group=4),
    "v3_gemv_t4": inputs.small_workload(W["v3_prefill_t16384"], name="v3_gemv_t4", T=4, d=384, E=64, I=384,
                                        n_group=8, topk_group=4),
    "v2lite_gemv_t2_noshared": inputs.small_workload(W["v2lite_t4096"], name="v2lite_gemv_t2_noshared", T=2, d=256,
                                                     E=16, I=256, k=6, n_shared=0),
}


@pytest.mark.parametrize("name", ["v3_small_t333", "v2lite_small_t1037", "v3_small_t1", "v3_small_t3",
                                  "v3_small_t1100", "v3_odd_t5", "v3_odd_t9", "v3_odd_t40", "v3_odd_t72",
                                  "v3_gemv_t64_zipf", "v3_gemv_t8", "v3_gemv_t4", "v2lite_gemv_t2_noshared"])
def test_fp8_layer_matches_oracle_on_dequantized_weights(name):
    wl = _fp8_copy(SMALL[name] if name in SMALL else FP8_ODD[name])
    li = inputs.make_inputs(wl, "cuda")
    _, out, idx, w, counts = run_layer(wl, li)
    r = oracle_route(li, wl)
    check_routing(_np(idx), _np(w), r, wl)
    keep = np.array([np.array_equal(np.sort(_np(idx)[t]), np.sort(r.idx[t])) for t in range(wl.T)])
    toks = np.arange(wl.T)[keep]
    want = orc.experts_forward(f64(li.x)[toks], r.idx[toks], r.gates[toks], _dequantized_accessor(li),
                               _dequantized_shared(li), wl.E)
    assert orc.relative_error(f64(out)[toks], want) <= TOL["bf16"]


@pytest.mark.parametrize("name", ["v3_decode_t1", "v3_decode_t8", "v3_decode_t64"])
def test_fp8_full_size_decode(name):
    wl = _fp8_copy(W[name])
    li = inputs.make_inputs(wl, "cuda")
    _, out, idx, w, counts = run_layer(wl, li)
    r = oracle_route(li, wl)
    check_routing(_np(idx), _np(w), r, wl)
    sample = np.sort(np.random.default_rng(7).choice(wl.T, min(wl.T, 12), replace=False))
    keep = np.array([np.array_equal(np.sort(_np(idx)[t]), np.sort(r.idx[t])) for t in sample])
    toks = sample[keep]
    want = orc.experts_forward(f64(li.x)[toks], r.idx[toks], r.gates[toks], _dequantized_accessor(li),
                               _dequantized_shared(li), wl.E)
    assert orc.relative_error(f64(out)[toks], want) <= TOL["bf16"]
    del li, out
    torch.cuda.empty_cache()
