"""moe_backward (the layer's gradients) against the oracle's backward, which is
pinned by central finite differences of the fp64 forward.

The backward recomputes the routing with the forward's kernels; the test reads
that choice through moe_gate_topk (same kernels, same result), checks it
against the oracle's routing rules, and runs the oracle backward on the same
choice.  Every gradient is compared element by element.  The library rounds
the operands of each product to bf16 (H, the gate-weighted upstream rows, dG
and dU; x and the weights are bf16 already): 2^-9 relative each, two to three
on every path, so an element of a sum over n rows is off by about
2^-8 * sum_r |term_r|, a few times 2^-8 of the element when the terms cancel.
Acceptance: the relative Frobenius error ||got - ref|| / ||ref|| <= TOL_FRO of
every gradient and of every used expert's slice (measured: 1.6e-3 to 2.4e-3,
the 2^-9 level), and, as a coarse bound on single elements of dx, dW_g and the
shared expert's gradients, max |got - ref| / RMS(ref) <= TOL_MAX.  A routed
expert's weight gradient is a sum over its few rows (one row at T=1: an outer
product), whose largest elements sit too far out in the tail of the RMS for
that bound; its elements are covered by the per-expert Frobenius bound."""
import numpy as np
import pytest
import torch

from mixture_experts_layer_85_b300 import _lib, inputs
from oracle import moe_oracle as orc
from tests._cfg import f64, oracle_cfg

pytestmark = pytest.mark.gpu

TOL_FRO = 1e-2
TOL_MAX = 1e-1
W = inputs.WORKLOADS
CASES = {
    # softmax greedy, fp32 gate weight, two shared experts
    "v2lite_bwd_t37": inputs.small_workload(W["v2lite_t4096"], name="v2lite_bwd_t37", T=37, d=256, E=16, I=128, k=6,
                                            n_shared=2),
    # softmax group-limited (max), scale 16
    "v2_bwd_t29": inputs.small_workload(W["v2_t8192"], name="v2_bwd_t29", T=29, d=256, E=32, I=128, n_group=8,
                                        topk_group=3),
    # sigmoid + bias, group-limited sum of top-2, renormalised, scale 2.5
    "v3_bwd_t53": inputs.small_workload(W["v3_prefill_t16384"], name="v3_bwd_t53", T=53, d=256, E=32, I=128,
                                        n_group=8, topk_group=4),
    "v3_bwd_t53_bf16out": inputs.small_workload(W["v3_prefill_t16384"], name="v3_bwd_t53_bf16out", T=53, d=256,
                                                E=32, I=128, n_group=8, topk_group=4, out_dtype="bf16"),
    # one token: most experts receive no row (their gradients are exact zeros)
    "v3_bwd_t1": inputs.small_workload(W["v3_decode_t1"], name="v3_bwd_t1", T=1, d=256, E=32, I=128, n_group=8,
                                       topk_group=4),
    # the V3 expert shape (d 7168, I 2048): full 256-row weight tiles, many 128-row
    # reduction stages per expert, shared expert and router at their real widths
    "v3_bwd_fullshape_t256": inputs.small_workload(W["v3_prefill_t16384"], name="v3_bwd_fullshape_t256", T=256,
                                                   E=8, k=4, n_group=4, topk_group=2),
}


def _run(wl):
    li = inputs.make_inputs(wl, "cuda")
    cfg = _lib.make_config(wl)
    g = torch.Generator().manual_seed(4242)
    dout = torch.randn((wl.T, wl.d), generator=g).to(torch.bfloat16 if wl.out_dtype == "bf16" else torch.float32)
    dout = dout.cuda()
    E, I, d, Is = wl.E, wl.I, wl.d, wl.I_s
    f32 = dict(dtype=torch.float32, device="cuda")
    outs = {"dx": torch.empty((wl.T, d), **f32), "dwg": torch.empty((E, d), **f32),
            "dw1": torch.full((E, I, d), float("nan"), **f32), "dw3": torch.full((E, I, d), float("nan"), **f32),
            "dw2": torch.full((E, d, I), float("nan"), **f32), "dws1": torch.empty((Is, d), **f32),
            "dws3": torch.empty((Is, d), **f32), "dws2": torch.empty((d, Is), **f32)}
    ws = torch.empty(_lib.moe_backward_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    _lib.moe_backward(cfg, li.x, li.wg, li.bias, li.w1, li.w3, li.w2, li.ws1, li.ws3, li.ws2, dout,
                      outs["dx"], outs["dwg"], outs["dw1"], outs["dw3"], outs["dw2"], outs["dws1"], outs["dws3"],
                      outs["dws2"], ws)
    torch.cuda.synchronize()
    code, word = _lib.moe_get_device_status(ws)
    assert code == _lib.MOE_OK, (_lib.moe_status_string(code), word)
    # the routing the backward used (same kernels)
    idx = torch.empty((wl.T, wl.k), dtype=torch.int32, device="cuda")
    w = torch.empty((wl.T, wl.k), dtype=torch.float32, device="cuda")
    fws = torch.empty(_lib.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    _lib.moe_gate_topk(cfg, li.x, li.wg, li.bias, idx, w, fws)
    torch.cuda.synchronize()
    return li, dout, outs, idx.cpu().numpy().astype(np.int64)


@pytest.mark.parametrize("name", list(CASES))
def test_backward_matches_oracle(name):
    wl = CASES[name]
    li, dout, outs, gidx = _run(wl)
    cfg = oracle_cfg(wl)
    bias = None if li.bias is None else li.bias.float().cpu().numpy()
    r = orc.route(orc.gate_logits(f64(li.x), f64(li.wg)), bias, cfg)
    same = (np.sort(gidx, 1) == np.sort(r.idx, 1)).all(1)
    assert (same | r.near_tie).all(), "expert sets differ on non-tie tokens"
    for t in np.nonzero(~same)[0]:
        assert orc.is_valid_selection(gidx[t], r.sel32[t], cfg), t
    shared = (f64(li.ws1), f64(li.ws3), f64(li.ws2)) if wl.n_shared else None
    ref = orc.moe_backward(f64(li.x), f64(li.wg), bias, f64(li.w1), f64(li.w3), f64(li.w2), shared, f64(dout), cfg,
                           idx_override=gidx)

    def fro(got, want):
        return float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-300))

    used = np.zeros(wl.E, bool)
    used[np.unique(gidx)] = True
    errs = {}
    for key in ("dx", "dwg", "dw1", "dw3", "dw2", "dws1", "dws3", "dws2"):
        if ref[key] is None:
            continue
        got = f64(outs[key])
        assert np.isfinite(got).all(), key
        errs[key] = (fro(got, ref[key]), orc.relative_error(got, ref[key]))
        if key in ("dw1", "dw3", "dw2"):
            worst = max(fro(got[e], ref[key][e]) for e in np.nonzero(used)[0])
            assert worst <= TOL_FRO, (key, "per expert", worst)
            # experts without a routed row: their gradients are exact zeros
            assert not got[~used].any(), key
    print(name, {k: f"fro {a:.1e} max {b:.1e}" for k, (a, b) in errs.items()})
    for key, (a, b) in errs.items():
        assert a <= TOL_FRO, (key, a)
        if key not in ("dw1", "dw3", "dw2"):
            assert b <= TOL_MAX, (key, b)


class _PerExpert:
    """w[e] of a device tensor as float64 numpy, fetched when asked for."""

    def __init__(self, t):
        self.t = t

    def __getitem__(self, e):
        return f64(self.t[e])


def test_backward_full_size_sampled():
    """V3 prefill at full size (T=16384, E=256, d=7168, I=2048, top-8): every
    gradient the oracle can form from part of the batch.  dx of sampled tokens
    depends on those tokens alone; a routed expert's weight gradients are sums
    over the rows routed to it (the most loaded expert, the least loaded one
    with rows, and a row count that is not a multiple of 128); the shared
    expert's are sums over every token (one fp64 pass over the batch).  Experts
    without rows must get exact zeros, and no gradient may hold a NaN.  dW_g
    sums dL/dlogits of every token, which needs every expert output of the
    batch in fp64: it is compared at the reduced sizes above, including the V3
    expert shape."""
    wl = W["v3_prefill_t16384"]
    li, dout, outs, gidx = _run(wl)
    cfg = oracle_cfg(wl)
    bias = None if li.bias is None else li.bias.float().cpu().numpy()
    x = f64(li.x)
    r = orc.route(orc.gate_logits(x, f64(li.wg)), bias, cfg)
    same = (np.sort(gidx, 1) == np.sort(r.idx, 1)).all(1)
    assert (same | r.near_tie).all(), "expert sets differ on non-tie tokens"
    for t in np.nonzero(~same)[0]:
        assert orc.is_valid_selection(gidx[t], r.sel32[t], cfg), t
    for key in ("dx", "dwg", "dw1", "dw3", "dw2", "dws1", "dws3", "dws2"):
        assert not torch.isnan(outs[key]).any(), key
    counts = np.bincount(gidx.ravel(), minlength=wl.E)
    unused = torch.from_numpy(counts == 0).cuda()
    for key in ("dw1", "dw3", "dw2"):
        assert not outs[key][unused].any(), key

    def fro(got, want):
        return float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-300))

    errs = {}
    dout64 = f64(dout)
    # dx of sampled tokens (token-local: their own experts and router row)
    sample = np.sort(np.random.default_rng(11).choice(wl.T, 8, replace=False))
    ref = orc.moe_backward(x[sample], f64(li.wg), bias, _PerExpert(li.w1), _PerExpert(li.w3), _PerExpert(li.w2),
                           (f64(li.ws1), f64(li.ws3), f64(li.ws2)), dout64[sample], cfg,
                           idx_override=gidx[sample], weight_grads=False)
    got = f64(outs["dx"][torch.from_numpy(sample).cuda()])
    errs["dx"] = (fro(got, ref["dx"]), orc.relative_error(got, ref["dx"]))
    # routed experts' weight gradients over all their rows
    used = np.nonzero(counts)[0]
    ragged = [e for e in used if counts[e] % 128 != 0]
    picks = sorted({int(used[np.argmax(counts[used])]), int(used[np.argmin(counts[used])]), int(ragged[0])})
    gates = orc.gate_values(r.scores, gidx, cfg)
    for e in picks:
        _, _, _, _, g1, g3, g2 = orc.expert_backward(x, dout64, gidx, gates, e, f64(li.w1[e]), f64(li.w3[e]),
                                                     f64(li.w2[e]))
        for key, want in (("dw1", g1), ("dw3", g3), ("dw2", g2)):
            errs[f"{key}[{e}] ({counts[e]} rows)"] = (fro(f64(outs[key][e]), want), None)
    # the shared expert over the whole batch
    _, g1, g3, g2 = orc.swiglu_backward(x, f64(li.ws1), f64(li.ws3), f64(li.ws2), dout64)
    for key, want in (("dws1", g1), ("dws3", g3), ("dws2", g2)):
        got = f64(outs[key])
        errs[key] = (fro(got, want), orc.relative_error(got, want))
    print({k: f"fro {a:.1e}" + ("" if b is None else f" max {b:.1e}") for k, (a, b) in errs.items()})
    for key, (a, b) in errs.items():
        assert a <= TOL_FRO, (key, a)
        if b is not None:
            assert b <= TOL_MAX, (key, b)
