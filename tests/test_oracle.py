"""The fp64 oracle against its pins (CPU only)."""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import moe_oracle as orc
from mixture_experts_layer_85_b300 import inputs
from tests import oracle_pins
from tests._cfg import oracle_cfg

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin()


def test_v3_workloads_match_v3_table():
    g = json.load(open(os.path.join(GOLDEN, "v3_moe_table.json")))
    for name in ["v3_prefill_t16384"] + [f"v3_decode_t{T}" for T in inputs.DECODE_T]:
        wl = inputs.WORKLOADS[name]
        assert wl.d == g["hidden_size"] and wl.E == g["n_routed_experts"]
        assert wl.k == g["num_experts_per_tok"] and wl.I == g["moe_intermediate_size"]
        assert wl.n_shared == g["n_shared_experts"]
        assert wl.E + wl.n_shared == g["experts_per_layer"] and wl.k + wl.n_shared == g["active_experts_per_layer"]


def test_tiny_workload_matches_moe_defaults():
    g = json.load(open(os.path.join(GOLDEN, "v2_moe_defaults.json")))
    wl = inputs.WORKLOADS["tiny_fp32_t128"]
    assert (wl.E, wl.k, wl.n_shared) == (g["n_routed_experts"], g["num_experts_per_tok"], g["n_shared_experts"])
    assert wl.I_s == wl.n_shared * wl.I


def test_decode_bias_calibration():
    """The stored Zipf strength reproduces the 50% top-10% share on the oracle."""
    g = json.load(open(os.path.join(GOLDEN, "decode_bias.json")))
    assert inputs.DECODE_ZIPF_BETA == g["beta"]
    wl = inputs.WORKLOADS["v3_decode_t512"]
    gen = torch.Generator().manual_seed(g["calibration_seed"])
    x = torch.randn((g["calibration_tokens"], wl.d), generator=gen).to(torch.bfloat16)
    wg, bias = inputs.make_router(wl)
    r = orc.route(orc.gate_logits(x.double().numpy(), wg.double().numpy()), bias.numpy(),
                  oracle_cfg(wl, T=x.shape[0]))
    n_top = math.ceil(0.1 * wl.E)
    share = np.sort(r.counts)[::-1][:n_top].sum() / r.counts.sum()
    assert abs(share - 0.5) <= 0.03


def test_tiny_workload_end_to_end_invariants():
    """The fp32 reference workload through the oracle: counts, gates, near ties."""
    wl = inputs.WORKLOADS["tiny_fp32_t128"]
    li = inputs.make_inputs(wl, "cpu")
    cfg = oracle_cfg(wl)
    out, r = orc.moe_forward(li.x.double().numpy(), li.wg.double().numpy(), None,
                             orc.stacked_experts(li.w1.double().numpy(), li.w3.double().numpy(),
                                                 li.w2.double().numpy()),
                             (li.ws1.double().numpy(), li.ws3.double().numpy(), li.ws2.double().numpy()), cfg)
    assert out.shape == (wl.T, wl.d) and np.isfinite(out).all()
    assert r.counts.sum() == wl.T * wl.k
    assert not r.near_tie.any()
    assert (r.gates.sum(1) <= 1.0 + 1e-12).all()


def test_near_tie_flag():
    cfg = orc.OracleConfig(T=2, d=1, E=4, I=1, k=1, n_shared=0, score_fn="sigmoid")
    logits = np.array([[0.3, 0.3 + 1e-9, -1.0, -2.0], [0.3, 0.5, -1.0, -2.0]])
    r = orc.route(logits, None, cfg)
    assert r.near_tie.tolist() == [True, False]
    assert orc.is_valid_selection([0], r.sel32[0], cfg) and orc.is_valid_selection([1], r.sel32[0], cfg)
    assert not orc.is_valid_selection([0], r.sel32[1], cfg)


def test_backward_parts_agree_with_the_whole():
    """The partial forms the full-size GPU test uses: dx without the weight
    gradients, and one expert's gradients from its own rows, equal the full
    backward's (same arithmetic, bit for bit)."""
    wl = inputs.small_workload(inputs.WORKLOADS["v3_prefill_t16384"], name="v3_parts", T=19, d=32, E=16, I=8,
                               n_group=4, topk_group=2)
    li = inputs.make_inputs(wl, "cpu")
    cfg = oracle_cfg(wl)
    f = lambda t: t.double().numpy()
    bias = li.bias.float().numpy()
    shared = (f(li.ws1), f(li.ws3), f(li.ws2))
    dout = np.random.default_rng(3).standard_normal((wl.T, wl.d))
    full = orc.moe_backward(f(li.x), f(li.wg), bias, f(li.w1), f(li.w3), f(li.w2), shared, dout, cfg)
    part = orc.moe_backward(f(li.x), f(li.wg), bias, f(li.w1), f(li.w3), f(li.w2), shared, dout, cfg,
                            weight_grads=False)
    assert part["dw1"] is None and np.array_equal(part["dx"], full["dx"])
    r = full["routing"]
    gates = orc.gate_values(r.scores, r.idx, cfg)
    for e in np.unique(r.idx):
        _, _, _, _, g1, g3, g2 = orc.expert_backward(f(li.x), dout, r.idx, gates, int(e), f(li.w1)[e],
                                                     f(li.w3)[e], f(li.w2)[e])
        assert np.array_equal(g1, full["dw1"][e]) and np.array_equal(g3, full["dw3"][e])
        assert np.array_equal(g2, full["dw2"][e])
