"""Writes tests/golden/decode_bias.json: the strength beta of the Zipf(1.2)
rank bias used by the V3-shaped decode workloads.

The decode workload asks for routing that follows Zipf(s=1.2) over the experts
with the 10% most-loaded experts taking about half of all assignments.  A bias
b_e = -1.2 * beta * ln(rank_e) is added to the sigmoid affinities (selection
only, as the V3 page's auxiliary-loss-free balancing does); beta is bisected so
that, on a seeded calibration batch of 4096 tokens routed by the fp64 oracle,
the top ceil(0.1*E) experts receive 50% of the T*k assignments.

Runs on the CPU and calls only the oracle (plus the seeded input generator):
    python tests/golden/calibrate_decode_bias.py
"""
import json
import math
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from oracle import moe_oracle as orc  # noqa: E402
from mixture_experts_layer_85_b300 import inputs  # noqa: E402

TARGET_SHARE = 0.50
CALIB_T = 4096


def top_share(counts: np.ndarray, frac: float = 0.1) -> float:
    n_top = int(math.ceil(frac * counts.size))
    return float(np.sort(counts)[::-1][:n_top].sum() / counts.sum())


def main():
    wl = inputs.WORKLOADS["v3_decode_t512"]
    cfg = orc.OracleConfig(T=CALIB_T, d=wl.d, E=wl.E, I=wl.I, k=wl.k, n_shared=wl.n_shared,
                           score_fn=wl.score_fn, topk_method=wl.topk_method, n_group=wl.n_group,
                           topk_group=wl.topk_group, group_score=wl.group_score,
                           group_top=wl.group_top, norm_topk=wl.norm_topk,
                           routed_scaling_factor=wl.routed_scaling_factor)
    g = torch.Generator().manual_seed(inputs.SEED_CALIB_X)
    x = torch.randn((CALIB_T, wl.d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    wg, _ = inputs.make_router(wl)
    logits = orc.gate_logits(x.double().numpy(), wg.double().numpy())

    def share(beta):
        b = inputs.decode_rank_bias(wl.E, beta).numpy()
        r = orc.route(logits, b, cfg)
        return top_share(r.counts), r

    lo, hi = 0.0, 1.0
    while share(hi)[0] < TARGET_SHARE:
        hi *= 2.0
    for _ in range(40):
        mid = 0.5 * (lo + hi)
        if share(mid)[0] < TARGET_SHARE:
            lo = mid
        else:
            hi = mid
    beta = 0.5 * (lo + hi)
    s, r = share(beta)
    touched = {T: int(np.unique(r.idx[:T]).size) for T in inputs.DECODE_T}
    out = {
        "beta": beta,
        "zipf_s": inputs.DECODE_ZIPF_S,
        "calibration_tokens": CALIB_T,
        "calibration_seed": inputs.SEED_CALIB_X,
        "top10pct_share": s,
        "experts_touched_by_first_T_calibration_tokens": touched,
        "how": "bisection of beta on the oracle's routing (tests/golden/calibrate_decode_bias.py)",
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "decode_bias.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
    print(json.dumps(out))


if __name__ == "__main__":
    main()
