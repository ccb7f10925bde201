"""Test-side adapters: a workload (seeded input recipe) as the oracle's config,
and torch tensors as float64 numpy arrays for the oracle."""
import numpy as np
import torch

from oracle import moe_oracle as orc


def oracle_cfg(wl, **over) -> "orc.OracleConfig":
    kw = dict(T=wl.T, d=wl.d, E=wl.E, I=wl.I, k=wl.k, n_shared=wl.n_shared,
              score_fn=wl.score_fn, topk_method=wl.topk_method, n_group=wl.n_group,
              topk_group=wl.topk_group, group_score=wl.group_score, group_top=wl.group_top,
              norm_topk=wl.norm_topk, routed_scaling_factor=wl.routed_scaling_factor)
    kw.update(over)
    return orc.OracleConfig(**kw)


def f64(t) -> np.ndarray:
    """Exact widening of a (bf16/fp32) tensor, on whatever device, to float64 numpy."""
    if t is None:
        return None
    return t.detach().to("cpu").to(torch.float64).numpy()


def expert_accessor(w1, w3, w2):
    """Per-expert float64 weights, fetched lazily (device tensors stay on device)."""
    cache = {}

    def get(e):
        if e not in cache:
            cache.clear()
            cache[e] = (f64(w1[e]), f64(w3[e]), f64(w2[e]))
        return cache[e]
    return get
