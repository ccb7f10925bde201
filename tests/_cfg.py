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


def output_error(got, want, out_dtype: str) -> float:
    """max |got - want| / RMS(want), the layer's acceptance measure.  A bf16-
    stored output also carries its own rounding, at most half a bf16 ulp
    (2^-8 of the value, 8 significant bits), which the fp64 oracle does not
    have; that allowance is taken off each element first, so the budget
    applies to the computation alone."""
    from oracle import moe_oracle as orc
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    if out_dtype != "bf16":
        return orc.relative_error(got, want)
    allow = 2.0 ** -8 * np.maximum(np.abs(got), np.abs(want)) * 1.01
    excess = np.maximum(np.abs(got - want) - allow, 0.0)
    return orc.relative_error(want + excess, want)
