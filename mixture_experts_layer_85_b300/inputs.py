"""Seeded synthetic workloads for the DeepSeekMoE layer forward.

This module only names layer shapes and draws random tensors; it holds none of
the layer's arithmetic.  Tests feed the same bytes to the CUDA library and to
the CPU oracle, and the benchmark draws its inputs here.

Shapes come from the pages:
  * ``tiny_fp32_t128`` - the ``MoE`` constructor defaults of the DeepSeek-V2
    walkthrough (12 routed experts, top-4, 2 shared experts) at d=64, I=32.
  * ``v2lite_t4096`` / ``v2_t8192`` - DeepSeek-V2-style softmax routers
    (greedy, and group-limited with a max group score).
  * ``v3_prefill_t16384`` / ``v3_decode_t{1,8,64,512}`` - the DeepSeek-V3
    MoE table of the "v3基本架构" page: hidden 7168, 256 routed experts of
    FFN width 2048, 8 per token, 1 shared expert; sigmoid affinities with a
    selection bias and node-limited (group-limited) routing.

Random recipe (one torch generator per tensor, seed = tensor id):
  x ~ N(0,1); W_g, W1, W3 ~ U(+-1/sqrt(d)); W2 ~ U(+-1/sqrt(I)); shared weights
  likewise with the shared hidden size; all drawn in float32 and rounded to the
  storage dtype.  Token inputs, the gate weight and the bias are drawn on the
  CPU generator (so they are the same bytes on every machine); the expert
  weights, which reach 22.6 GB in the V3 shapes, are drawn on the device the
  caller names, one expert at a time.
  V3 prefill bias: b ~ N(0, 0.1).  V3 decode bias: a Zipf(1.2) rank bias
  b_e = -1.2 * beta * ln(rank_e) over a seeded permutation of the experts, with
  beta stored below (calibrated by tests/golden/calibrate_decode_bias.py so the
  10% most-loaded experts take about half of the assignments).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Dict, Optional

import torch

SEED_X, SEED_WG, SEED_W1, SEED_W3, SEED_W2, SEED_WS1, SEED_WS3, SEED_WS2, SEED_BIAS, SEED_RANK = range(10)
SEED_DECODE_X = 10
SEED_CALIB_X = 11

# Zipf(1.2) decode-bias strength; written by tests/golden/calibrate_decode_bias.py
DECODE_ZIPF_S = 1.2
DECODE_ZIPF_BETA = 0.04655457510807537


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    E: int
    I: int
    k: int
    n_shared: int
    score_fn: str = "softmax"            # "softmax" | "sigmoid"
    topk_method: str = "greedy"          # "greedy" | "group_limited_greedy"
    n_group: int = 1
    topk_group: int = 1
    group_score: str = "max"             # "max" | "sum_top"
    group_top: int = 1
    norm_topk: bool = False
    routed_scaling_factor: float = 1.0
    act_dtype: str = "bf16"              # "f32" | "bf16"
    gate_w_dtype: str = "f32"            # "f32" | "bf16"
    bias: str = "none"                   # "none" | "normal0.1" | "zipf"
    out_dtype: str = "f32"               # layer output h' ("f32": the listing's fp32 weighted sum)
    expert_w_dtype: str = "act"          # packed expert weights: "act" (as activations) | "fp8" (e4m3 blocks)

    @property
    def I_s(self) -> int:
        return self.n_shared * self.I

    @property
    def R(self) -> int:
        return self.T * self.k

    def with_T(self, T: int) -> "Workload":
        return replace(self, T=T, name=f"{self.name.rsplit('_t', 1)[0]}_t{T}")

    def flops(self) -> float:
        """Algorithmic FLOPs of one forward: gate GEMM + routed + shared SwiGLU."""
        return (2.0 * self.T * self.d * self.E + 6.0 * self.d * self.I * self.R
                + 6.0 * self.d * self.I_s * self.T)


def _v3(T: int, bias: str) -> Workload:
    return Workload(name=f"v3_{'prefill' if bias == 'normal0.1' else 'decode'}_t{T}", T=T, d=7168,
                    E=256, I=2048, k=8, n_shared=1, score_fn="sigmoid",
                    topk_method="group_limited_greedy", n_group=8, topk_group=4,
                    group_score="sum_top", group_top=2, norm_topk=True,
                    routed_scaling_factor=2.5, act_dtype="bf16", gate_w_dtype="bf16", bias=bias)


WORKLOADS: Dict[str, Workload] = {}
for _w in [
    Workload(name="tiny_fp32_t128", T=128, d=64, E=12, I=32, k=4, n_shared=2,
             act_dtype="f32", gate_w_dtype="f32"),
    Workload(name="v2lite_t4096", T=4096, d=2048, E=64, I=1408, k=6, n_shared=2,
             act_dtype="bf16", gate_w_dtype="f32"),
    Workload(name="v2_t8192", T=8192, d=5120, E=160, I=1536, k=6, n_shared=2,
             topk_method="group_limited_greedy", n_group=8, topk_group=3, group_score="max",
             routed_scaling_factor=16.0, act_dtype="bf16", gate_w_dtype="f32"),
    _v3(16384, "normal0.1"),
    _v3(1, "zipf"), _v3(8, "zipf"), _v3(64, "zipf"), _v3(512, "zipf"),
]:
    WORKLOADS[_w.name] = _w

# FP8 expert weights (e4m3 blocks of 64 with power-of-two scales) of the
# decode and prefill layers.
for _T in (1, 8, 64, 512):
    _w = replace(WORKLOADS[f"v3_decode_t{_T}"], name=f"v3_decode_fp8_t{_T}", expert_w_dtype="fp8")
    WORKLOADS[_w.name] = _w
WORKLOADS["v3_prefill_fp8_t16384"] = replace(WORKLOADS["v3_prefill_t16384"], name="v3_prefill_fp8_t16384",
                                             expert_w_dtype="fp8")

# A V3-shaped layer cut to 8 experts and 1024 tokens (1.4 GB of weights):
# the case the kernel profiler captures, still larger than L2.
WORKLOADS["v3_profile_e8_t1024"] = Workload(
    name="v3_profile_e8_t1024", T=1024, d=7168, E=8, I=2048, k=4, n_shared=1, score_fn="sigmoid",
    topk_method="group_limited_greedy", n_group=4, topk_group=2, group_score="sum_top", group_top=2,
    norm_topk=True, routed_scaling_factor=2.5, act_dtype="bf16", gate_w_dtype="bf16", bias="normal0.1")

# A V3-shaped decode step (one token, top-8) over 16 experts with FP8 weights
# (0.7 GB of e4m3 weights): the profiler's case for the FP8 expert kernel.
WORKLOADS["v3_profile_fp8_e16_t1"] = Workload(
    name="v3_profile_fp8_e16_t1", T=1, d=7168, E=16, I=2048, k=8, n_shared=1, score_fn="sigmoid",
    topk_method="group_limited_greedy", n_group=1, topk_group=1, group_score="sum_top", group_top=2,
    norm_topk=True, routed_scaling_factor=2.5, act_dtype="bf16", gate_w_dtype="bf16", bias="zipf",
    expert_w_dtype="fp8")

# A V3-shaped decode step (one token, top-8) over 16 experts with bf16 weights
# (1.4 GB): the profiler's case for the decode-sized expert kernel.
WORKLOADS["v3_profile_e16_t1"] = replace(WORKLOADS["v3_profile_fp8_e16_t1"], name="v3_profile_e16_t1",
                                         expert_w_dtype="act")

# The V3 prefill layer's routing at full size (T=16384, d=7168, 256 experts,
# top-8, the same gate weights and bias) with the expert hidden size cut to 128:
# the router, dispatch, gather and combine kernels see exactly the prefill
# shapes in about 8 GB of device memory (the profiler's case for them).
WORKLOADS["v3_profile_route_t16384"] = replace(WORKLOADS["v3_prefill_t16384"], name="v3_profile_route_t16384",
                                               I=128)

CONFIG_ORDER = ["tiny_fp32_t128", "v2lite_t4096", "v2_t8192", "v3_prefill_t16384",
                "v3_decode_t1", "v3_decode_t8", "v3_decode_t64", "v3_decode_t512"]
DECODE_T = (1, 8, 64, 512)


def torch_dtype(name: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _uniform(shape, bound: float, seed: int, device, dtype: torch.dtype, per_leading: bool) -> torch.Tensor:
    g = _gen(seed, device)
    out = torch.empty(shape, dtype=dtype, device=device)
    if per_leading:
        for e in range(shape[0]):
            chunk = torch.rand(shape[1:], generator=g, device=device, dtype=torch.float32)
            out[e].copy_(chunk.mul_(2.0 * bound).sub_(bound))
    else:
        chunk = torch.rand(shape, generator=g, device=device, dtype=torch.float32)
        out.copy_(chunk.mul_(2.0 * bound).sub_(bound))
    return out


@dataclass
class LayerInputs:
    wl: Workload
    x: torch.Tensor                 # [T,d] act dtype
    wg: torch.Tensor                # [E,d] gate dtype
    bias: Optional[torch.Tensor]    # [E] float32 or None
    w1: torch.Tensor                # [E,I,d]
    w3: torch.Tensor                # [E,I,d]
    w2: torch.Tensor                # [E,d,I]
    ws1: torch.Tensor               # [I_s,d]
    ws3: torch.Tensor               # [I_s,d]
    ws2: torch.Tensor               # [d,I_s]
    extra: dict = field(default_factory=dict)


def decode_rank_bias(E: int, beta: float, s: float = DECODE_ZIPF_S) -> torch.Tensor:
    """b_e = -s * beta * ln(rank_e), rank from a seeded permutation (1 = hottest)."""
    perm = torch.randperm(E, generator=_gen(SEED_RANK))
    rank = torch.empty(E, dtype=torch.float64)
    rank[perm] = torch.arange(1, E + 1, dtype=torch.float64)
    return (-s * beta * torch.log(rank)).to(torch.float32)


def make_tokens(wl: Workload) -> torch.Tensor:
    """Token inputs x [T,d] on the CPU.  Decode batches are the first T rows of
    one seeded [512, d] draw, so the four decode sizes share their tokens."""
    act = torch_dtype(wl.act_dtype)
    if wl.bias == "zipf":
        full = torch.randn((512, wl.d), generator=_gen(SEED_DECODE_X), dtype=torch.float32)
        return full[: wl.T].to(act).contiguous()
    return torch.randn((wl.T, wl.d), generator=_gen(SEED_X), dtype=torch.float32).to(act)


def make_router(wl: Workload):
    """Gate weight [E,d] and selection bias [E] (or None) on the CPU."""
    wg = _uniform((wl.E, wl.d), 1.0 / math.sqrt(wl.d), SEED_WG, "cpu",
                  torch_dtype(wl.gate_w_dtype), per_leading=False)
    if wl.bias == "none":
        bias = None
    elif wl.bias == "normal0.1":
        bias = torch.randn((wl.E,), generator=_gen(SEED_BIAS), dtype=torch.float32) * 0.1
    elif wl.bias == "zipf":
        bias = decode_rank_bias(wl.E, DECODE_ZIPF_BETA)
    else:
        raise ValueError(wl.bias)
    return wg, bias


def make_experts(wl: Workload, device="cpu"):
    """Routed and shared expert weights in nn.Linear layout, drawn on ``device``
    (the shared ones None for a layer without a shared expert)."""
    act = torch_dtype(wl.act_dtype)
    bd, bi = 1.0 / math.sqrt(wl.d), 1.0 / math.sqrt(wl.I)
    w1 = _uniform((wl.E, wl.I, wl.d), bd, SEED_W1, device, act, per_leading=True)
    w3 = _uniform((wl.E, wl.I, wl.d), bd, SEED_W3, device, act, per_leading=True)
    w2 = _uniform((wl.E, wl.d, wl.I), bi, SEED_W2, device, act, per_leading=True)
    if wl.I_s == 0:
        return w1, w3, w2, None, None, None
    bs = 1.0 / math.sqrt(wl.I_s)
    ws1 = _uniform((wl.I_s, wl.d), bd, SEED_WS1, device, act, per_leading=False)
    ws3 = _uniform((wl.I_s, wl.d), bd, SEED_WS3, device, act, per_leading=False)
    ws2 = _uniform((wl.d, wl.I_s), bs, SEED_WS2, device, act, per_leading=False)
    return w1, w3, w2, ws1, ws3, ws2


def make_inputs(wl: Workload, device="cpu", expert_device=None) -> LayerInputs:
    """All inputs of one layer call.  Tokens, gate and bias come from the CPU
    generator and are moved to ``device``; expert weights are drawn on
    ``expert_device`` (default ``device``)."""
    expert_device = device if expert_device is None else expert_device
    x = make_tokens(wl).to(device)
    wg, bias = make_router(wl)
    wg = wg.to(device)
    bias = None if bias is None else bias.to(device)
    w1, w3, w2, ws1, ws3, ws2 = make_experts(wl, expert_device)
    return LayerInputs(wl=wl, x=x, wg=wg, bias=bias, w1=w1, w3=w3, w2=w2, ws1=ws1, ws3=ws3, ws2=ws2)


def small_workload(base: Workload, **kw) -> Workload:
    """A reduced copy of a workload for fast parity cases (same routing rules)."""
    name = kw.pop("name", base.name + "_small")
    return replace(base, name=name, **kw)


# ------------------------------------------------------- stage-level test data
SEED_STAGE = 1000


def random_idx(T: int, E: int, k: int, seed: int, one_hot_expert: Optional[int] = None) -> torch.Tensor:
    """[T,k] int32 expert choices, k distinct experts per token, seeded.  With
    ``one_hot_expert`` every token's first choice is that expert (a degenerate,
    maximally skewed load)."""
    g = _gen(SEED_STAGE + seed)
    keys = torch.rand((T, E), generator=g)
    if one_hot_expert is not None:
        keys[:, one_hot_expert] = -1.0
    return keys.argsort(dim=1)[:, :k].to(torch.int32).contiguous()


def random_rows(n: int, d: int, seed: int, dtype: torch.dtype = torch.bfloat16) -> torch.Tensor:
    g = _gen(SEED_STAGE + seed)
    return torch.randn((n, d), generator=g).to(dtype)


def random_gates(T: int, k: int, seed: int) -> torch.Tensor:
    g = _gen(SEED_STAGE + seed)
    return torch.rand((T, k), generator=g).contiguous()


def random_counts(E: int, R: int, seed: int) -> torch.Tensor:
    """[E] int32 row counts summing to R: some experts empty, one large."""
    g = _gen(SEED_STAGE + seed)
    w = torch.rand((E,), generator=g)
    w[torch.randperm(E, generator=g)[: max(1, E // 4)]] = 0.0
    w[int(torch.randint(E, (1,), generator=g))] += w.sum() + 1.0
    c = torch.floor(w / w.sum() * R).to(torch.int64)
    c[int(torch.argmax(w))] += R - int(c.sum())
    return c.to(torch.int32)
