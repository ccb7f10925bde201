#!/usr/bin/env python3
"""Benchmark of the DeepSeekMoE layer forward on B300.

One step = one whole layer forward (router, permutation, grouped SwiGLU
experts, shared expert, combine) over one batch of seeded synthetic tokens,
through the library's C ABI (moe_forward).  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the fp64 CPU oracle on host cores

Multi-GPU (torchrun, one process per GPU): every rank runs its own replica of
the layer on its own batch (tokens are independent, no collective on the
data path); the value is all ranks' tokens over the slowest rank's time.
"""
import argparse
import dataclasses
import datetime
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from mixture_experts_layer_85_b300 import inputs  # noqa: E402

METRIC = "routed tokens/s per MoE layer fwd"
UNIT = "tokens/s"
DEFAULT_WORKLOAD = "v3_prefill_t16384"


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(inputs.WORKLOADS))
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-per-config", dest="per_config", action="store_false",
                   help="skip the per_config lines (every other config, measured after the headline)")
    p.add_argument("--cpu-sample", type=int, default=0, help="tokens in the oracle's timed sample (0 = auto)")
    p.add_argument("--oracle-one-core", default=None, help=argparse.SUPPRESS)
    p.add_argument("--pass", dest="pass_", choices=["forward", "backward"], default="forward",
                   help="backward: time moe_backward (gradients of the layer) instead of the forward")
    return p.parse_args(argv)


# ------------------------------------------------------------------ ranks

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int) -> float:
    """The slowest rank's time (every rank gets the same answer)."""
    if world <= 1:
        return value
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, seconds_max: float) -> float:
    return units_per_rank * world / seconds_max


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 50 ms in the background;
    stop(t0, t1) keeps the samples whose timestamps fall in the host-time window
    [t0, t1] of the timed region (padded by one sampling interval)."""

    FIELDS = ("timestamp,index,uuid,clocks.sm,clocks.max.sm,power.draw.instant,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,power.limit")
    INTERVAL_MS = 50

    def __init__(self):
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", str(self.INTERVAL_MS), "-f", self.path], stdout=subprocess.DEVNULL,
                                         stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        # the timed region starts once the sampler is producing rows
        t0 = time.time()
        while time.time() - t0 < 5.0 and os.path.getsize(self.path) == 0:
            time.sleep(0.02)

    @staticmethod
    def _num(s):
        try:
            return float(s)
        except ValueError:
            return None

    def stop(self, t0: float, t1: float):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(2 * self.INTERVAL_MS / 1e3)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        uuid = None
        try:
            uuid = str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
        except Exception:
            pass
        pad = self.INTERVAL_MS / 1e3
        rows = []
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 12:
                continue
            if uuid and uuid not in f[2] and f[2].replace("GPU-", "") not in uuid:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                continue
            if t0 - pad <= ts <= t1 + pad:
                rows.append(f[1:])
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples inside the timed region"]}
        sm = [v for v in (self._num(r[2]) for r in rows) if v is not None]
        mx = [v for v in (self._num(r[3]) for r in rows) if v is not None]
        pw = [v for v in (self._num(r[4]) for r in rows) if v is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i].lower().startswith("active")})
        lim = [v for v in (self._num(r[10]) for r in rows) if v is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "power_w_instant_max": max(pw) if pw else None,
                "power_w_instant_median": statistics.median(pw) if pw else None,
                "power_limit_w": max(lim) if lim else None}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        p = json.load(open(path))
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


# --------------------------------------------------------- algorithmic work

def layer_bytes(wl, counts: np.ndarray) -> float:
    """Bytes the method must move: x in, out, W_g, idx/w, the weights of the
    experts that received tokens, the shared weights."""
    eb = 2 if wl.act_dtype == "bf16" else 4
    ob = 2 if wl.out_dtype == "bf16" else 4
    gb = 2 if wl.gate_w_dtype == "bf16" else 4
    wb = expert_weight_bytes(wl)
    touched = int((counts > 0).sum())
    return (wl.T * wl.d * (eb + ob) + wl.E * wl.d * gb + wl.T * wl.k * 8
            + touched * 3 * wl.d * wl.I * wb + 3 * wl.d * wl.I_s * wb)


def expert_weight_bytes(wl) -> float:
    """Bytes per stored expert weight: the activation dtype, or one e4m3 byte
    plus a 4-byte scale per 64 weights."""
    if wl.expert_w_dtype == "fp8":
        return 1.0 + 4.0 / 64.0
    return 2 if wl.act_dtype == "bf16" else 4


def experts_work(wl, counts: np.ndarray):
    """(FLOPs, algorithmic bytes) of the expert kernel (GEMM1 + SwiGLU and
    GEMM2 of every routed assignment and of the shared expert): x rows of every
    assignment and every token, the weights of the touched experts and of the
    shared expert, the hidden rows written and read back, the fp32 expert
    outputs written."""
    eb = 2 if wl.act_dtype == "bf16" else 4
    wb = expert_weight_bytes(wl)
    flops = 6.0 * wl.R * wl.d * wl.I + 6.0 * wl.T * wl.d * wl.I_s
    touched = int((counts > 0).sum())
    byts = ((wl.R + wl.T) * wl.d * eb + touched * 3 * wl.I * wl.d * wb + 3 * wl.I_s * wl.d * wb
            + 2 * (wl.R * wl.I + wl.T * wl.I_s) * eb + (wl.R + wl.T) * wl.d * 4)
    return flops, byts


# ----------------------------------------------------------- oracle timing

def oracle_sample_size(wl, requested: int) -> int:
    if requested > 0:
        return min(requested, wl.T)
    if wl.d >= 7168:
        return min(wl.T, 8)
    if wl.d >= 2048:
        return min(wl.T, 16)
    return wl.T


def oracle_cfg(wl):
    from oracle import moe_oracle as orc
    return orc.OracleConfig(T=wl.T, d=wl.d, E=wl.E, I=wl.I, k=wl.k, n_shared=wl.n_shared, score_fn=wl.score_fn,
                            topk_method=wl.topk_method, n_group=wl.n_group, topk_group=wl.topk_group,
                            group_score=wl.group_score, group_top=wl.group_top, norm_topk=wl.norm_topk,
                            routed_scaling_factor=wl.routed_scaling_factor)


def time_oracle(wl, li, tokens: np.ndarray):
    """Seconds the fp64 oracle takes for the layer on `tokens` (weights are read
    per expert from wherever they live and widened to float64)."""
    from oracle import moe_oracle as orc

    def f64(t):
        return t.detach().to("cpu").to(torch.float64).numpy()

    cfg = oracle_cfg(wl)
    cfg.T = int(tokens.size)
    x = f64(li.x)[tokens]
    wg = f64(li.wg)
    bias = None if li.bias is None else li.bias.detach().cpu().float().numpy()

    def expert(e):
        return f64(li.w1[e]), f64(li.w3[e]), f64(li.w2[e])

    shared = None if wl.n_shared == 0 else (f64(li.ws1), f64(li.ws3), f64(li.ws2))
    t0 = time.perf_counter()
    orc.moe_forward(x, wg, bias, expert, shared, cfg)
    return time.perf_counter() - t0


def host_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def time_end_to_end_serial(layer, x, out_dtype, K, stream, world) -> float:
    """Seconds for K steps of host tokens -> layer -> host output on one stream."""
    T, d = x.shape
    x_h = x.cpu().pin_memory()
    out_h = torch.empty((T, d), dtype=out_dtype).pin_memory()
    x_d = torch.empty_like(x)
    out_d = torch.empty((T, d), dtype=out_dtype, device=x.device)

    def run(n):
        for _ in range(n):
            x_d.copy_(x_h, non_blocking=True)
            layer.forward(x_d, out_d, stream=stream)
            out_h.copy_(out_d, non_blocking=True)

    run(2)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier(world)
    e0.record(stream)
    run(K)
    e1.record(stream)
    torch.cuda.synchronize()
    return max_over_ranks(e0.elapsed_time(e1) / 1e3, world)


def time_end_to_end(layer, x, out_dtype, K, stream, world) -> float:
    """Seconds for K pipelined steps of host tokens -> layer -> host output."""
    T, d = x.shape
    x_h = x.cpu().pin_memory()
    out_h = [torch.empty((T, d), dtype=out_dtype).pin_memory() for _ in range(2)]
    x_d = [torch.empty_like(x) for _ in range(2)]
    out_d = [torch.empty((T, d), dtype=out_dtype, device=x.device) for _ in range(2)]
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()

    def run(n, e0=None):
        fwd_done = [torch.cuda.Event() for _ in range(2)]
        h2d_done = [torch.cuda.Event() for _ in range(2)]
        d2h_done = [torch.cuda.Event() for _ in range(2)]
        used = [False, False]
        if e0 is not None:
            h2d.wait_event(e0)
        for i in range(n):
            s = i % 2
            if used[s]:
                h2d.wait_event(fwd_done[s])
            with torch.cuda.stream(h2d):
                x_d[s].copy_(x_h, non_blocking=True)
            h2d_done[s].record(h2d)
            stream.wait_event(h2d_done[s])
            if used[s]:
                stream.wait_event(d2h_done[s])
            layer.forward(x_d[s], out_d[s], stream=stream)
            fwd_done[s].record(stream)
            d2h.wait_event(fwd_done[s])
            with torch.cuda.stream(d2h):
                out_h[s].copy_(out_d[s], non_blocking=True)
            d2h_done[s].record(d2h)
            used[s] = True
        for s in range(2):
            if used[s]:
                stream.wait_event(d2h_done[s])

    run(2)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier(world)
    e0.record(stream)
    run(K, e0)
    e1.record(stream)
    torch.cuda.synchronize()
    return max_over_ranks(e0.elapsed_time(e1) / 1e3, world)


# ------------------------------------------------------------- measurement

# Every config of the layer, beside the headline line: the fp32 reference
# layer, the V2-shaped layers and the V3 decode batches (the V3 prefill layer
# is the headline itself).
PER_CONFIG = ["tiny_fp32_t128", "v2lite_t4096", "v2_t8192", "v3_decode_t1", "v3_decode_t8", "v3_decode_t64",
              "v3_decode_t512"]
NOMINAL_HBM_GBS = 8000.0


class L2Flush:
    """Before a timed decode step: writes a buffer of twice the device's L2
    size, so nothing the previous step read is left in L2, then reads another
    buffer as large, so the lines that write left dirty go back to HBM now and
    not inside the timed step."""

    def __init__(self, dev):
        l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 126 << 20)) or (126 << 20)
        n = 2 * l2 // 4 + 256
        self.buf = torch.empty(n, dtype=torch.int32, device=dev)
        self.rd = torch.zeros(n, dtype=torch.int32, device=dev)
        self.sink = torch.zeros((), dtype=torch.int64, device=dev)
        self.n = 0

    def __call__(self):
        self.n += 1
        self.buf.fill_(self.n)
        torch.sum(self.rd, dim=0, dtype=torch.int64, out=self.sink)


def needs_flush(wl) -> bool:
    """Decode batches: the token batch fits in L2, and so might the weights
    touched by the previous step."""
    return wl.T <= 512


def time_steps(layer, x, out, counts, K, flush=None, stream=None, per_step=None):
    """Average ms of one layer step over K timed steps (CUDA events on the
    stream).  With `flush`, L2 is flushed before every step and each step is
    timed on its own, the flush outside the events (their times are appended
    to `per_step` when given)."""
    stream = stream or torch.cuda.current_stream()
    if flush is None:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(K):
            layer.forward(x, out, counts=counts)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / K
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for a, b in evs:
        flush()
        a.record(stream)
        layer.forward(x, out, counts=counts)
        b.record(stream)
    torch.cuda.synchronize()
    times = [a.elapsed_time(b) for a, b in evs]
    if per_step is not None:
        per_step.extend(times)
    return sum(times) / K


def stage_times(layer, x, out, counts, n, flush=None):
    """Average ms of each stage of moe_forward over n steps (events between the
    stages split the kernels' launch overlap, so this runs outside the timed
    steps)."""
    from mixture_experts_layer_85_b300 import _lib
    S = _lib.MOE_FORWARD_STAGES
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(n * (S + 1))]
    _lib.moe_profile_arm(ev)
    for _ in range(n):
        if flush is not None:
            flush()
        layer.forward(x, out, counts=counts)
    torch.cuda.synchronize()
    _lib.moe_profile_arm(None)
    res = {}
    for s_ in range(S):
        v = [ev[i * (S + 1) + s_].elapsed_time(ev[i * (S + 1) + s_ + 1]) for i in range(n)]
        res[_lib.moe_forward_stage_name(s_)] = sum(v) / len(v)
    return res


# DRAM traffic of the expert kernel per forward (dram__bytes_read.sum + dram__bytes_write.sum over the
# launches of one forward, one ncu pass on the full-size workload) for the workloads captured with the
# current kernel source; the summary and the command that made it are in the named profiles/ file.
EXPERT_TRAFFIC = {
    "v3_prefill_t16384": (32.03e9, "profiles/launches_v3_prefill_t16384.md"),
    # the same 9 experts' weights (8 routed + shared) as the 16-expert capture
    "v3_decode_fp8_t1": (424.9e6, "profiles/gemv_fp8_decode_v3shape_e16_t1.md"),
}
GEMV_MAX_T = 64   # FP8 layers of at most this many tokens run the expert GEMV


def expert_kernel(wl):
    """The expert stage's kernel and its launches per forward."""
    if wl.act_dtype != "bf16":
        return "swiglu_simt_h_kernel, swiglu_simt_y_kernel (fp32 SIMT)", 2
    if wl.expert_w_dtype == "fp8" and wl.T <= GEMV_MAX_T:
        return "gemv_fp8_kernel (GEMM1 + SwiGLU, then GEMM2)", 2
    name = "pair_gemm_kernel<true> (FP8 weights; " if wl.expert_w_dtype == "fp8" else "pair_gemm_kernel ("
    if wl.T * wl.k <= 8192:
        return name + "GEMM1 + SwiGLU and GEMM2 in one launch)", 1
    return name + "GEMM1 + SwiGLU, then GEMM2)", 2


def expert_roofline(wl, cnt, expert_ms, peaks):
    """The expert kernel (the dominant one) against its roof: tensor when its
    FLOP per algorithmic byte reaches the ridge of the measured peaks, else HBM."""
    flops, byts = experts_work(wl, cnt)
    secs = expert_ms / 1e3
    ridge = peaks["bf16_tflops_sustained"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    if flops / byts >= ridge:
        achieved = flops / secs / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 2), "peak": peaks["bf16_tflops_sustained"],
                "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops_sustained"], 4),
                "frac_of_burst_peak": round(achieved / peaks["bf16_tflops"], 4),
                "peak_source": peaks["source"] + " sustained bf16"}
    else:
        achieved = byts / secs / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4), "peak_source": peaks["source"] + " HBM copy"}
    traffic, source = EXPERT_TRAFFIC.get(wl.name, (None, None))
    if traffic is not None:
        roof["traffic_source"] = source
        roof["traffic_over_algorithmic"] = round(traffic / byts, 3)
    kernel, launches = expert_kernel(wl)
    roof.update({"kernel": kernel, "launches_per_forward": launches, "traffic": traffic,
                 "per_launch_flops": flops, "per_launch_algorithmic_bytes": byts,
                 "avg_launch_ms": round(expert_ms, 4)})
    return roof


def layer_summary(wl, ms_step, cnt, peaks):
    flops = wl.flops()
    byts = layer_bytes(wl, cnt)
    sec = ms_step / 1e3
    tf = flops / sec / 1e12
    gbs = byts / sec / 1e9
    return {"ms_per_step": round(ms_step, 4), "tokens_per_s": round(wl.T / sec, 1),
            "assignments_per_s": round(wl.T * wl.k / sec, 1), "tflops": round(tf, 2),
            "tflops_frac_of_peak": {"burst": round(tf / peaks["bf16_tflops"], 4),
                                    "sustained": round(tf / peaks["bf16_tflops_sustained"], 4)},
            "gbs_algorithmic": round(gbs, 1),
            "gbs_frac_of_hbm": {"measured": round(gbs / peaks["hbm_gbs"], 4),
                                "nominal_8tbs": round(gbs / NOMINAL_HBM_GBS, 4)},
            "experts_touched": int((cnt > 0).sum())}


def blas_threads() -> int:
    """Threads numpy's BLAS (OpenBLAS) uses: OPENBLAS_NUM_THREADS / OMP_NUM_THREADS
    when set, else one per usable core (at most 64, the library's build limit)."""
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        v = os.environ.get(var)
        if v and v.isdigit() and int(v) > 0:
            return int(v)
    return min(64, host_threads())


def oracle_rate(wl, li, n_tok, seed=0):
    """Oracle tokens/s on a seeded sample of n_tok tokens, on this process's cores."""
    toks = np.sort(np.random.default_rng(seed).choice(wl.T, min(n_tok, wl.T), replace=False))
    secs = time_oracle(wl, li, toks)
    return {"value": round(toks.size / secs, 3), "unit": UNIT, "cores": blas_threads(), "host_cpus": host_threads(),
            "kind": "oracle", "sample": f"{toks.size} seeded tokens of {wl.name} through the fp64 oracle "
                                        f"(routing + experts + shared), {secs:.1f} s"}


def oracle_rate_one_core(name: str, n_tok: int):
    """The oracle on a single host core: a child process whose BLAS is held to
    one thread (the thread count is fixed when numpy loads)."""
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-one-core", name, "--cpu-sample",
                        str(n_tok)], env=env, capture_output=True, text=True, timeout=600)
    if r.returncode != 0:
        return {"unavailable": r.stderr.strip().splitlines()[-1] if r.stderr.strip() else f"rc {r.returncode}"}
    return json.loads(r.stdout.strip().splitlines()[-1])


def per_config_lines(base_layer, base_li, dev, K, W, peaks, with_oracle):
    """One summary per config of PER_CONFIG: the V3 decode batches reuse the
    headline layer's packed experts (same layer, another batch and bias)."""
    from mixture_experts_layer_85_b300.layer import MoELayer
    flush = L2Flush(dev)
    res = {}
    for name in PER_CONFIG:
        wl = inputs.WORKLOADS[name]
        if name.startswith("v3_decode") and base_layer is not None:
            x = inputs.make_tokens(wl).to(dev)
            _, bias = inputs.make_router(wl)
            layer = base_layer.variant(wl, bias)
            li = dataclasses.replace(base_li, wl=wl, x=x, bias=bias)
        else:
            li = inputs.make_inputs(wl, dev)
            layer = MoELayer(wl, li, dev)
            x = li.x
        out = torch.empty((wl.T, wl.d), dtype=inputs.torch_dtype(wl.out_dtype), device=dev)
        counts = torch.empty((wl.E,), dtype=torch.int32, device=dev)
        fl = flush if needs_flush(wl) else None
        for _ in range(max(W, 0)):
            layer.forward(x, out, counts=counts)
        code, word = layer.device_status()
        if code != 0:
            raise RuntimeError(f"{name}: device status after warm-up {code} ({word})")
        clocks = ClockSampler()
        clocks.start()
        t0 = time.time()
        steps_ms = []
        ms = time_steps(layer, x, out, counts, K, fl, per_step=steps_ms)
        clk = clocks.stop(t0, time.time())
        st = stage_times(layer, x, out, counts, max(3, min(K, 10)), fl)
        code, word = layer.device_status()
        if code != 0:
            raise RuntimeError(f"{name}: device status after timed steps {code} ({word})")
        cnt = counts.cpu().numpy()
        line = {"workload": name, "T": wl.T, "d": wl.d, "E": wl.E, "I": wl.I, "k": wl.k,
                "dtype": "bf16" if wl.act_dtype == "bf16" else "f32",
                "l2": "flushed before every timed step (2x L2 written, then 2x L2 read, outside the timed step)"
                      if fl else "no flush: weights larger than L2",
                **layer_summary(wl, ms, cnt, peaks), "stage_ms": {k: round(v, 4) for k, v in st.items()},
                "roofline": expert_roofline(wl, cnt, st["experts"], peaks), "clocks": clk}
        if steps_ms:
            line["ms_per_step_median"] = round(statistics.median(steps_ms), 4)
        if with_oracle:
            line["oracle"] = oracle_rate(wl, li, oracle_sample_size(wl, 0))
        res[name] = line
        del layer, li, out, counts
        torch.cuda.empty_cache()
    return res


# ---------------------------------------------------------------- our arm

def run_ours(args, world, rank):
    from mixture_experts_layer_85_b300 import _lib
    from mixture_experts_layer_85_b300.layer import MoELayer

    wl = inputs.WORKLOADS[args.workload]
    dev = torch.device("cuda", torch.cuda.current_device())
    li = inputs.make_inputs(wl, dev)
    layer = MoELayer(wl, li, dev)
    x = li.x
    out = torch.empty((wl.T, wl.d), dtype=inputs.torch_dtype(wl.out_dtype), device=dev)
    counts = torch.empty((wl.E,), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()

    for _ in range(max(args.warmup, 0)):
        layer.forward(x, out, counts=counts)
    code, word = layer.device_status()
    if code != 0:
        raise RuntimeError(f"device status after warm-up: {_lib.moe_status_string(code)} ({word})")
    torch.cuda.synchronize()

    K = args.steps
    # decode batches: L2 flushed before every step, each step timed on its own
    # (the flush outside its events), as in the per-config lines
    fl = L2Flush(dev) if needs_flush(wl) else None
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler()
    clocks.start()
    # the GPU idled while the sampler started: a few untimed steps first
    for _ in range(3):
        layer.forward(x, out, counts=counts)
    barrier(world)
    torch.cuda.synchronize()
    launches0 = _lib.moe_launch_count()
    host_t0 = time.time()
    if fl is None:
        t_start.record(stream)
        for _ in range(K):
            layer.forward(x, out, counts=counts)
        t_end.record(stream)
        torch.cuda.synchronize()
        step_ms = None
    else:
        per_step = []
        step_ms = time_steps(layer, x, out, counts, K, fl, stream, per_step=per_step)
    host_t1 = time.time()
    launches = _lib.moe_launch_count() - launches0
    barrier(world)
    clk = clocks.stop(host_t0, host_t1)
    code, word = layer.device_status()
    if code != 0:
        raise RuntimeError(f"device status after timed steps: {_lib.moe_status_string(code)} ({word})")

    elapsed_s = (t_start.elapsed_time(t_end) if step_ms is None else step_ms * K) / 1e3
    elapsed_max = max_over_ranks(elapsed_s, world)
    value = whole_job_rate(wl.T * K, world, elapsed_max)

    # Stage breakdown in a separate pass: events recorded between the stages
    # split the kernels' launch overlap, so they stay out of the timed steps.
    stage_ms = stage_times(layer, x, out, counts, max(3, min(K, 10)), fl)

    cnt = counts.cpu().numpy()
    peaks = measured_peaks()
    ms_step = elapsed_s * 1e3 / K
    flops = wl.flops()
    byts = layer_bytes(wl, cnt)
    roof = expert_roofline(wl, cnt, stage_ms["experts"], peaks)

    # end to end through the C ABI with host buffers: every step copies its
    # tokens host -> device, runs the layer and copies h' device -> host.  Two
    # buffer slots and two copy streams let step i's copies overlap the
    # neighbouring steps' forwards, as a serving loop would run them.
    # Small batches move few bytes and the cross-stream hand-offs cost more
    # than they hide, so both loops are timed and the faster one is reported
    # under its name.
    e2e_pipe = time_end_to_end(layer, x, out.dtype, K, stream, world)
    e2e_serial = time_end_to_end_serial(layer, x, out.dtype, K, stream, world)
    e2e_s = min(e2e_pipe, e2e_serial)
    eb = x.element_size()
    e2e = {"value": round(whole_job_rate(wl.T * K, world, e2e_s), 1), "unit": UNIT,
           "h2d_bytes_per_step": wl.T * wl.d * eb, "d2h_bytes_per_step": wl.T * wl.d * out.element_size(),
           "loop": ("pipelined: H2D of step i+1 and D2H of step i-1 overlap the forward of step i (2 slots)"
                    if e2e_pipe <= e2e_serial else "serial: H2D, forward, D2H in order on one stream"),
           "pipelined_value": round(whole_job_rate(wl.T * K, world, e2e_pipe), 1),
           "serial_value": round(whole_job_rate(wl.T * K, world, e2e_serial), 1)}

    # host-side cost of one moe_forward call (argument checks, tensor maps, launches)
    torch.cuda.synchronize()
    h0 = time.perf_counter()
    for _ in range(10):
        layer.forward(x, out, counts=counts)
    host_us = (time.perf_counter() - h0) / 10 * 1e6
    torch.cuda.synchronize()

    cpu = None
    with_oracle = rank == 0 and world == 1 and not args.no_cpu_baseline
    if with_oracle:
        cpu = oracle_rate(wl, li, oracle_sample_size(wl, args.cpu_sample))
        # the same oracle on one host core, on a 64-token sample of a smaller layer
        cpu["one_core"] = oracle_rate_one_core("v2lite_t4096", 64)

    per_config = None
    if args.per_config and args.workload == DEFAULT_WORKLOAD:
        per_config = per_config_lines(layer, li, dev, max(3, min(K, 20)), args.warmup, peaks, with_oracle)

    res = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if wl.act_dtype == "bf16" else "f32", "data": "synthetic",
        "config": {"workload": wl.name, "T": wl.T, "d": wl.d, "E": wl.E, "I": wl.I, "k": wl.k,
                   "n_shared": wl.n_shared, "router": f"{wl.score_fn}/{wl.topk_method}",
                   "expert_weights": "fp8 e4m3, 64-wide blocks" if wl.expert_w_dtype == "fp8" else wl.act_dtype,
                   "parallelism": f"replicas x{world}",
                   "l2": "flushed before every timed step (2x L2 written, then 2x L2 read, outside the timed step)"
                   if fl is not None else "inputs larger than L2 (expert weights and token batch exceed 126 MB)"},
        "tflops": round(flops / (elapsed_s / K) / 1e12, 2),
        "tflops_frac_of_peak": {"burst": round(flops / (elapsed_s / K) / 1e12 / peaks["bf16_tflops"], 4),
                                "sustained": round(flops / (elapsed_s / K) / 1e12 / peaks["bf16_tflops_sustained"], 4)},
        "gbs_algorithmic": round(byts / (elapsed_s / K) / 1e9, 1),
        "gbs_frac_of_hbm": round(byts / (elapsed_s / K) / 1e9 / peaks["hbm_gbs"], 4),
        "gbs_frac_of_nominal_8tbs": round(byts / (elapsed_s / K) / 1e9 / NOMINAL_HBM_GBS, 4),
        "stage_ms": {k: round(v, 4) for k, v in stage_ms.items()},
        "experts_touched": int((cnt > 0).sum()),
        "roofline": roof,
        "cpu_baseline": cpu,
        "per_config": per_config,
        "e2e": e2e,
        "gpu_launches": int(launches),
        "host_us_per_forward_call": round(host_us, 1),
        "clocks": clk,
    }
    if step_ms is not None:
        res["ms_per_step_median"] = round(statistics.median(per_step), 4)
    return res


# ----------------------------------------------------------- reference arm

def run_backward(args, world, rank):
    """Layer backward (moe_backward) on the workload: W warm-ups, then K timed
    calls bracketed by CUDA events on the stream."""
    from mixture_experts_layer_85_b300 import _lib

    wl = inputs.WORKLOADS[args.workload]
    dev = torch.device("cuda", torch.cuda.current_device())
    li = inputs.make_inputs(wl, dev)
    cfg = _lib.make_config(wl)
    g = torch.Generator().manual_seed(4242)
    dout = torch.randn((wl.T, wl.d), generator=g).to(inputs.torch_dtype(wl.out_dtype)).to(dev)
    E, I, d, Is = wl.E, wl.I, wl.d, wl.I_s
    f32 = dict(dtype=torch.float32, device=dev)
    grads = [torch.empty((wl.T, d), **f32), torch.empty((E, d), **f32), torch.empty((E, I, d), **f32),
             torch.empty((E, I, d), **f32), torch.empty((E, d, I), **f32), torch.empty((Is, d), **f32),
             torch.empty((Is, d), **f32), torch.empty((d, Is), **f32)]
    ws = torch.empty(_lib.moe_backward_workspace_size(cfg), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        _lib.moe_backward(cfg, li.x, li.wg, li.bias, li.w1, li.w3, li.w2, li.ws1, li.ws3, li.ws2, dout, *grads, ws)

    for _ in range(max(args.warmup, 0)):
        step()
    torch.cuda.synchronize()
    K = args.steps
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler()
    barrier(world)
    clocks.start()
    host_t0 = time.time()
    t0.record(stream)
    for _ in range(K):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    host_t1 = time.time()
    barrier(world)
    clk = clocks.stop(host_t0, host_t1)
    code, word = _lib.moe_get_device_status(ws)
    if code != 0:
        raise RuntimeError(f"device status after timed steps: {_lib.moe_status_string(code)} ({word})")
    elapsed = max_over_ranks(t0.elapsed_time(t1) / 1e3, world)
    # algorithmic FLOPs: the expert GEMMs of the forward recomputation (6 d I
    # per routed row and per token for the shared expert) and of the backward
    # proper (twice that: data and weight gradients), plus the router's
    # logits, d logits -> dW_g and dx (2 d E per token each)
    fwd = 6.0 * d * I * wl.T * wl.k + 6.0 * d * Is * wl.T
    flops = 3.0 * fwd + 6.0 * d * E * wl.T
    peaks = measured_peaks()
    tflops = flops / (elapsed / K) / 1e12
    return {"metric": "tokens/s per MoE layer bwd", "value": round(whole_job_rate(wl.T * K, world, elapsed), 1),
            "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": round(elapsed / K * 1e3, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": wl.name, "T": wl.T, "d": d, "E": E, "I": I, "k": wl.k, "n_shared": wl.n_shared,
                       "pass": "backward", "parallelism": f"replicas x{world}"},
            "tflops": round(tflops, 2),
            "roofline": {"bound": "tensor", "achieved": round(tflops, 2), "peak": peaks["bf16_tflops_sustained"],
                         "unit": "TFLOP/s", "frac": round(tflops / peaks["bf16_tflops_sustained"], 4),
                         "kernel": "whole backward (expert-kernel products + elementwise kernels)", "traffic": None,
                         "peak_source": peaks["source"] + " sustained bf16"},
            "clocks": clk}


def run_reference(args, world, rank):
    if rank != 0:
        return None
    wl = inputs.WORKLOADS[args.workload]
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    li = inputs.make_inputs(wl, "cpu", expert_device=dev)
    S_tok = oracle_sample_size(wl, args.cpu_sample if args.cpu_sample else (4 if wl.d >= 7168 else 0))
    rng = np.random.default_rng(1)
    for _ in range(max(args.warmup, 0)):
        time_oracle(wl, li, np.sort(rng.choice(wl.T, S_tok, replace=False)))
    total = 0.0
    for _ in range(args.steps):
        total += time_oracle(wl, li, np.sort(rng.choice(wl.T, S_tok, replace=False)))
    value = S_tok * args.steps / total
    cpu = {"value": round(value, 3), "unit": UNIT, "cores": torch.get_num_threads(), "host_cpus": host_threads(),
           "kind": "oracle", "sample": f"{S_tok} seeded tokens of {wl.name} per step through the fp64 oracle"}
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total / args.steps * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "T": wl.T, "d": wl.d, "E": wl.E, "I": wl.I, "k": wl.k,
                   "n_shared": wl.n_shared, "router": f"{wl.score_fn}/{wl.topk_method}",
                   "parallelism": "host cores"},
        "cpu_baseline": cpu,
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    args = parse_args(argv)
    if args.oracle_one_core:
        # child of oracle_rate_one_core: BLAS already held to one thread by the environment
        wl = inputs.WORKLOADS[args.oracle_one_core]
        print(json.dumps(oracle_rate(wl, inputs.make_inputs(wl, "cpu"), args.cpu_sample or 64)))
        return
    world, rank, _ = dist_setup()
    if args.impl == "reference":
        res = run_reference(args, world, rank)
    else:
        if not torch.cuda.is_available():
            raise SystemExit("bench.py needs a CUDA GPU for --impl ours")
        res = run_backward(args, world, rank) if args.pass_ == "backward" else run_ours(args, world, rank)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
