"""The expert kernel needs no co-residency of its clusters.

Its tiles are handed out at run time from a ticket counter, so a cluster only
ever waits on tiles that running clusters hold.  Here another kernel holds
most of the GPU's SMs (on another stream, for a bounded 200 ms) while a
one-launch (decode-sized) layer runs with its wait limit cut to 20 ms: the
layer must finish with MOE_OK and match the oracle.  Had tiles been dealt to
clusters that cannot start, a resident cluster's GEMM2 tile would wait for
them past the limit.

The SM-holding kernel is test scaffolding compiled here with NVRTC: each of
its CTAs takes most of an SM's shared memory and sleeps on %globaltimer until
its time is up (no kernel waits on another).  It runs in clusters of two, as
the expert kernel does, so the SMs it leaves free come in pairs that can hold
the expert kernel's clusters."""
import ctypes

import pytest
import torch

from mixture_experts_layer_85_b300 import _lib, inputs
from mixture_experts_layer_85_b300.layer import MoELayer
from tests.test_gpu_parity import check_layer

pytestmark = pytest.mark.gpu

HOLD_SRC = rb"""
extern "C" __global__ void __cluster_dims__(2, 1, 1) hold_sm(unsigned long long ns, int* out) {
  extern __shared__ int smem[];
  unsigned long long t0, t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  do {
    __nanosleep(2000);
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  } while (t - t0 < ns);
  smem[threadIdx.x] = (int)(t - t0);
  __syncthreads();
  if (threadIdx.x == 0) out[blockIdx.x] = smem[0];
}
"""
HOLD_SMEM = 200 * 1024
HOLD_NS = 200_000_000


def _check(res):
    err = res[0]
    assert int(err) == 0, err
    return res[1:] if len(res) > 2 else (res[1] if len(res) == 2 else None)


def _hold_kernel():
    from cuda.bindings import driver, nvrtc
    major, minor = torch.cuda.get_device_capability()
    prog = _check(nvrtc.nvrtcCreateProgram(HOLD_SRC, b"hold.cu", 0, [], []))
    opts = [f"--gpu-architecture=sm_{major}{minor}a".encode()]
    _check(nvrtc.nvrtcCompileProgram(prog, len(opts), opts))
    n = _check(nvrtc.nvrtcGetCUBINSize(prog))
    cubin = b" " * n
    _check(nvrtc.nvrtcGetCUBIN(prog, cubin))
    mod = _check(driver.cuModuleLoadData(cubin))
    fn = _check(driver.cuModuleGetFunction(mod, b"hold_sm"))
    _check(driver.cuFuncSetAttribute(fn, driver.CUfunction_attribute.CU_FUNC_ATTRIBUTE_MAX_DYNAMIC_SHARED_SIZE_BYTES,
                                     HOLD_SMEM))
    return driver, mod, fn


def _nonblocking_stream(driver):
    st = _check(driver.cuStreamCreate(driver.CUstream_flags.CU_STREAM_NON_BLOCKING.value))
    return st, torch.cuda.ExternalStream(int(st))


def test_expert_kernel_finishes_while_other_work_holds_most_sms():
    T = 64
    wl = inputs.small_workload(inputs.WORKLOADS["v3_prefill_t16384"], name="v3_sched_t64", T=T, d=1024, E=64,
                               I=512, n_group=8, topk_group=4)
    li = inputs.make_inputs(wl, "cuda")
    layer = MoELayer(wl, li, "cuda")
    layer.forward(li.x)
    assert layer.device_status()[0] == _lib.MOE_OK
    torch.cuda.synchronize()

    driver, mod, fn = _hold_kernel()
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    n_hold = 2 * (n_sm // 4)                               # half the SMs, in pairs
    hold_raw, hold_s = _nonblocking_stream(driver)
    run_raw, run_s = _nonblocking_stream(driver)
    out = torch.zeros(n_hold, dtype=torch.int32, device="cuda")
    args = ((HOLD_NS, out.data_ptr()), (ctypes.c_ulonglong, ctypes.c_void_p))
    idx = torch.empty((T, wl.k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, wl.k), dtype=torch.float32, device="cuda")
    counts = torch.empty((wl.E,), dtype=torch.int32, device="cuda")
    y = torch.empty((T, wl.d), dtype=torch.float32, device="cuda")
    ev = {n: torch.cuda.Event(enable_timing=True) for n in ("start", "held", "layer0", "layer1")}
    # load every kernel used below before the SMs are held (a first launch may
    # load its module, which waits for the device)
    with torch.cuda.stream(run_s):
        torch.cuda._sleep(1000)
        layer.forward(li.x, y, idx=idx, w=w, counts=counts, stream=run_s)
    torch.cuda.synchronize()
    _lib.moe_debug_inject(_lib.MOE_DEBUG_WAIT_LIMIT_NS, 20_000_000)
    try:
        ev["start"].record(hold_s)
        _check(driver.cuLaunchKernel(fn, n_hold, 1, 1, 32, 1, 1, HOLD_SMEM, hold_raw, args, 0))
        ev["held"].record(hold_s)
        with torch.cuda.stream(run_s):
            torch.cuda._sleep(2_000_000)                   # let the holding CTAs become resident first
            ev["layer0"].record(run_s)
            layer.forward(li.x, y, idx=idx, w=w, counts=counts, stream=run_s)
            ev["layer1"].record(run_s)
        torch.cuda.synchronize()
        code, word = layer.device_status()
    finally:
        _lib.moe_debug_inject(_lib.MOE_DEBUG_WAIT_LIMIT_NS, 0)
        torch.cuda.synchronize()
        driver.cuModuleUnload(mod)
        driver.cuStreamDestroy(hold_raw)
        driver.cuStreamDestroy(run_raw)
    t = {n: ev["start"].elapsed_time(e) for n, e in ev.items() if n != "start"}
    assert code == _lib.MOE_OK, (_lib.moe_status_string(code), word, t)
    assert int((out > 0).sum()) == n_hold
    # the layer ran while the SMs were held (it finished before the holder did)
    assert t["layer1"] < t["held"], t
    check_layer(wl, li, y, idx, w, counts)
