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
    n_hold = n_sm - 48                                     # leaves 24 pairs of SMs (n_sm is even)
    side = torch.cuda.Stream()
    out = torch.zeros(n_hold, dtype=torch.int32, device="cuda")
    args = ((HOLD_NS, out.data_ptr()), (ctypes.c_ulonglong, ctypes.c_void_p))
    idx = torch.empty((T, wl.k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, wl.k), dtype=torch.float32, device="cuda")
    counts = torch.empty((wl.E,), dtype=torch.int32, device="cuda")
    _lib.moe_debug_inject(_lib.MOE_DEBUG_WAIT_LIMIT_NS, 20_000_000)
    try:
        start = torch.cuda.Event(enable_timing=True)
        start.record(side)
        _check(driver.cuLaunchKernel(fn, n_hold, 1, 1, 32, 1, 1, HOLD_SMEM, driver.CUstream(side.cuda_stream),
                                     args, 0))
        # the layer on the default stream, while the SMs are held
        torch.cuda._sleep(1_000_000)                       # let the holding CTAs become resident first
        y = layer.forward(li.x, idx=idx, w=w, counts=counts)
        done = torch.cuda.Event(enable_timing=True)
        done.record()
        held = torch.cuda.Event(enable_timing=True)
        held.record(side)
        torch.cuda.synchronize()
        code, word = layer.device_status()
    finally:
        _lib.moe_debug_inject(_lib.MOE_DEBUG_WAIT_LIMIT_NS, 0)
        torch.cuda.synchronize()
        driver.cuModuleUnload(mod)
    assert code == _lib.MOE_OK, (_lib.moe_status_string(code), word)
    assert int((out > 0).sum()) == n_hold
    # the layer ran while the SMs were held (it finished before the holder did)
    assert start.elapsed_time(done) < start.elapsed_time(held), (start.elapsed_time(done), start.elapsed_time(held))
    check_layer(wl, li, y, idx, w, counts)
