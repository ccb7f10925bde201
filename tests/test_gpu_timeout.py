"""The device-side time-out path of the expert GEMM kernel, exercised without a
fault: the host makes one bounded wait impossible to satisfy (every GEMM2 tile
of a one-launch expert kernel waits for one more GEMM1 completion than its
group produces) and shortens the wait limit to 1 ms.  The call must end on its
own, report MOE_ERR_DEVICE_TIMEOUT through the status word, and leave the
context usable: the next normal call on the same layer matches the oracle."""
import pytest
import torch

from mixture_experts_layer_85_b300 import _lib, inputs
from mixture_experts_layer_85_b300.layer import MoELayer
from tests.test_gpu_parity import check_layer, run_layer

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T", [3, 200])
def test_stalled_gemm2_wait_times_out_and_the_next_call_is_correct(T):
    wl = inputs.small_workload(inputs.WORKLOADS["v3_prefill_t16384"], name=f"v3_timeout_t{T}", T=T, d=512,
                               E=64, I=256, n_group=8, topk_group=4)
    li = inputs.make_inputs(wl, "cuda")
    layer = MoELayer(wl, li, "cuda")
    layer.forward(li.x)                       # a normal call first
    assert layer.device_status()[0] == _lib.MOE_OK
    _lib.moe_debug_inject(_lib.MOE_DEBUG_WAIT_LIMIT_NS, 1_000_000)
    _lib.moe_debug_inject(_lib.MOE_DEBUG_STALL_GEMM2, 1)
    try:
        layer.forward(li.x)
        code, word = layer.device_status()
    finally:
        _lib.moe_debug_inject(_lib.MOE_DEBUG_STALL_GEMM2, 0)
        _lib.moe_debug_inject(_lib.MOE_DEBUG_WAIT_LIMIT_NS, 0)
    assert code == _lib.MOE_ERR_DEVICE_TIMEOUT and (word & 1), (code, word)
    torch.cuda.synchronize()
    _, out, idx, w, counts = run_layer(wl, li)
    check_layer(wl, li, out, idx, w, counts)
