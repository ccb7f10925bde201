"""The C ABI library on the CPU: it loads, exports every declared symbol, and
rejects bad arguments on the host before any launch (no GPU needed)."""
import ctypes
import os
import re

import pytest

from mixture_experts_layer_85_b300 import _lib, inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    return re.findall(r"^MOE_API\s+[\w\s\*]+?\b(moe_\w+)\(", src, flags=re.M)


def test_exports_every_declared_symbol():
    names = declared_symbols()
    assert len(names) >= 12
    lib = ctypes.CDLL(_lib.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(names) == sorted(_lib.EXPORTED)


def test_status_strings():
    for code in range(8):
        assert _lib.moe_status_string(code).startswith("MOE_")
    assert _lib.moe_status_string(_lib.MOE_ERR_DEVICE_RANGE) == "MOE_ERR_DEVICE_RANGE"
    assert _lib.moe_status_string(99) == "MOE_ERR_UNKNOWN"


@pytest.mark.parametrize("name", inputs.CONFIG_ORDER)
def test_sizes_for_every_workload(name):
    wl = inputs.WORKLOADS[name]
    cfg = _lib.make_config(wl)
    ws = _lib.moe_workspace_size(cfg)
    pk = _lib.moe_packed_size(cfg)
    eb = 2 if wl.act_dtype == "bf16" else 4
    # packed blob holds all expert weights exactly once (plus alignment)
    weights = (3 * wl.E * wl.I * wl.d + 3 * wl.I_s * wl.d) * eb
    assert weights <= pk <= weights + 4 * 256
    # workspace holds at least the permuted rows, hidden and outputs
    assert ws >= (2 * wl.R * wl.d + wl.R * wl.I) * eb
    # router (+ the fp32 gate-weight split on the tensor-core path), dispatch
    # (one block up to 4096 tokens, four kernels above), gather, the expert
    # GEMMs (one fused launch on the tensor-core path, two SIMT kernels in fp32),
    # combine
    bf16 = wl.act_dtype == "bf16"
    gate = 2 + (1 if bf16 and wl.gate_w_dtype == "f32" else 0)
    dispatch = 1 if wl.T <= 4096 else 4
    experts = (1 if wl.T * wl.k <= 8192 else 2) if bf16 else 2   # one fused launch for small batches
    assert _lib.moe_forward_kernel_count(cfg) == gate + dispatch + 1 + experts + 1


@pytest.mark.parametrize("name,experts", [("v3_decode_fp8_t1", 2), ("v3_decode_fp8_t64", 2),
                                          ("v3_decode_fp8_t512", 1), ("v3_prefill_fp8_t16384", 2)])
def test_fp8_kernel_count(name, experts):
    """FP8 layers: batches of at most 64 tokens run the GEMV (GEMM1, then
    GEMM2); larger ones the tensor-core kernel, fused up to 8192 rows."""
    wl = inputs.WORKLOADS[name]
    cfg = _lib.make_config(wl)
    dispatch = 1 if wl.T <= 4096 else 4
    assert _lib.moe_forward_kernel_count(cfg) == 2 + dispatch + 1 + experts + 1


def _cfg(**kw):
    c = _lib.make_config(inputs.WORKLOADS["v3_prefill_t16384"])
    for k, v in kw.items():
        setattr(c, k, v)
    return c


@pytest.mark.parametrize("kw,code", [
    (dict(E=0), _lib.MOE_ERR_INVALID_ARG),
    (dict(k=300), _lib.MOE_ERR_INVALID_ARG),
    (dict(act_dtype=7), _lib.MOE_ERR_INVALID_ARG),
    (dict(n_group=3), _lib.MOE_ERR_INVALID_ARG),            # 256 % 3 != 0
    (dict(topk_group=9), _lib.MOE_ERR_INVALID_ARG),         # > n_group
    (dict(topk_group=1, k=40), _lib.MOE_ERR_INVALID_ARG),   # k > experts in kept groups
    (dict(group_top=0), _lib.MOE_ERR_INVALID_ARG),
    (dict(T=-1), _lib.MOE_ERR_INVALID_ARG),
    (dict(T=1 << 28), _lib.MOE_ERR_INVALID_ARG),            # T*k overflows the row index
    (dict(E=512, n_group=8), _lib.MOE_ERR_UNSUPPORTED),
    (dict(I=2000), _lib.MOE_ERR_UNSUPPORTED),               # bf16 tiles need I % 128 == 0
    (dict(d=7000), _lib.MOE_ERR_UNSUPPORTED),
])
def test_bad_config_rejected(kw, code):
    c = _cfg(**kw)
    n = ctypes.c_size_t(0)
    assert _lib.raw_call("moe_workspace_size", ctypes.byref(c), ctypes.byref(n)) == code


def test_null_and_misaligned_pointers_rejected_before_launch():
    c = _cfg(T=64)
    ws_need = _lib.moe_workspace_size(c)
    fake = 1 << 40                     # never dereferenced: validation fails first
    assert _lib.raw_call("moe_forward", ctypes.byref(c), None, fake, None, fake, fake, None, None, None,
                         fake, ws_need, None) == _lib.MOE_ERR_INVALID_ARG
    assert _lib.raw_call("moe_forward", ctypes.byref(c), fake + 8, fake, None, fake, fake, None, None, None,
                         fake, ws_need, None) == _lib.MOE_ERR_INVALID_ARG
    assert _lib.raw_call("moe_forward", ctypes.byref(c), fake, fake, None, fake, fake, None, None, None,
                         fake, ws_need - 1, None) == _lib.MOE_ERR_WORKSPACE
    assert _lib.raw_call("moe_gate_topk", ctypes.byref(c), fake, fake, None, None, fake, fake, ws_need,
                         None) == _lib.MOE_ERR_INVALID_ARG
    assert _lib.raw_call("moe_prepack_experts", ctypes.byref(c), fake, fake, fake, fake, fake, fake, fake, 16,
                         None) == _lib.MOE_ERR_WORKSPACE
    assert _lib.raw_call("moe_combine", None, fake, fake, fake, fake, fake, fake, ws_need,
                         None) == _lib.MOE_ERR_INVALID_ARG


def test_empty_batch_launches_nothing():
    c = _cfg(T=0)
    before = _lib.moe_launch_count()
    fake = 1 << 40
    ws = _lib.moe_workspace_size(c)
    assert _lib.raw_call("moe_forward", ctypes.byref(c), fake, fake, None, fake, fake, None, None, None,
                         fake, ws, None) == _lib.MOE_OK
    assert _lib.moe_forward_kernel_count(c) == 0
    assert _lib.moe_launch_count() == before


def test_backward_workspace_and_argument_checks():
    """moe_backward: bf16 layers with bf16 expert weights only; its workspace
    holds the forward's; null, misaligned or short arguments are rejected
    before any launch."""
    c = _cfg(T=64)
    need = _lib.moe_backward_workspace_size(c)
    assert need > _lib.moe_workspace_size(c)
    for kw in (dict(act_dtype=_lib.MOE_F32, gate_w_dtype=_lib.MOE_F32, out_dtype=_lib.MOE_F32,
                    expert_w_dtype=_lib.MOE_F32),
               dict(expert_w_dtype=_lib.MOE_FP8_E4M3)):
        bad = _cfg(T=64, **kw)
        n = ctypes.c_size_t(0)
        assert _lib.raw_call("moe_backward_workspace_size", ctypes.byref(bad), ctypes.byref(n)) == \
            _lib.MOE_ERR_UNSUPPORTED
    fake = 1 << 40                     # never dereferenced: validation fails first
    ptrs = [fake] * 18                 # x, Wg, bias, W1, W3, W2, Ws1, Ws3, Ws2, dout, dx, dWg, dW1..dWs2
    before = _lib.moe_launch_count()
    args = list(ptrs)
    args[0] = None                     # x
    assert _lib.raw_call("moe_backward", ctypes.byref(c), *args, fake, need, None) == _lib.MOE_ERR_INVALID_ARG
    args = list(ptrs)
    args[11] = fake + 4                # dWg misaligned
    assert _lib.raw_call("moe_backward", ctypes.byref(c), *args, fake, need, None) == _lib.MOE_ERR_INVALID_ARG
    assert _lib.raw_call("moe_backward", ctypes.byref(c), *ptrs, fake, need - 1, None) == _lib.MOE_ERR_WORKSPACE
    assert _lib.moe_launch_count() == before


@pytest.mark.parametrize("name", ["v3_decode_fp8_t1", "v3_prefill_fp8_t16384", "v3_profile_fp8_e16_t1"])
def test_fp8_packed_size_is_the_stage_image_layout(name):
    """FP8 packed experts: each matrix as (rows / 128 + 1) tiles of K / 128 stage
    blocks of 128 x 128 e4m3 bytes plus 2 x 128 int32 scale exponents, 256-byte
    aligned, then the reference exponents int32 [E + 1][3]."""
    wl = inputs.WORKLOADS[name]
    cfg = _lib.make_config(wl)
    stage = 128 * 128 + 2 * 128 * 4
    al = lambda v: (v + 255) // 256 * 256
    tiled = lambda rows, cols: (rows // 128 + 1) * (cols // 128) * stage
    E, I, d, Is = wl.E, wl.I, wl.d, wl.I_s
    total = 0
    for rows, cols in ((2 * E * I, d), (E * d, I), (2 * Is, d), (d, Is)):
        total = al(total + tiled(rows, cols))
    total = al(total + (E + 1) * 3 * 4)
    assert _lib.moe_packed_size(cfg) == total
    # about 1.0625 bytes per weight (plus one padding tile per matrix)
    weights = 3 * E * I * d + 3 * Is * d
    assert 1.0625 * weights <= total <= 1.0625 * weights + 4 * (d // 128 + I // 128) * stage * 2 + 4096


def test_debug_inject_validates_knobs():
    assert _lib.raw_call("moe_debug_inject", 7, 0) == _lib.MOE_ERR_INVALID_ARG
    assert _lib.raw_call("moe_debug_inject", _lib.MOE_DEBUG_WAIT_LIMIT_NS, -1) == _lib.MOE_ERR_INVALID_ARG
    assert _lib.raw_call("moe_debug_inject", _lib.MOE_DEBUG_WAIT_LIMIT_NS, 10) == _lib.MOE_ERR_INVALID_ARG
    assert _lib.raw_call("moe_debug_inject", _lib.MOE_DEBUG_STALL_GEMM2, 2) == _lib.MOE_ERR_INVALID_ARG
    assert _lib.raw_call("moe_debug_inject", _lib.MOE_DEBUG_WAIT_LIMIT_NS, 1000000) == _lib.MOE_OK
    assert _lib.raw_call("moe_debug_inject", _lib.MOE_DEBUG_WAIT_LIMIT_NS, 0) == _lib.MOE_OK
    assert _lib.raw_call("moe_debug_inject", _lib.MOE_DEBUG_STALL_GEMM2, 0) == _lib.MOE_OK


@pytest.mark.parametrize("d,I,E,n_shared", [(320, 128, 12, 1), (2048, 1408, 64, 2), (7168, 2048, 256, 1)])
def test_bf16_packed_size_is_the_stage_block_layout(d, I, E, n_shared):
    """bf16 packed experts: each matrix as groups x ceil(rows / 128) x ceil(cols / 128)
    blocks of 128 x 128 bf16 (32 KB), each matrix 256-byte aligned."""
    wl = inputs.small_workload(inputs.WORKLOADS["v3_prefill_t16384"], name="pk", T=8, d=d, E=E, I=I,
                               n_shared=n_shared, n_group=4, topk_group=2, k=4)
    cfg = _lib.make_config(wl)
    blk = 128 * 128 * 2

    def mat(groups, rows, cols):
        return groups * -(-rows // 128) * -(-cols // 128) * blk

    Is = n_shared * I
    parts = [mat(E, 2 * I, d), mat(E, d, I), mat(1, 2 * Is, d), mat(1, d, Is)]
    total = 0
    for part in parts:
        total = -(-(total + part) // 256) * 256
    assert _lib.moe_packed_size(cfg) == total


@pytest.mark.parametrize("name", sorted(inputs.WORKLOADS))
def test_bench_expert_kernel_matches_the_library(name):
    """The bench line's roofline names the expert stage's kernel and its
    launches per forward; the count agrees with the library's own."""
    import sys
    sys.path.insert(0, ROOT)
    import bench
    wl = inputs.WORKLOADS[name]
    cfg = _lib.make_config(wl)
    kernel, launches = bench.expert_kernel(wl)
    bf16 = wl.act_dtype == "bf16"
    gate = 2 + (1 if bf16 and wl.gate_w_dtype == "f32" else 0)
    dispatch = 1 if wl.T <= 4096 else 4
    assert _lib.moe_forward_kernel_count(cfg) == gate + dispatch + 1 + launches + 1
    assert kernel.startswith("gemv_fp8_kernel") == (wl.expert_w_dtype == "fp8" and wl.T <= 64)
