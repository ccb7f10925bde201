"""moe_permute_noalloc against moe_permute, through the C ABI.

The no-allocation entry point serves callers that cannot call cudaMalloc or
hand the library a workspace (a host framework owns their device memory, a
hard memory budget, or a loop that must not risk cudaMalloc blocking the
device).  Its scratch is one fixed array in the library's device image that
every call reuses, so calls in a row must each match the workspace version
exactly (integer outputs and copied rows: bit for bit).  Batches above 4096
tokens take the multi-block dispatch, the only path that reads the array's
per-chunk tables.  This file is collected last on purpose."""
import ctypes

import pytest
import torch

from mixture_experts_layer_85_b300 import _lib, inputs

pytestmark = pytest.mark.gpu


def _case(T, E, k, d, seed):
    wl = inputs.small_workload(inputs.WORKLOADS["v2lite_t4096"], name="noalloc", T=T, d=d, E=E, I=128, k=k)
    cfg = _lib.make_config(wl)
    idx = inputs.random_idx(T, E, k, seed=seed).cuda()
    x = inputs.random_rows(T, d, seed=seed).cuda()
    return wl, cfg, idx, x


def _outputs(T, E, k, d):
    i32 = dict(dtype=torch.int32, device="cuda")
    return {"counts": torch.full((E,), -1, **i32), "offsets": torch.full((E + 1,), -1, **i32),
            "row2tok": torch.full((T * k,), -1, **i32), "tok2row": torch.full((T, k), -1, **i32),
            "x_perm": torch.zeros((T * k, d), dtype=torch.bfloat16, device="cuda")}


def _run_both(T, E, k, d, seed):
    wl, cfg, idx, x = _case(T, E, k, d, seed)
    ref = _outputs(T, E, k, d)
    ws = torch.empty(_lib.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    _lib.moe_permute(cfg, x, idx, ref["counts"], ref["offsets"], ref["row2tok"], ref["tok2row"], ref["x_perm"], ws)
    got = _outputs(T, E, k, d)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    _lib.moe_permute_noalloc(cfg, x, idx, got["counts"], got["offsets"], got["row2tok"], got["tok2row"],
                             got["x_perm"], status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert _lib.moe_get_device_status(ws)[0] == _lib.MOE_OK
    for name in ref:
        assert torch.equal(got[name], ref[name]), name


def test_noalloc_matches_workspace_version_calls_in_a_row():
    # Every call reuses the array the one before left behind.  Both shapes take
    # the multi-block path; the second has more chunks and fewer experts, so a
    # table entry the first call wrote and the second failed to overwrite would
    # show up in its counts or rows.
    _run_both(T=4133, E=256, k=8, d=256, seed=1)
    _run_both(T=9000, E=160, k=6, d=128, seed=2)
    _run_both(T=777, E=160, k=6, d=128, seed=3)     # one-block path after the multi-block ones


def test_noalloc_at_its_exact_capacity():
    # 128 chunks of 128 tokens times 256 experts fill both tables exactly
    _run_both(T=16384, E=256, k=8, d=128, seed=4)


def test_noalloc_empty_batch_clears_status():
    wl, cfg, idx, x = _case(T=8, E=16, k=2, d=128, seed=5)
    cfg.T = 0
    out = _outputs(8, 16, 2, 128)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    _lib.moe_permute_noalloc(cfg, x, idx, out["counts"], out["offsets"], out["row2tok"], out["tok2row"],
                             out["x_perm"], status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert int(out["counts"].abs().sum()) == 0 and int(out["offsets"].abs().sum()) == 0


def test_noalloc_rejects_sizes_beyond_its_array():
    wl, cfg, idx, x = _case(T=8, E=16, k=2, d=128, seed=3)
    cfg.T, cfg.E = 16385 + 128, 256           # 130 chunks * 256 experts > 32768 entries
    big = 1 << 40                             # never touched: the size check comes first
    rc = _lib.raw_call("moe_permute_noalloc", ctypes.byref(cfg), big, big, big, big, big, big, big, None, None)
    assert rc == _lib.MOE_ERR_WORKSPACE
