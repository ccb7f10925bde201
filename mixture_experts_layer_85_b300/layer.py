"""A DeepSeekMoE layer object over the C ABI: packs the experts once, owns the
workspace, and runs ``moe_forward`` (or the four stages) on a stream.

Plumbing only: torch allocates device memory; the library's kernels compute.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import _lib
from .inputs import LayerInputs, Workload, torch_dtype


class MoELayer:
    def __init__(self, wl: Workload, li: LayerInputs, device="cuda", stream=None, keep_unpacked: bool = False):
        self.wl = wl
        self.cfg = _lib.make_config(wl)
        self.device = torch.device(device)
        self.act = torch_dtype(wl.act_dtype)
        self.out_dtype = torch_dtype(wl.out_dtype)
        self.wg = li.wg.to(self.device)
        self.bias = None if li.bias is None else li.bias.to(self.device, torch.float32).contiguous()
        self.packed = torch.empty(_lib.moe_packed_size(self.cfg), dtype=torch.uint8, device=self.device)
        _lib.moe_prepack_experts(self.cfg, li.w1, li.w3, li.w2, li.ws1, li.ws3, li.ws2, self.packed, stream)
        self.ws = torch.empty(_lib.moe_workspace_size(self.cfg), dtype=torch.uint8, device=self.device)
        if keep_unpacked:
            self.unpacked = (li.w1, li.w3, li.w2, li.ws1, li.ws3, li.ws2)

    def variant(self, wl: Workload, bias: Optional[torch.Tensor]) -> "MoELayer":
        """The same layer (packed experts and gate weight shared, not copied)
        under another workload of identical shape: another batch size or
        selection bias.  It owns its own workspace."""
        for f in ("d", "E", "I", "n_shared", "act_dtype", "gate_w_dtype", "expert_w_dtype"):
            if getattr(wl, f) != getattr(self.wl, f):
                raise ValueError(f"variant changes the layer's {f}")
        v = object.__new__(MoELayer)
        v.wl, v.cfg, v.device = wl, _lib.make_config(wl), self.device
        v.act, v.out_dtype = self.act, torch_dtype(wl.out_dtype)
        v.wg, v.packed = self.wg, self.packed
        v.bias = None if bias is None else bias.to(self.device, torch.float32).contiguous()
        v.ws = torch.empty(_lib.moe_workspace_size(v.cfg), dtype=torch.uint8, device=self.device)
        return v

    def forward(self, x: torch.Tensor, out: Optional[torch.Tensor] = None, idx=None, w=None, counts=None,
                stream=None) -> torch.Tensor:
        if out is None:
            out = torch.empty((self.wl.T, self.wl.d), dtype=self.out_dtype, device=self.device)
        _lib.moe_forward(self.cfg, x, self.wg, self.bias, self.packed, out, self.ws, idx, w, counts, stream)
        return out

    def forward_staged(self, x: torch.Tensor, events=None, stream=None):
        """gate_topk -> permute -> grouped_swiglu -> combine as four calls, with
        optional CUDA events recorded between them.  Returns a dict of outputs."""
        T, k, d, E = self.wl.T, self.wl.k, self.wl.d, self.wl.E
        dev = self.device
        o = {
            "idx": torch.empty((T, k), dtype=torch.int32, device=dev),
            "w": torch.empty((T, k), dtype=torch.float32, device=dev),
            "counts": torch.empty((E,), dtype=torch.int32, device=dev),
            "offsets": torch.empty((E + 1,), dtype=torch.int32, device=dev),
            "row2tok": torch.empty((T * k,), dtype=torch.int32, device=dev),
            "tok2row": torch.empty((T, k), dtype=torch.int32, device=dev),
            "x_perm": torch.empty((T * k, d), dtype=self.act, device=dev),
            "y_perm": torch.empty((T * k, d), dtype=torch.float32, device=dev),
            "y_shared": torch.empty((T, d), dtype=torch.float32, device=dev),
            "out": torch.empty((T, d), dtype=self.out_dtype, device=dev),
        }
        rec = (lambda i: events[i].record(stream)) if events is not None else (lambda i: None)
        rec(0)
        _lib.moe_gate_topk(self.cfg, x, self.wg, self.bias, o["idx"], o["w"], self.ws, stream)
        rec(1)
        _lib.moe_permute(self.cfg, x, o["idx"], o["counts"], o["offsets"], o["row2tok"], o["tok2row"], o["x_perm"],
                         self.ws, stream)
        rec(2)
        _lib.moe_grouped_swiglu(self.cfg, o["x_perm"], o["offsets"], x, self.packed, o["y_perm"], o["y_shared"],
                                self.ws, stream)
        rec(3)
        _lib.moe_combine(self.cfg, o["y_perm"], o["y_shared"], o["tok2row"], o["w"], o["out"], self.ws, stream)
        rec(4)
        return o

    def device_status(self, stream=None):
        return _lib.moe_get_device_status(self.ws, stream)
