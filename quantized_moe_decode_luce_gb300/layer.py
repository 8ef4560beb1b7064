"""One MoE-FFN decode step through the C ABI, with torch-owned buffers.

:class:`MoEStep` allocates (once, with torch) every intermediate buffer of
the step for a fixed token count and runs the five calls of the step in the
pages' order on one stream: route select + weights, q8_1 quantization of
the FFN input, expert grouping (one fused launch for the first three when
it fits one CTA), gate/up pair + SwiGLU, down + combine.
Allocation is torch's; all arithmetic is in libluce_moe's kernels.
"""
from __future__ import annotations

import torch

from . import binding as B
from .workloads import QK, Q8_1_BYTES


class MoEStep:
    def __init__(self, T: int, H: int, I: int, E: int, k: int, shared: bool, clamp: float, device="cuda"):
        self.T, self.H, self.I, self.E, self.k = T, H, I, E, k
        self.shared, self.clamp = shared, float(clamp)
        dev = torch.device(device)
        rows = T * k + (T if shared else 0)
        self.ids = torch.empty((T, k), dtype=torch.int32, device=dev)
        self.weights = torch.empty((T, k), dtype=torch.float32, device=dev)
        self.xq = torch.empty((T, H // QK, Q8_1_BYTES), dtype=torch.uint8, device=dev)
        self.counts = torch.empty(E, dtype=torch.int32, device=dev)
        self.offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
        self.routes = torch.empty(max(1, T * k), dtype=torch.int32, device=dev)
        self.h = torch.empty((max(1, rows), I), dtype=torch.float32, device=dev)
        self.hq = torch.empty((max(1, rows), I // QK, Q8_1_BYTES), dtype=torch.uint8, device=dev)
        self.out = torch.empty((T, H), dtype=torch.float32, device=dev)
        # luce_moe_layer's workspace: its barrier count (first 8 bytes, zero) and scratch
        self.workspace = torch.zeros(B.luce_moe_layer_workspace_bytes(T, k, H, I), dtype=torch.uint8, device=dev)
        self.fused_prep = True
        # "layer": luce_moe_layer -- one cooperative launch for T <= 8, T*k <= 64,
        # E <= 256 (bitwise the results of the split launches), the grouped
        # tensor-core path for more tokens; "split": the separate launches.
        self.path = "split" if (T <= 8 and T * k <= 64 and E > 256) else "layer"

    def run(self, layer, x, logits, bias=None, stream=None, out=None) -> torch.Tensor:
        """layer: object with wg, wu, wd (+ wsg, wsu, wsd) uint8 CUDA tensors.
        Writes the layer output into `out` (default: this step's own buffer)."""
        out = self.out if out is None else out
        T, H, I, E, k = self.T, self.H, self.I, self.E, self.k
        wsg = layer.wsg if self.shared else None
        wsu = layer.wsu if self.shared else None
        wsd = layer.wsd if self.shared else None
        if self.path == "layer":
            try:
                B.luce_moe_layer(logits, bias, x, k, I, layer.wg, layer.wu, layer.wd, wsg, wsu, wsd, self.clamp,
                                 self.ids, self.weights, self.xq, self.counts, self.offsets, self.routes, self.h,
                                 self.hq, out, self.workspace, stream)
                return out
            except B.LuceError as err:
                if err.status != B.LUCE_ERR_UNSUPPORTED:
                    raise
                self.path = "split"  # beyond the one-launch limits: the split launches (nothing ran)
        if self.fused_prep:
            B.luce_moe_prep(logits, bias, x, k, self.ids, self.weights, self.xq, self.counts, self.offsets,
                            self.routes, stream)
        else:
            B.luce_route_topk(logits, bias, k, self.ids, self.weights, stream)
            B.luce_quantize_q8_1(x, self.xq, stream)
            B.luce_moe_group(self.ids, E, self.counts, self.offsets, self.routes, stream)
        B.luce_moe_glu_pair(layer.wg, layer.wu, wsg, wsu, self.xq, self.offsets, self.routes, T, k, E, H, I,
                            self.clamp, self.h, self.hq, 0, stream)
        B.luce_moe_down_combine(layer.wd, wsd, self.hq, self.ids, self.weights, self.offsets, self.routes,
                                T, k, E, H, I, out, 0, stream)
        return out


class Argmax:
    """Greedy argmax over [R, V] logits with its own zero-filled workspace."""

    def __init__(self, R: int, V: int, device="cuda"):
        self.R, self.V = R, V
        n = max(16, B.luce_argmax_workspace_bytes(R, V))
        self.workspace = torch.zeros(n, dtype=torch.uint8, device=device)
        self.idx = torch.empty(R, dtype=torch.int32, device=device)
        self.val = torch.empty(R, dtype=torch.float32, device=device)

    def run(self, logits, stream=None):
        B.luce_argmax(logits, self.idx, self.val, self.workspace, stream)
        return self.idx, self.val
