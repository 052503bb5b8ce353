"""Device buffers for one MoE layer shape and a convenience wrapper around moe_layer.

PyTorch provides the device memory and the stream; every step of the layer
runs in the CUDA library through the C ABI (binding.py).
"""
from __future__ import annotations

import torch

from . import binding as B
from .binding import Shape


class LayerBuffers:
    """Caller-owned buffers sized by moe_query_layout (torch allocations are
    512-byte aligned, which covers the ABI's 256-byte rule)."""

    def __init__(self, shape: Shape, device="cuda"):
        self.shape = shape
        self.layout = L = B.moe_query_layout(shape)
        T, k = shape.T, shape.k
        dev = torch.device(device)
        self.dispatch = torch.empty(L["dispatch_bytes"], dtype=torch.uint8, device=dev)
        self.combine = torch.empty(L["combine_bytes"], dtype=torch.uint8, device=dev)
        self.workspace = torch.empty(max(256, L["workspace_bytes"]), dtype=torch.uint8, device=dev)
        self.routing = dict(
            topk_idx=torch.empty((T, k), dtype=torch.int32, device=dev),
            topk_w=torch.empty((T, k), dtype=torch.float32, device=dev),
            phys_idx=torch.empty((T, k), dtype=torch.int32, device=dev),
            expert_counts=torch.empty(shape.E_phys, dtype=torch.int32, device=dev),
            rank_counts=torch.empty((shape.n_ranks, shape.n_src_ranks), dtype=torch.int32, device=dev),
            expert_offsets=torch.empty(shape.E_phys + 1, dtype=torch.int32, device=dev),
            expert_rows=torch.empty(T * k, dtype=torch.int32, device=dev),
        )
        self.out = torch.empty((T, shape.H), dtype=torch.bfloat16, device=dev)

    # views into the static buffers
    def dispatch_rows(self) -> torch.Tensor:
        L, s = self.layout, self.shape
        n = s.n_ranks * s.n_src_ranks * L["max_tokens"]
        return self.dispatch[: n * L["dispatch_row_bytes"]].view(n, L["dispatch_row_bytes"])

    def dispatch_meta(self) -> torch.Tensor:
        """[slots, 4] int32 view: (scale bits, src_rank, batch_slot, route_slot)."""
        L, s = self.layout, self.shape
        n = s.n_ranks * s.n_src_ranks * L["max_tokens"]
        off = L["dispatch_meta_offset"]
        return self.dispatch[off: off + 16 * n].view(torch.int32).view(n, 4)

    def combine_rows(self) -> torch.Tensor:
        L, s = self.layout, self.shape
        n = s.T * s.k
        return self.combine[: n * L["combine_row_bytes"]].view(s.T, s.k, L["combine_row_bytes"])

    def combine_scales(self) -> torch.Tensor:
        L, s = self.layout, self.shape
        off = L["combine_scale_offset"]
        return self.combine[off: off + 4 * s.T * s.k].view(torch.float32).view(s.T, s.k)


class MoELayer:
    """One MoE layer with resident INT8 expert weights.

    forward(logits, x) runs route -> FusedDispatch -> experts -> FusedCombine
    through moe_layer and returns the bf16 output tensor (a view of the
    layer's output buffer)."""

    def __init__(self, shape: Shape, w_gate_up, s_gate_up, w_down, s_down, rep_table=None,
                 n_copies=None, phys_to_weight=None, device="cuda"):
        self.shape = shape
        self.w = (w_gate_up, s_gate_up, w_down, s_down)
        self.rep_table, self.n_copies, self.phys_to_weight = rep_table, n_copies, phys_to_weight
        self.buf = LayerBuffers(shape, device)

    def forward(self, logits: torch.Tensor, x: torch.Tensor, stream=None) -> torch.Tensor:
        b = self.buf
        B.moe_layer(self.shape, logits, x, *self.w, b.routing, b.dispatch, b.combine, b.workspace,
                    b.out, rep_table=self.rep_table, n_copies=self.n_copies,
                    phys_to_weight=self.phys_to_weight, stream=stream)
        return b.out


class GraphedLayer:
    """The decode layer replayed from CUDA graphs over `n_sets` static buffer
    sets (two: double buffering).  Step i copies its inputs into set
    i % n_sets, launches that set's graph (one moe_layer captured by
    moe_layer_graph_create) and returns that set's output buffer, so two
    consecutive steps never share dispatch, combine or output buffers."""

    def __init__(self, layer: MoELayer, n_sets: int = 2, device="cuda"):
        s = layer.shape
        self.layer = layer
        self.sets = []
        self.next = 0
        cap = torch.cuda.Stream(device=device)
        dev = torch.device(device)
        for _ in range(n_sets):
            buf = LayerBuffers(s, device)
            lg = torch.zeros((s.T, s.E_log), dtype=torch.float32, device=dev)
            x = torch.zeros((s.T, s.H), dtype=torch.bfloat16, device=dev)
            g = B.moe_layer_graph_create(s, lg, x, *layer.w, buf.routing, buf.dispatch, buf.combine,
                                         buf.workspace, buf.out, cap, rep_table=layer.rep_table,
                                         n_copies=layer.n_copies, phys_to_weight=layer.phys_to_weight)
            self.sets.append((buf, lg, x, g))

    def step(self, logits: torch.Tensor, x: torch.Tensor, stream=None) -> torch.Tensor:
        buf, lg, xs, g = self.sets[self.next]
        self.next = (self.next + 1) % len(self.sets)
        st = stream if stream is not None else torch.cuda.current_stream()
        with torch.cuda.stream(st):
            lg.copy_(logits)
            xs.copy_(x)
        B.moe_graph_launch(g, st)
        return buf.out

    def close(self) -> None:
        for _, _, _, g in self.sets:
            B.moe_graph_destroy(g)
        self.sets = []

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
