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
        a = self._alloc
        self.dispatch = a((L["dispatch_bytes"],), torch.uint8, dev)
        self.combine = a((L["combine_bytes"],), torch.uint8, dev)
        self.workspace = a((max(256, L["workspace_bytes"]),), torch.uint8, dev)
        self.routing = dict(
            topk_idx=a((T, k), torch.int32, dev),
            topk_w=a((T, k), torch.float32, dev),
            phys_idx=a((T, k), torch.int32, dev),
            expert_counts=a((shape.E_phys,), torch.int32, dev),
            rank_counts=a((shape.n_ranks, shape.n_src_ranks), torch.int32, dev),
            expert_offsets=a((shape.E_phys + 1,), torch.int32, dev),
            expert_rows=a((T * k,), torch.int32, dev),
        )
        self.out = a((T, shape.H), torch.bfloat16, dev)

    def _alloc(self, shape, dtype, device) -> torch.Tensor:
        return torch.empty(shape, dtype=dtype, device=device)

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
    layer's output buffer).

    f16_weights=True also keeps exact fp16 copies of the two weight arrays
    (moe_weights_to_f16, made once here): batches above the decode size then
    run the tensor-core GEMMs on them, with the same outputs bit for bit, at
    twice the weight bytes held."""

    def __init__(self, shape: Shape, w_gate_up, s_gate_up, w_down, s_down, rep_table=None,
                 n_copies=None, phys_to_weight=None, device="cuda", buffers: LayerBuffers | None = None,
                 f16_weights: bool = False):
        self.shape = shape
        self.w = (w_gate_up, s_gate_up, w_down, s_down)
        self.w_f16 = (B.moe_weights_to_f16(w_gate_up), B.moe_weights_to_f16(w_down)) \
            if f16_weights else None
        self.rep_table, self.n_copies, self.phys_to_weight = rep_table, n_copies, phys_to_weight
        self.buf = buffers if buffers is not None else LayerBuffers(shape, device)

    def forward(self, logits: torch.Tensor, x: torch.Tensor, stream=None) -> torch.Tensor:
        b = self.buf
        B.moe_layer(self.shape, logits, x, *self.w, b.routing, b.dispatch, b.combine, b.workspace,
                    b.out, rep_table=self.rep_table, n_copies=self.n_copies,
                    phys_to_weight=self.phys_to_weight, stream=stream, w_f16=self.w_f16)
        return b.out

    def forward_host(self, h_logits: torch.Tensor, h_x: torch.Tensor, h_out: torch.Tensor,
                     stream=None) -> None:
        """Host to host through moe_layer_host: h_logits f32 [T, E_log], h_x and
        h_out 16-bit [T, H] CPU tensors (page-locked for asynchronous copies).
        h_out holds the output once `stream` has passed this call."""
        b = self.buf
        if not hasattr(self, "_stage"):
            s = self.shape
            dev = b.out.device
            self._stage = (torch.empty((s.T, s.E_log), dtype=torch.float32, device=dev),
                           torch.empty((s.T, s.H), dtype=torch.int16, device=dev))
        d_lg, d_x = self._stage
        B.moe_layer_host(self.shape, h_logits, h_x, h_out, d_lg, d_x, *self.w, b.routing, b.dispatch,
                         b.combine, b.workspace, b.out, rep_table=self.rep_table,
                         n_copies=self.n_copies, phys_to_weight=self.phys_to_weight, stream=stream,
                         w_f16=self.w_f16)


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
                                         n_copies=layer.n_copies, phys_to_weight=layer.phys_to_weight,
                                         w_f16=layer.w_f16)
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
