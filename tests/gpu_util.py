"""Helpers shared by the GPU parity tests: build/load the library, put a
workload's seeded inputs on the device, and draw the oracle's view of them."""
from __future__ import annotations

import numpy as np
import torch

from expert_dispatch_combine_gb300 import binding as B
from expert_dispatch_combine_gb300 import synth
from expert_dispatch_combine_gb300.build import build
from expert_dispatch_combine_gb300.layer import LayerBuffers, MoELayer

# bf16 output tolerance of the layer (max abs error, relative L2)
MAX_ABS = 2e-2
REL_L2 = 1e-3

_built = False


def lib():
    global _built
    if not _built:
        build()
        _built = True
    return B.load()


def shape_of(w: synth.Workload, dfmt=B.MOE_MSG_INT8, cfmt=B.MOE_MSG_INT8) -> B.Shape:
    return B.Shape(w.T, w.H, w.E_log, w.E_phys, w.k, w.I, w.R, w.S, dfmt, cfmt)


def bits_to_bf16_tensor(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def bf16_tensor_to_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def eplb_map(w: synth.Workload):
    """Replica map of a workload: plan from the unreplicated routing counts."""
    import oracle
    lg = synth.logits(w)
    _, _, _, cnt = oracle.route(lg, w.k)
    from oracle import eplb
    rep, nc, p2l = eplb.plan(cnt[None, :].astype(np.float64), w.E_phys, w.placement_ranks)
    return rep, nc, p2l


def compare_bf16(got_bits: np.ndarray, ref_bits: np.ndarray):
    g = synth.bf16_bits_to_f32(got_bits).astype(np.float64)
    r = synth.bf16_bits_to_f32(ref_bits).astype(np.float64)
    max_abs = float(np.abs(g - r).max()) if g.size else 0.0
    rel = float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30))
    return max_abs, rel


CANARY_BYTES = 4096
CANARY = 0xA5


def _guarded(nbytes: int, dtype, shape, device, tails: list):
    """A caller buffer of `nbytes` followed by CANARY_BYTES of the canary byte
    (a separate allocation per buffer, so its start keeps torch's alignment);
    the tail view goes to `tails`."""
    raw = torch.empty(nbytes + CANARY_BYTES, dtype=torch.uint8, device=device)
    raw[nbytes:].fill_(CANARY)
    tails.append(raw[nbytes:])
    return raw[:nbytes].view(dtype).view(shape)


class CanaryBuffers(LayerBuffers):
    """LayerBuffers in which every buffer the library writes (dispatch,
    combine, workspace, output, routing arrays) is followed by canary bytes;
    check() asserts that no kernel wrote past the end of any of them."""

    def __init__(self, shape, device="cuda"):
        dev = torch.device(device)
        self.tails = []
        self._dev = dev
        super().__init__(shape, device)

    def _alloc(self, shape, dtype, device):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        return _guarded(n, dtype, shape, self._dev, self.tails)

    def check(self):
        torch.cuda.synchronize()
        for t in self.tails:
            assert bool((t == CANARY).all()), "a kernel wrote past the end of a caller buffer"


def make_layer(w: synth.Workload, cfmt=B.MOE_MSG_INT8, device="cuda", canary=True, f16_weights=False):
    """MoELayer with the workload's weights resident on the device (plus the
    EPLB map for replicated workloads); with `canary` its buffers carry
    canary tails (CanaryBuffers); with `f16_weights` it also keeps the fp16
    weight copies that the tensor-core GEMMs of large batches read."""
    shape = shape_of(w, B.MOE_MSG_INT8, cfmt)
    w_gu, s_gu, w_d, s_d = synth.all_weights_torch(w, device)
    rep = nc = p2l = None
    if w.eplb:
        r, n, p = eplb_map(w)
        rep, nc, p2l = (torch.from_numpy(a).to(device) for a in (r, n, p))
    return MoELayer(shape, w_gu, s_gu, w_d, s_d, rep_table=rep, n_copies=nc, phys_to_weight=p2l,
                    device=device, buffers=CanaryBuffers(shape, device) if canary else None,
                    f16_weights=f16_weights)


__all__ = ["lib", "shape_of", "bits_to_bf16_tensor", "bf16_tensor_to_bits", "compare_bf16",
           "make_layer", "eplb_map", "LayerBuffers", "CanaryBuffers", "MAX_ABS", "REL_L2"]
