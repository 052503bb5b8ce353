"""The EPLB loop of one MoE layer ("xDeepServe on CloudMatrix384", section
"专家负载均衡"):

1. Collect (P068): moe_route counts the messages of every physical expert in
   each forward; moe_eplb_collect folds them into the logical experts' load of
   the current time slice on the device.
2. Plan (P069-P076): after a window of n_slices slices, the per-slice loads
   are read back once and the host planner (moe_eplb_plan) selects and places
   the E_phys - E_log redundant copies.
3. Switch (P077): the new map is written into the inactive one of two device
   map versions and the layer takes it from the next forward on.  All of it is
   ordered on the layer's stream, so a forward sees either the old or the new
   map, never a mixture.  Redundant copies alias the weights of their logical
   expert (phys_to_weight), so no weights move.
4. Route (P078-P079): each forward spreads a logical expert's tokens over its
   copies round-robin by token position (inside moe_route).
"""
from __future__ import annotations

import numpy as np
import torch

from . import binding as B
from .layer import MoELayer


class EplbLoop:
    """Drives `layer` (E_phys >= E_log) and re-plans its replica map after
    every window of `n_slices * steps_per_slice` forwards."""

    def __init__(self, layer: MoELayer, n_slices: int = 4, steps_per_slice: int = 8,
                 device="cuda"):
        s = layer.shape
        if s.E_phys < s.E_log or n_slices < 1 or steps_per_slice < 1:
            raise ValueError("EplbLoop needs E_phys >= E_log and positive window sizes")
        self.layer = layer
        self.E_log, self.E_phys, self.R = s.E_log, s.E_phys, s.n_ranks
        self.n_slices, self.steps_per_slice = n_slices, steps_per_slice
        self.max_copies = s.E_phys - s.E_log + 1
        dev = torch.device(device)
        self.load = torch.zeros((n_slices, s.E_log), dtype=torch.int64, device=dev)
        self.maps = [dict(rep=torch.full((s.E_log, self.max_copies), -1, dtype=torch.int32, device=dev),
                          nc=torch.zeros(s.E_log, dtype=torch.int32, device=dev),
                          p2l=torch.zeros(s.E_phys, dtype=torch.int32, device=dev))
                     for _ in range(2)]
        self.version = 0
        self.steps = 0
        self.slice = 0
        self.plans = []  # (loads [n_slices, E_log], rep, n_copies, phys_to_logical) per switch
        # before any statistics: the plan of a uniform load
        self._install(np.ones((1, s.E_log), np.float64), version=0)

    def _install(self, loads: np.ndarray, version: int, stream=None) -> None:
        rep, nc, p2l = B.moe_eplb_plan(loads, self.E_phys, self.R, max_copies=self.max_copies,
                                       trim=False)
        m = self.maps[version]
        st = stream if stream is not None else torch.cuda.current_stream()
        with torch.cuda.stream(st):
            m["rep"].copy_(torch.from_numpy(rep))
            m["nc"].copy_(torch.from_numpy(nc))
            m["p2l"].copy_(torch.from_numpy(p2l))
        self.layer.rep_table, self.layer.n_copies = m["rep"], m["nc"]
        self.layer.phys_to_weight = m["p2l"]
        self.version = version
        self.plans.append((loads, rep, nc, p2l))

    def step(self, logits: torch.Tensor, x: torch.Tensor, stream=None) -> torch.Tensor:
        """One forward with the current map, then Collect; at the end of a
        window, plan and switch to the new map."""
        out = self.layer.forward(logits, x, stream)
        B.moe_eplb_collect(self.layer.buf.routing["expert_counts"], self.load[self.slice],
                           self.maps[self.version]["p2l"], stream)
        self.steps += 1
        if self.steps % self.steps_per_slice == 0:
            self.slice += 1
            if self.slice == self.n_slices:
                self._replan(stream)
                self.slice = 0
        return out

    def _replan(self, stream=None) -> None:
        st = stream if stream is not None else torch.cuda.current_stream()
        with torch.cuda.stream(st):
            loads = self.load.cpu().numpy().astype(np.float64)  # the window's one read-back
            self.load.zero_()
        self._install(loads, version=1 - self.version, stream=st)
