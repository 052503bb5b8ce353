#!/usr/bin/env python
"""Benchmark of the decode-time MoE layer on GB300.

One step = one pass of the whole layer (gate top-k route -> INT8
FusedDispatch -> grouped W8A8 SwiGLU experts -> FusedCombine) over one batch
of the seeded synthetic workload, through moe_layer.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...     # the CPU oracle on host cores

Prints one JSON line (rank 0).  With N > 1 (torchrun) every rank runs an
independent replica of the layer (no data-path collective) and `value` is
the aggregate tokens/s over all ranks (weak scaling).
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from expert_dispatch_combine_gb300 import synth  # noqa: E402

DEFAULT_WORKLOAD = "c2_decode_zipf"
METRIC = "routed tokens/s per MoE layer on 1 GB300; dispatch/combine us and % HBM roofline"
UNIT = "tokens/s"
L2_BYTES = 129 * 1024 * 1024


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


FFN_TC_SRC = os.path.join(ROOT, "expert_dispatch_combine_gb300", "csrc", "ffn_tc.cu")
FFN_GEMV_SRC = os.path.join(ROOT, "expert_dispatch_combine_gb300", "csrc", "ffn_gemv.cu")


TRAFFIC_PROFILES = {  # kernel -> (committed ncu summary, source file it was taken on)
    "tc": ("gemm_tc_gate_up_prof_e32.md", FFN_TC_SRC),
    "tc_f16": ("gemm_tc_gate_up_f16_prof_e32.md", FFN_TC_SRC),
    "gemv": ("gemv_gate_up_prof_decode_e32.md", FFN_GEMV_SRC),
}


def measured_traffic(alg_bytes: int, kind: str = "tc"):
    """DRAM bytes per launch of the gate/up kernel (tensor-core GEMM on the int8
    weights or on their fp16 copies, or the matrix-vector kernel of the decode
    path) for a launch of `alg_bytes` algorithmic bytes: the traffic /
    algorithmic ratio the committed ncu summary measured on its small workload
    (prof_e32, prof_decode_e32), times alg_bytes; None unless that summary was
    taken with the current kernel source.  The kernel's traffic grows with the
    units it serves (weights per touched expert, rows, h), so the ratio
    carries over."""
    name, src_file = TRAFFIC_PROFILES[kind]
    try:
        txt = open(os.path.join(ROOT, "profiles", name)).read()
        src = hashlib.sha1(open(src_file, "rb").read()).hexdigest()
    except OSError:
        return None
    keys = ("source_sha1:", "traffic_bytes_per_launch:", "algorithmic_bytes_per_launch:")
    kv = dict(l.split(":", 1) for l in txt.splitlines() if l.startswith(keys))
    if kv.get("source_sha1", "").strip() != src:
        return None
    try:
        ratio = int(kv["traffic_bytes_per_launch"]) / int(kv["algorithmic_bytes_per_launch"])
    except (KeyError, ValueError, ZeroDivisionError):
        return None
    return int(round(ratio * alg_bytes))


# ------------------------------------------------------------- bookkeeping
def algorithmic(w: synth.Workload) -> dict:
    """Algorithmic bytes / ops per step of each stage (INT8 messages, msg = H+16)."""
    T, H, k, I, E = w.T, w.H, w.k, w.I, w.E_phys
    route = T * w.E_log * 4 + T * k * 4 * 3 + E * 4
    dispatch = T * 2 * H + T * k * (H + 16) + T * k * 4 * 2      # read x, write msgs + rows
    combine = T * k * (H + 4) + T * k * 4 + T * 2 * H            # read msgs + w, write out
    ffn_ops = T * k * 6 * H * I                                   # 2 flops x 3 H*I MACs
    gate_up_ops = T * k * 4 * H * I                               # gate|up GEMM alone
    return dict(route_bytes=route, dispatch_bytes=dispatch, combine_bytes=combine, ffn_ops=ffn_ops,
                gate_up_ops=gate_up_ops, down_ops=ffn_ops - gate_up_ops)


def message_bytes(w: synth.Workload, bf16: bool) -> tuple[int, int]:
    """Algorithmic bytes of FusedDispatch and FusedCombine alone with bf16
    (unquantised) or INT8 + scale messages."""
    T, H, k = w.T, w.H, w.k
    row = 2 * H if bf16 else H
    dispatch = T * 2 * H + T * k * (row + 16) + T * k * 4 * 2
    combine = T * k * row + (0 if bf16 else T * k * 4) + T * k * 4 + T * 2 * H
    return dispatch, combine


def replica_aggregate(ms: float, units: int, world: int, device=None) -> tuple[float, float]:
    """Whole-job figure of N independent replicas (one per rank, no
    data-path collective): the slowest rank's time per step (max over ranks)
    and the units all ranks processed per second.  The reduction runs in the
    process group's backend on `device` (a CUDA device with NCCL, the CPU
    with gloo)."""
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return ms, world * units / (ms / 1000.0)


class ClockSampler:
    """nvidia-smi clocks/throttle sampling during the timed region."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.path = tempfile.mktemp(suffix=".csv")
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(index), "--query-gpu=" + self.FIELDS, "--format=csv,noheader",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self, t0: float, t1: float) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        self.proc.wait()
        sm, smax, reasons, n_all = [], None, set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            n_all += 1
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                continue
            if not (t0 - 0.1 <= ts <= t1 + 0.1):
                continue
            try:
                sm.append(float(parts[2].split()[0]))
                smax = float(parts[3].split()[0])
            except ValueError:
                continue
            for n, v in zip(names, parts[6:10]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ oracle
WEIGHT_FORMS = {
    "f16copy": "int8 W8A8, plus exact fp16 copies read by the tensor-core GEMMs of large batches",
    "int8": "int8 W8A8 only (tensor-core GEMMs convert int8 tiles on the SM)",
}


def config_of(w: synth.Workload, world: int, weight_bytes: int | None = None,
              weights: str = "f16copy") -> dict:
    """The `config` object of both arms' JSON lines (same keys, same values)."""
    wb = weight_bytes if weight_bytes is not None else 3 * w.E_log * w.H * w.I
    form = (" (the tensor-core GEMMs read their fp16 copies, twice the bytes, for experts above "
            "8 rows in batches above the decode size)" if weights == "f16copy" else "")
    inputs = (f"{wb / 1e9:.3f} GB of int8 weights of the touched experts{form} streamed every step "
              f"and {2 * w.T * w.H / 1e6:.1f} MB of bf16 hidden rows")
    l2 = ("inputs larger than L2 (129 MB): " if wb + 2 * w.T * w.H > L2_BYTES else
          "inputs fit in L2 (129 MB), not flushed between steps: ") + inputs
    return {"workload": w.name, "T": w.T, "H": w.H, "E_log": w.E_log, "E_phys": w.E_phys, "k": w.k,
            "I": w.I, "ranks": w.R, "src_ranks": w.S, "messages": "int8 dispatch, int8 combine",
            "weights": WEIGHT_FORMS[weights], "l2": l2, "parallelism": f"replicas x{world}"}


_ORC_CACHE = {}


def _oracle_inputs(w: synth.Workload, n: int):
    """The first n tokens of the workload (n a multiple of n_src_ranks) and the
    expert weights they route to."""
    import oracle

    key = (w.name, n)
    if key not in _ORC_CACHE:
        _ORC_CACHE.clear()
        lg = np.ascontiguousarray(synth.logits(w)[:n])
        x = np.random.default_rng([w.seed, 3]).standard_normal((w.T, w.H), dtype=np.float32)[:n]
        xb = synth.f32_to_bf16_bits(np.ascontiguousarray(x))
        rep = nc = p2l = None
        if w.eplb:
            _, _, _, cnt = oracle.route(synth.logits(w), w.k)
            from oracle import eplb
            rep, nc, p2l = eplb.plan(cnt[None, :].astype(np.float64), w.E_phys, w.placement_ranks)
        _, _, pidx, _ = oracle.route(lg, w.k, w.E_phys, rep, nc)
        need = set(int(p2l[p]) if p2l is not None else int(p) for p in np.unique(pidx))
        weights = {e: synth.expert_weights_np(w, e) for e in need}
        _ORC_CACHE[key] = (lg, xb, weights, rep, nc, p2l)
    return _ORC_CACHE[key]


def oracle_run(w: synth.Workload, n: int) -> dict:
    """One pass of the oracle's four stages over the first n tokens, with the
    workload's source ranks (n_src_ranks = S): tokens/s and ms per stage."""
    import oracle

    lg, xb, weights, rep, nc, p2l = _oracle_inputs(w, n)
    ms = {}
    t0 = time.perf_counter()
    _, wt, pidx, _ = oracle.route(lg, w.k, w.E_phys, rep, nc)
    t1 = time.perf_counter()
    xq, xs = oracle.quantize_bf16(xb)
    oracle.dispatch(xb, pidx, w.E_phys, w.R, w.S, fmt=1)
    t2 = time.perf_counter()
    cb, cs = oracle.ffn_all(xq, xs, pidx, weights, w.I, 1, p2l)
    t3 = time.perf_counter()
    oracle.combine(cb, cs, wt, 1)
    t4 = time.perf_counter()
    ms = {"route": 1e3 * (t1 - t0), "quantise_dispatch": 1e3 * (t2 - t1), "ffn": 1e3 * (t3 - t2),
          "combine": 1e3 * (t4 - t3)}
    return {"value": n / (t4 - t0), "tokens": n, "seconds": t4 - t0, "threads": oracle.num_threads(),
            "stages_ms": ms}


def oracle_tokens(w: synth.Workload, target_s: float) -> int:
    """Tokens (a multiple of n_src_ranks) for one oracle pass of about target_s."""
    n = w.S * max(1, 16 // w.S)
    r = oracle_run(w, n)
    n2 = int(target_s * n / max(r["seconds"], 1e-9)) // w.S * w.S
    return int(min(w.T, max(n, n2)))


def cpu_baseline(w: synth.Workload, target_s: float) -> dict:
    """The oracle on the host: the workload sampled on all OpenMP threads,
    plus one thread on the tiny layer and on a slice of the decode batch."""
    import oracle

    threads = oracle.num_threads()
    n = oracle_tokens(w, target_s)
    r = oracle_run(w, n)
    single = {}
    oracle.set_num_threads(1)
    try:
        for name, tokens in (("c0_tiny", None), ("c1_decode", 32)):
            ws = synth.WORKLOADS[name]
            nt = ws.T if tokens is None else tokens
            o = oracle_run(ws, nt)
            single[name] = {"value": o["value"], "unit": UNIT, "tokens": nt, "of": ws.T,
                            "stages_ms": o["stages_ms"]}
    finally:
        oracle.set_num_threads(threads)
    return {"value": r["value"], "unit": UNIT, "cores": r["threads"], "threads": r["threads"],
            "host_cores": os.cpu_count(), "kind": "oracle",
            "sample": (f"first {n} of {w.T} tokens ({w.S} source ranks) through the oracle's route, "
                       f"quantise + dispatch, expert FFN and combine ({r['seconds']:.1f} s)"),
            "stages_ms": r["stages_ms"], "single_thread": single}


def run_reference(args, rank: int, world: int):
    if rank != 0:
        return
    import oracle

    w = synth.WORKLOADS[args.workload]
    # the experts the whole batch touches (the GPU arm's `config` counts the same)
    rep = nc = p2l = None
    if w.eplb:
        _, _, _, cnt0 = oracle.route(synth.logits(w), w.k)
        from oracle import eplb
        rep, nc, p2l = eplb.plan(cnt0[None, :].astype(np.float64), w.E_phys, w.placement_ranks)
    _, _, _, cnt = oracle.route(synth.logits(w), w.k, w.E_phys, rep, nc)
    touched = np.nonzero(cnt)[0]
    if p2l is not None:
        touched = np.unique(p2l[touched])
    n = oracle_tokens(w, args.ref_sample_s)
    times, stages = [], {}
    for i in range(args.warmup + args.steps):
        r = oracle_run(w, n)
        if i >= args.warmup:
            times.append(r["seconds"])
            for k_, v in r["stages_ms"].items():
                stages[k_] = stages.get(k_, 0.0) + v / args.steps
    total = sum(times)
    value = args.steps * n / total
    sample = f"first {n} of {w.T} tokens per step ({w.S} source ranks) through the whole oracle layer"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 0,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int8 (exact int64 accumulation), f32 epilogue", "data": "synthetic",
        "config": config_of(w, world, len(touched) * 3 * w.H * w.I, args.weights),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(),
                         "threads": oracle.num_threads(), "host_cores": os.cpu_count(),
                         "kind": "oracle", "sample": sample, "stages_ms": stages},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


# ------------------------------------------------------------------- ours
def run_ours(args, rank: int, world: int):
    import torch
    import torch.distributed as dist

    from expert_dispatch_combine_gb300 import binding as B
    from expert_dispatch_combine_gb300.build import build
    from expert_dispatch_combine_gb300.layer import LayerBuffers, MoELayer

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build()
    B.load()
    w = synth.WORKLOADS[args.workload]
    shape = B.Shape(w.T, w.H, w.E_log, w.E_phys, w.k, w.I, w.R, w.S, B.MOE_MSG_INT8, B.MOE_MSG_INT8)
    w_gu, s_gu, w_d, s_d = synth.all_weights_torch(w, dev)
    rep = nc = p2l = None
    if w.eplb:
        # Collect step: per-expert loads of the unreplicated routing (moe_route),
        # then the host planner (moe_eplb_plan) builds the replica map.
        s0 = B.Shape(w.T, w.H, w.E_log, w.E_log, w.k, w.I, w.placement_ranks, w.S)
        lg0 = torch.from_numpy(synth.logits(w)).to(dev)
        ti = torch.empty((w.T, w.k), dtype=torch.int32, device=dev)
        tw = torch.empty((w.T, w.k), dtype=torch.float32, device=dev)
        tp = torch.empty((w.T, w.k), dtype=torch.int32, device=dev)
        cnt = torch.empty(w.E_log, dtype=torch.int32, device=dev)
        B.moe_route(s0, lg0, ti, tw, tp, cnt)
        r_, n_, p_ = B.moe_eplb_plan(cnt.cpu().numpy().astype(np.float64), w.E_phys, w.placement_ranks)
        rep, nc, p2l = (torch.from_numpy(a).to(dev) for a in (r_, n_, p_))
    layer = MoELayer(shape, w_gu, s_gu, w_d, s_d, rep_table=rep, n_copies=nc, phys_to_weight=p2l,
                     device=dev, f16_weights=args.weights == "f16copy")
    lg_h = synth.logits(w)
    x_h = synth.hidden_bits(w)
    logits = torch.from_numpy(lg_h).to(dev)
    x = torch.from_numpy(x_h.view(np.int16)).to(dev).view(torch.bfloat16)
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(args.warmup):
        layer.forward(logits, x)
    torch.cuda.synchronize()

    # ---- timed region: K steps through moe_layer
    sampler = ClockSampler(local)
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    n0 = B.moe_launch_count()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    ev0.record(stream)
    for _ in range(args.steps):
        layer.forward(logits, x)
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier()
    wall1 = time.time()
    launches = B.moe_launch_count() - n0
    clocks = sampler.stop(wall0, wall1)
    ms = ev0.elapsed_time(ev1) / args.steps
    ms_all, value = replica_aggregate(ms, w.T, world, dev)

    # ---- per-stage timing: the four steps inside moe_layer (the library's
    # events around them; on the tensor-core path its dispatch also writes the
    # FFN's input rows), and the four entry points called one by one (same
    # stream, CUDA events between the calls)
    b = layer.buf
    r = b.routing
    names = ["route", "dispatch", "ffn", "combine"]
    acc = {n: 0.0 for n in names}
    sep = {n: 0.0 for n in names}
    kern = {"gemm_gate_up": 0.0, "gemm_down": 0.0, "narrow_gate_up": 0.0, "narrow_down": 0.0}
    reps = max(1, min(args.steps, 5))
    B.moe_profile_enable(True)
    stage_sampler = ClockSampler(local)
    time.sleep(0.3)
    swall0 = time.time()
    for _ in range(reps):
        # keep the GPU busy for about 2 ms so that the host has enqueued all
        # the calls before the first event: the stage times then hold device
        # time only, not the host's launch latency of a call on an idle GPU
        torch.cuda._sleep(4_000_000)
        layer.forward(logits, x)
        torch.cuda.synchronize()
        prof = B.moe_profile_read(8)
        kern["gemm_gate_up"] += prof[0] / reps
        kern["gemm_down"] += prof[1] / reps
        kern["narrow_gate_up"] += max(prof[2], 0.0) / reps
        kern["narrow_down"] += max(prof[3], 0.0) / reps
        for i, n in enumerate(names):
            acc[n] += prof[4 + i] / reps
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
        torch.cuda._sleep(4_000_000)
        evs[0].record(stream)
        B.moe_route(shape, logits, r["topk_idx"], r["topk_w"], r["phys_idx"], r["expert_counts"],
                    rep, nc)
        evs[1].record(stream)
        B.moe_dispatch(shape, x, r["phys_idx"], b.dispatch, r["rank_counts"], r["expert_offsets"],
                       r["expert_rows"], b.workspace)
        evs[2].record(stream)
        B.moe_expert_ffn(shape, b.dispatch, r["expert_offsets"], r["expert_rows"], w_gu, s_gu, w_d,
                         s_d, b.combine, b.workspace, phys_to_weight=p2l, w_f16=layer.w_f16)
        evs[3].record(stream)
        B.moe_combine(shape, b.combine, r["topk_w"], b.out)
        evs[4].record(stream)
        torch.cuda.synchronize()
        for i, n in enumerate(names):
            sep[n] += evs[i].elapsed_time(evs[i + 1]) / reps
    stage_clocks = stage_sampler.stop(swall0, time.time())
    B.moe_profile_enable(False)
    fused_ms = None
    if B.moe_expert_ffn_path(shape) == B.MOE_FFN_TENSOR_CORE:
        # the expert FFN with the combine folded in (each token's combine waits
        # for its k return messages inside one persistent kernel), same inputs
        fused_out = torch.empty_like(b.out)
        fused_ms = 0.0
        for _ in range(reps):
            fa, fb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda._sleep(4_000_000)
            fa.record(stream)
            B.moe_expert_ffn_combine(shape, b.dispatch, r["expert_offsets"], r["expert_rows"], w_gu,
                                     s_gu, w_d, s_d, r["topk_w"], b.combine, fused_out, b.workspace,
                                     phys_to_weight=p2l, w_f16=layer.w_f16)
            fb.record(stream)
            torch.cuda.synchronize()
            fused_ms += fa.elapsed_time(fb) / reps
        assert B.moe_device_status(b.workspace) == 0
        del fused_out
    tramp_us = None
    if w.S < w.R:
        # trampoline forward (A2E + A2E'): same outputs as moe_dispatch, two hops
        tbuf = torch.empty(B.moe_trampoline_bytes(shape), dtype=torch.uint8, device=dev)
        t_ms = 0.0
        for _ in range(reps):
            ta, tb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda._sleep(4_000_000)
            ta.record(stream)
            B.moe_dispatch_trampoline(shape, x, r["phys_idx"], tbuf, b.dispatch, r["rank_counts"],
                                      r["expert_offsets"], r["expert_rows"], b.workspace)
            tb.record(stream)
            torch.cuda.synchronize()
            t_ms += ta.elapsed_time(tb) / reps
        tramp_us = 1000 * t_ms
        del tbuf
    # the whole layer as one launch: moe_layer captured once in a CUDA graph on
    # the same inputs and buffers, replayed back to back like the timed loop
    cap = torch.cuda.Stream(device=dev)
    graph = B.moe_layer_graph_create(shape, logits, x, *layer.w, r, b.dispatch, b.combine, b.workspace,
                                     b.out, cap, rep_table=rep, n_copies=nc, phys_to_weight=p2l,
                                     w_f16=layer.w_f16)
    try:
        for _ in range(2):
            B.moe_graph_launch(graph, stream)
        torch.cuda.synchronize()
        ga, gb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(4_000_000)
        ga.record(stream)
        for _ in range(args.steps):
            B.moe_graph_launch(graph, stream)
        gb.record(stream)
        torch.cuda.synchronize()
        graph_ms = ga.elapsed_time(gb) / args.steps
    finally:
        B.moe_graph_destroy(graph)
    assert B.moe_device_status(b.workspace) == 0
    alg = algorithmic(w)
    cnt_h = layer.buf.routing["expert_counts"].cpu().numpy()
    p2l_h = p2l.cpu().numpy() if p2l is not None else None

    def weight_sets(mask):
        idx = np.nonzero(mask)[0]
        return np.unique(p2l_h[idx]) if p2l_h is not None else idx

    touched = weight_sets(cnt_h > 0)
    ffn_path = B.moe_expert_ffn_path(shape)
    narrow = B.moe_expert_ffn_narrow_rows(shape)
    # the kernel measured as the dominant one: the tensor-core gate|up GEMM over
    # the experts with more than `narrow` rows (the narrow ones run on the
    # matrix-vector kernels), or the matrix-vector kernel of the decode path;
    # its bytes: int8 gate/up rows of the weight sets it touches, the expert
    # rows it reads (fp16 codes for the tensor cores, int8 dispatch rows for
    # the matrix-vector kernel) and the f32 h it writes
    wide = cnt_h > narrow if ffn_path != B.MOE_FFN_GEMV else cnt_h > 0
    rows_k = int(cnt_h[wide].sum())
    act_bytes = 1 if ffn_path == B.MOE_FFN_GEMV else 2
    # the fp16 weight copies serve batches above the decode size (more than 32
    # routed rows per physical expert on average)
    f16_used = (layer.w_f16 is not None and ffn_path == B.MOE_FFN_TENSOR_CORE
                and w.T * w.k > 32 * w.E_phys)
    w_bytes = 2 if f16_used else 1
    tkind = "gemv" if ffn_path == B.MOE_FFN_GEMV else "tc_f16" if f16_used else "tc"
    alg["gate_up_ops"] = rows_k * 4 * w.H * w.I
    # weights, expert rows (fp16 codes) in, g and u (f32, 2I per row) out
    alg["gate_up_bytes"] = (len(weight_sets(wide)) * 2 * w.I * w.H * w_bytes + rows_k * w.H * act_bytes
                            + rows_k * 2 * w.I * 4)
    peaks, peak_kind = _peaks()
    hbm = peaks["hbm_gbs"]
    # inside moe_layer on the tensor-core path the dispatch also writes each
    # message's fp16 expert input row and its scale (M * (2H + 4) bytes), which
    # the FFN then does not assemble
    staged = ffn_path == B.MOE_FFN_TENSOR_CORE
    staged_bytes = w.T * w.k * (2 * w.H + 4) if staged else 0
    stages = {
        "as_run_in": "moe_layer (library events around its four steps)",
        "route_us": 1000 * acc["route"],
        "dispatch_us": 1000 * acc["dispatch"],
        "ffn_us": 1000 * acc["ffn"],
        "combine_us": 1000 * acc["combine"],
        "dispatch_stages_ffn_rows": staged,
        "dispatch_gbs": (alg["dispatch_bytes"] + staged_bytes) / (acc["dispatch"] / 1000) / 1e9,
        "combine_gbs": alg["combine_bytes"] / (acc["combine"] / 1000) / 1e9,
        "separate_calls": {
            "route_us": 1000 * sep["route"], "dispatch_us": 1000 * sep["dispatch"],
            "ffn_us": 1000 * sep["ffn"], "combine_us": 1000 * sep["combine"],
            "dispatch_gbs": alg["dispatch_bytes"] / (sep["dispatch"] / 1000) / 1e9,
            "note": "moe_route, moe_dispatch, moe_expert_ffn (with its assembly step), moe_combine"},
    }
    if tramp_us is not None:
        stages["dispatch_trampoline_us"] = tramp_us
    # one launch (the captured layer) against the timed loop's moe_layer calls
    stages["graph_replay"] = {"ms_per_layer": graph_ms, "moe_layer_ms": ms,
                              "note": "moe_layer captured in a CUDA graph (moe_layer_graph_create), "
                                      "replayed back to back on the timed loop's inputs"}
    if fused_ms is not None:
        # against separate_calls' ffn_us + combine_us (both assemble the input rows)
        stages["ffn_combine_fused_us"] = 1000 * fused_ms
    if narrow > 0 and ffn_path == B.MOE_FFN_TENSOR_CORE:
        nmask = (cnt_h > 0) & (cnt_h <= narrow)
        nsets = len(weight_sets(nmask))
        nrows = int(cnt_h[nmask].sum())
        n_us = 1000 * (kern["narrow_gate_up"] + kern["narrow_down"])
        n_bytes = nsets * 3 * w.H * w.I + nrows * (w.H + 4 * w.I + 2 * w.I + 4 * w.H)
        stages["narrow_experts"] = {
            "max_rows": narrow, "experts": int(nmask.sum()), "rows": nrows,
            "gate_up_us": 1000 * kern["narrow_gate_up"], "down_us": 1000 * kern["narrow_down"],
            "gbs": n_bytes / (n_us / 1e6) / 1e9 if n_us > 0 else None,
            "kernels": "gemv_kernel<gate|up>, gemv_kernel<down> (int8 dp4a weight streaming)"}
    # FusedDispatch + FusedCombine as message movement (the separate entry
    # points: the dispatch writes the messages only)
    dc_bytes = alg["dispatch_bytes"] + alg["combine_bytes"]
    dc_s = (sep["dispatch"] + sep["combine"]) / 1000
    stages["dispatch_combine_hbm_frac"] = dc_bytes / dc_s / 1e9 / hbm
    ffn_tflops = alg["ffn_ops"] / (acc["ffn"] / 1000) / 1e12
    stages["ffn_tflops"] = ffn_tflops
    # the tensor peak that applies: the burst figure while the SM clock held its
    # maximum with no power cap during the stage timing (the kernels are timed in
    # short runs), else the sustained figure under the power cap; both fractions
    # are reported
    burst, sustained = peaks["bf16_tflops"], peaks["bf16_tflops_sustained"]
    at_max = (stage_clocks.get("sm_mhz") is not None and stage_clocks.get("sm_max_mhz")
              and stage_clocks["sm_mhz"] >= 0.97 * stage_clocks["sm_max_mhz"])
    capped = "sw_power_cap" in stage_clocks.get("reasons", [])
    use_burst = bool(at_max) and not capped
    peak_tc = burst if use_burst else sustained
    peak_tc_name = ("burst (SM clock at its maximum, no power cap during the stage timing)" if use_burst
                    else "sustained (SM clock below its maximum or power-capped during the stage timing)")
    stages["ffn_frac_burst"] = ffn_tflops / burst
    stages["ffn_frac_sustained"] = ffn_tflops / sustained
    stages["clocks"] = stage_clocks
    gu_name = ("gemv_kernel<gate|up> (int8 dp4a weight streaming)" if ffn_path == B.MOE_FFN_GEMV
               else "gemm_tc_kernel<gate|up> (exact int8 on tcgen05 kind::f16, "
                    + ("both operands from shared memory, fp16 weight copies" if f16_used
                       else "int8 weights converted into tensor memory")
                    + f"; experts with more than {narrow} routed rows)")
    if kern["gemm_gate_up"] > 0:
        # dominant kernel: the gate|up expert GEMM, timed by CUDA events on its stream
        gu_tflops = alg["gate_up_ops"] / (kern["gemm_gate_up"] / 1000) / 1e12
        stages["gemm_gate_up_us"] = 1000 * kern["gemm_gate_up"]
        stages["gemm_down_us"] = 1000 * kern["gemm_down"]
        rows_dn = int(cnt_h[wide].sum())
        stages["gemm_down_tflops"] = rows_dn * 2 * w.H * w.I / (kern["gemm_down"] / 1000) / 1e12
        # bound by the kernel's arithmetic intensity against the measured ridge point
        intensity = alg["gate_up_ops"] / alg["gate_up_bytes"]
        ridge = peak_tc * 1e12 / (hbm * 1e9)
        if intensity >= ridge:
            roofline = {"bound": "tensor", "achieved": gu_tflops, "peak": peak_tc, "unit": "TFLOP/s",
                        "frac": gu_tflops / peak_tc,
                        "traffic": measured_traffic(alg["gate_up_bytes"], tkind),
                        "traffic_source": "scaled from the small-workload ncu capture (profiles/)",
                        "kernel": gu_name,
                        "algorithmic_ops_per_launch": alg["gate_up_ops"],
                        "algorithmic_bytes_per_launch": alg["gate_up_bytes"],
                        "frac_burst": gu_tflops / burst, "frac_sustained": gu_tflops / sustained,
                        "peak_source": (f"{peak_kind} bf16 {peak_tc_name}; exact int8 runs on the "
                                        "fp16 tensor path")}
        else:  # decode-sized batches stream the weights: HBM-bound
            gu_gbs = alg["gate_up_bytes"] / (kern["gemm_gate_up"] / 1000) / 1e9
            roofline = {"bound": "hbm", "achieved": gu_gbs, "peak": hbm, "unit": "GB/s",
                        "frac": gu_gbs / hbm,
                        "traffic": measured_traffic(alg["gate_up_bytes"], tkind),
                        "traffic_source": "scaled from the small-workload ncu capture (profiles/)",
                        "kernel": gu_name,
                        "algorithmic_ops_per_launch": alg["gate_up_ops"],
                        "algorithmic_bytes_per_launch": alg["gate_up_bytes"],
                        "peak_source": f"{peak_kind} HBM copy bandwidth"}
    else:  # CUDA-core expert path (shapes the tensor-core kernel does not take)
        roofline = {"bound": "alu", "achieved": ffn_tflops, "peak": None, "unit": "TFLOP/s",
                    "frac": None, "traffic": None, "kernel": "moe_expert_ffn (dp4a path)"}

    # ---- end to end through the C ABI with host buffers (moe_layer_host): every
    # step copies its inputs in from page-locked host memory, runs the layer and
    # copies the output back, all enqueued by the library.  A serving loop
    # alternates two streams and two buffer sets, so one step's copies overlap
    # the other step's kernels.
    h_lg = torch.from_numpy(lg_h).pin_memory()
    h_x = torch.from_numpy(x_h.view(np.int16)).pin_memory()
    h_out = [torch.empty((w.T, w.H), dtype=torch.int16).pin_memory() for _ in range(2)]
    layers = [layer, MoELayer(shape, w_gu, s_gu, w_d, s_d, rep_table=rep, n_copies=nc,
                              phys_to_weight=p2l, device=dev)]
    layers[1].w_f16 = layer.w_f16  # one set of fp16 copies serves both buffer sets
    streams = [torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)]
    for i in range(2):  # warm-up of both sets
        layers[i].forward_host(h_lg, h_x, h_out[i], stream=streams[i])
    torch.cuda.synchronize()
    barrier()
    e_steps = max(2, args.steps)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for st_ in streams:
        st_.wait_event(e0)
    for i in range(e_steps):
        layers[i % 2].forward_host(h_lg, h_x, h_out[i % 2], stream=streams[i % 2])
    for st_ in streams:
        done = torch.cuda.Event()
        done.record(st_)
        stream.wait_event(done)
    e1.record(stream)
    torch.cuda.synchronize()
    # the host copies hold the layer's output (same inputs every step)
    ref_bits = layer.buf.out.view(torch.int16).cpu()
    e2e_checked = bool(torch.equal(h_out[0], ref_bits) and torch.equal(h_out[1], ref_bits))
    del layers[1]
    e_ms, e_value = replica_aggregate(e0.elapsed_time(e1) / e_steps, w.T, world, dev)
    e2e = {"value": e_value, "unit": UNIT,
           "h2d_bytes_per_step": lg_h.nbytes + x_h.nbytes, "d2h_bytes_per_step": w.T * w.H * 2,
           "steps": e_steps, "api": "moe_layer_host (C ABI, host buffers)",
           "output_checked": e2e_checked,
           "pipelining": "two streams and two buffer sets: one step's copies overlap the "
                         "other step's kernels"}
    formats = None
    if w.msg_formats:
        # FusedDispatch and FusedCombine alone, with bf16 (unquantised) and with
        # INT8 + scale messages, on this step's routing
        formats = {}
        for fname, fmt in (("int8", B.MOE_MSG_INT8), ("bf16", B.MOE_MSG_BF16)):
            fs = B.Shape(w.T, w.H, w.E_log, w.E_phys, w.k, w.I, w.R, w.S, fmt, fmt)
            fb = b if fmt == B.MOE_MSG_INT8 else LayerBuffers(fs, dev)
            if fmt == B.MOE_MSG_BF16:
                # return messages: any bf16 values (the combine's time does not depend on them)
                fb.combine_rows().view(torch.bfloat16).copy_(
                    torch.randn((w.T, w.k, w.H), device=dev).to(torch.bfloat16))
            d_ms = c_ms = 0.0
            for _ in range(reps):
                e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
                torch.cuda._sleep(4_000_000)
                e[0].record(stream)
                B.moe_dispatch(fs, x, r["phys_idx"], fb.dispatch, fb.routing["rank_counts"],
                               fb.routing["expert_offsets"], fb.routing["expert_rows"], fb.workspace)
                e[1].record(stream)
                B.moe_combine(fs, fb.combine, r["topk_w"], fb.out)
                e[2].record(stream)
                torch.cuda.synchronize()
                d_ms += e[0].elapsed_time(e[1]) / reps
                c_ms += e[1].elapsed_time(e[2]) / reps
            db, cb = message_bytes(w, fmt == B.MOE_MSG_BF16)
            hbm_gbs = _peaks()[0]["hbm_gbs"]
            formats[fname] = {"dispatch_us": 1000 * d_ms, "combine_us": 1000 * c_ms,
                              "dispatch_gbs": db / (d_ms / 1000) / 1e9,
                              "combine_gbs": cb / (c_ms / 1000) / 1e9,
                              "dispatch_combine_hbm_frac": (db + cb) / ((d_ms + c_ms) / 1000) / 1e9 / hbm_gbs}
            if fb is not b:
                del fb
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    if formats is not None:
        stages["standalone_messages"] = formats

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, target_s=args.ref_sample_s)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_all, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "int8 (exact int32 accumulation), f32 epilogue",
            "data": "synthetic",
            "config": config_of(w, world, len(touched) * 3 * w.H * w.I, args.weights),
            "stages": stages,
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches,
            "clocks": clocks,
            "routed_rows_per_s": value * w.k,
        }
        print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=list(synth.WORKLOADS))
    ap.add_argument("--ref-sample-s", type=float, default=8.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--weights", default="f16copy", choices=list(WEIGHT_FORMS),
                    help="f16copy: also keep exact fp16 copies of the int8 weights for the "
                         "tensor-core GEMMs of large batches; int8: the int8 weights alone")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    try:
        run_ours(args, rank, world)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
