"""Thin Python binding of the C ABI in include/moe.h (ctypes; argument marshalling only).

Every function here has the name of the C entry point it calls and takes
torch tensors (device memory owned by the caller) or numpy arrays for the
host-only entry points.  All arithmetic runs in the CUDA library; if the
library is missing this module raises on first use -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libmoe_gb300.so")

MOE_MSG_BF16, MOE_MSG_INT8 = 0, 1
STATUS = {0: "ok", 1: "invalid argument", 2: "buffer or workspace too small",
          3: "static buffer capacity exceeded", 4: "CUDA launch error",
          5: "device wait timed out", 6: "unsupported configuration",
          7: "device-side index check failed"}
MOE_OK, MOE_ERR_CAPACITY, MOE_ERR_TIMEOUT, MOE_ERR_INDEX = 0, 3, 5, 7


class MoeError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn}: {STATUS.get(code, code)} (status {code})")
        self.code = code


class moe_shape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("T", "H", "E_log", "E_phys", "k", "I", "n_ranks", "n_src_ranks",
                 "dispatch_fmt", "combine_fmt")]


class moe_layout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in
                ("max_tokens", "dispatch_row_bytes", "dispatch_meta_offset", "dispatch_bytes",
                 "combine_row_bytes", "combine_scale_offset", "combine_bytes", "workspace_bytes")]


class moe_expert_weights(ctypes.Structure):
    _fields_ = [("w_gate_up", ctypes.c_void_p), ("s_gate_up", ctypes.c_void_p),
                ("w_down", ctypes.c_void_p), ("s_down", ctypes.c_void_p),
                ("n_sets", ctypes.c_int32), ("phys_to_weight", ctypes.c_void_p),
                ("w_gate_up_f16", ctypes.c_void_p), ("w_down_f16", ctypes.c_void_p)]


class moe_routing(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("topk_idx", "topk_w", "phys_idx", "expert_counts", "rank_counts",
                 "expert_offsets", "expert_rows")]


EXPORTED = ("moe_status_string", "moe_static_buffer_bytes", "moe_query_layout", "moe_eplb_plan",
            "moe_route", "moe_dispatch", "moe_expert_ffn", "moe_combine", "moe_layer",
            "moe_gemm_workspace_bytes", "moe_grouped_gemm_s8", "moe_launch_count",
            "moe_device_status", "moe_last_cuda_error", "moe_profile_enable", "moe_profile_read",
            "moe_dispatch_noalloc", "moe_dispatch_noalloc_max_scratch", "moe_layer_graph_create",
            "moe_graph_launch", "moe_graph_destroy", "moe_eplb_collect", "moe_expert_ffn_combine",
            "moe_trampoline_bytes", "moe_dispatch_trampoline", "moe_expert_ffn_path",
            "moe_layer_host", "moe_expert_ffn_combine_ex", "moe_expert_ffn_narrow_rows",
            "moe_weights_to_f16")

_lib = None


def load(path: str = LIB_PATH):
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libmoe_gb300.so not built ({path}); run "
                           "`python -m expert_dispatch_combine_gb300.build`")
    lib = ctypes.CDLL(path)
    P, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    PS = ctypes.POINTER(moe_shape)
    sig = {
        "moe_status_string": ([ctypes.c_int], ctypes.c_char_p),
        "moe_static_buffer_bytes": ([i64, i64, i64, i64, i64, ctypes.POINTER(i64)], ctypes.c_int),
        "moe_query_layout": ([PS, ctypes.POINTER(moe_layout)], ctypes.c_int),
        "moe_expert_ffn_path": ([PS, ctypes.POINTER(i32)], ctypes.c_int),
        "moe_expert_ffn_narrow_rows": ([PS, ctypes.POINTER(i32)], ctypes.c_int),
        "moe_eplb_plan": ([i32, i32, i32, i32, P, i32, P, P, P], ctypes.c_int),
        "moe_route": ([PS, P, P, P, i32, P, P, P, P, P], ctypes.c_int),
        "moe_dispatch": ([PS, P, P, P, i64, P, P, P, P, i64, P], ctypes.c_int),
        "moe_expert_ffn": ([PS, P, i64, P, P, ctypes.POINTER(moe_expert_weights), P, i64, P, i64, P],
                           ctypes.c_int),
        "moe_combine": ([PS, P, i64, P, P, P], ctypes.c_int),
        "moe_layer": ([PS, P, P, P, P, i32, ctypes.POINTER(moe_expert_weights),
                       ctypes.POINTER(moe_routing), P, i64, P, i64, P, i64, P, P], ctypes.c_int),
        "moe_layer_host": ([PS, P, P, P, P, P, P, P, i32, ctypes.POINTER(moe_expert_weights),
                            ctypes.POINTER(moe_routing), P, i64, P, i64, P, i64, P, P], ctypes.c_int),
        "moe_gemm_workspace_bytes": ([i32, i64, i32], i64),
        "moe_device_status": ([P, ctypes.POINTER(i32), P], ctypes.c_int),
        "moe_launch_count": ([], i64),
        "moe_last_cuda_error": ([], ctypes.c_char_p),
        "moe_profile_enable": ([i32], ctypes.c_int),
        "moe_dispatch_noalloc": ([PS, P, P, P, i64, P, P, P, P], ctypes.c_int),
        "moe_dispatch_noalloc_max_scratch": ([], i64),
        "moe_profile_read": ([P, i32], ctypes.c_int),
        "moe_grouped_gemm_s8": ([i32, P, i64, P, P, i64, P, i32, i32, P, P, i64, P], ctypes.c_int),
        "moe_layer_graph_create": ([PS, P, P, P, P, i32, ctypes.POINTER(moe_expert_weights),
                                    ctypes.POINTER(moe_routing), P, i64, P, i64, P, i64, P, P,
                                    ctypes.POINTER(P)], ctypes.c_int),
        "moe_graph_launch": ([P, P], ctypes.c_int),
        "moe_graph_destroy": ([P], ctypes.c_int),
        "moe_eplb_collect": ([i32, i32, P, P, P, P], ctypes.c_int),
        "moe_trampoline_bytes": ([PS, ctypes.POINTER(i64)], ctypes.c_int),
        "moe_dispatch_trampoline": ([PS, P, P, P, i64, P, i64, P, P, P, P, i64, P], ctypes.c_int),
        "moe_expert_ffn_combine": ([PS, P, i64, P, P, ctypes.POINTER(moe_expert_weights), P, P, i64,
                                    P, P, i64, P], ctypes.c_int),
        "moe_expert_ffn_combine_ex": ([PS, P, i64, P, P, ctypes.POINTER(moe_expert_weights), P, P, i64,
                                       P, P, i64, i32, i64, P], ctypes.c_int),
        "moe_weights_to_f16": ([P, i64, P, P], ctypes.c_int),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    _lib = lib
    return lib


# ----------------------------------------------------------------- helpers
def _ptr(t):
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    assert t.is_contiguous(), "tensors passed to the library must be contiguous"
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def _check(fn, rc):
    if rc != 0:
        if rc == 4:  # MOE_ERR_CUDA: attach the CUDA error text
            raise MoeError(fn + " [" + load().moe_last_cuda_error().decode() + "]", rc)
        raise MoeError(fn, rc)


@dataclass(frozen=True)
class Shape:
    T: int
    H: int
    E_log: int
    E_phys: int
    k: int
    I: int
    n_ranks: int
    n_src_ranks: int
    dispatch_fmt: int = MOE_MSG_INT8
    combine_fmt: int = MOE_MSG_INT8

    def c(self) -> moe_shape:
        return moe_shape(self.T, self.H, self.E_log, self.E_phys, self.k, self.I, self.n_ranks,
                         self.n_src_ranks, self.dispatch_fmt, self.combine_fmt)


def moe_status_string(code: int) -> str:
    return load().moe_status_string(code).decode()


def moe_static_buffer_bytes(rank_num, local_batch, topk, experts_per_rank, msg_size) -> int:
    out = ctypes.c_int64(0)
    _check("moe_static_buffer_bytes",
           load().moe_static_buffer_bytes(rank_num, local_batch, topk, experts_per_rank, msg_size,
                                          ctypes.byref(out)))
    return out.value


def moe_query_layout(shape: Shape) -> dict:
    L = moe_layout()
    cs = shape.c()
    _check("moe_query_layout", load().moe_query_layout(ctypes.byref(cs), ctypes.byref(L)))
    return {n: getattr(L, n) for n, _ in moe_layout._fields_}


MOE_FFN_CUDA_CORE, MOE_FFN_TENSOR_CORE, MOE_FFN_GEMV = 0, 1, 2


def moe_expert_ffn_path(shape: Shape) -> int:
    """Which kernels run the expert FFN of moe_expert_ffn / moe_layer for
    `shape`: MOE_FFN_CUDA_CORE, MOE_FFN_TENSOR_CORE or MOE_FFN_GEMV."""
    out = ctypes.c_int32(0)
    cs = shape.c()
    _check("moe_expert_ffn_path", load().moe_expert_ffn_path(ctypes.byref(cs), ctypes.byref(out)))
    return out.value


def moe_expert_ffn_narrow_rows(shape: Shape) -> int:
    """Experts with 1..n routed rows run on the matrix-vector kernels beside
    the tensor-core GEMMs (0: none)."""
    out = ctypes.c_int32(0)
    cs = shape.c()
    _check("moe_expert_ffn_narrow_rows", load().moe_expert_ffn_narrow_rows(ctypes.byref(cs), ctypes.byref(out)))
    return out.value


def moe_eplb_plan(token_count: np.ndarray, E_phys: int, n_ranks: int, max_copies: int | None = None,
                  trim: bool = True):
    """Host planner.  token_count [n_slices, E_log] (or [E_log]).
    Returns (rep_table [E_log, max_copies], n_copies [E_log], phys_to_logical [E_phys]);
    with trim the table keeps only the columns the plan uses."""
    tc = np.ascontiguousarray(np.atleast_2d(token_count), dtype=np.float64)
    ns, E = tc.shape
    mc = max_copies or (E_phys - E + 1)
    rep = np.empty((E, mc), np.int32)
    nc = np.empty(E, np.int32)
    p2l = np.empty(E_phys, np.int32)
    _check("moe_eplb_plan", load().moe_eplb_plan(ns, E, E_phys, n_ranks, tc.ctypes.data, mc,
                                                 rep.ctypes.data, nc.ctypes.data, p2l.ctypes.data))
    if not trim:
        return rep, nc, p2l
    used = max(1, int(nc.max()))
    return np.ascontiguousarray(rep[:, :used]), nc, p2l


def moe_eplb_collect(expert_counts, logical_load, phys_to_logical=None, stream=None) -> None:
    """logical_load[e] += expert_counts summed over the physical copies of logical
    expert e (device int32 [E_phys] counts, device int64 [E_log] loads)."""
    _check("moe_eplb_collect", load().moe_eplb_collect(
        int(logical_load.numel()), int(expert_counts.numel()), _ptr(expert_counts),
        _ptr(phys_to_logical), _ptr(logical_load), _stream(stream)))


def moe_route(shape: Shape, logits, topk_idx, topk_w, phys_idx, expert_counts,
              rep_table=None, n_copies=None, stream=None):
    cs = shape.c()
    mc = int(rep_table.shape[1]) if rep_table is not None else 0
    _check("moe_route", load().moe_route(ctypes.byref(cs), _ptr(logits), _ptr(rep_table),
                                         _ptr(n_copies), mc, _ptr(topk_idx), _ptr(topk_w),
                                         _ptr(phys_idx), _ptr(expert_counts), _stream(stream)))


def moe_dispatch(shape: Shape, x, phys_idx, dispatch_buf, rank_counts, expert_offsets,
                 expert_rows, workspace, stream=None):
    cs = shape.c()
    _check("moe_dispatch", load().moe_dispatch(
        ctypes.byref(cs), _ptr(x), _ptr(phys_idx), _ptr(dispatch_buf), dispatch_buf.numel(),
        _ptr(rank_counts), _ptr(expert_offsets), _ptr(expert_rows), _ptr(workspace),
        workspace.numel(), _stream(stream)))


def moe_dispatch_noalloc(shape: Shape, x, phys_idx, dispatch_buf, rank_counts, expert_offsets,
                         expert_rows, stream=None):
    """moe_dispatch for callers that cannot allocate a workspace (the scratch is a
    fixed device array inside the library; see include/moe.h)."""
    cs = shape.c()
    _check("moe_dispatch_noalloc", load().moe_dispatch_noalloc(
        ctypes.byref(cs), _ptr(x), _ptr(phys_idx), _ptr(dispatch_buf), dispatch_buf.numel(),
        _ptr(rank_counts), _ptr(expert_offsets), _ptr(expert_rows), _stream(stream)))


def moe_dispatch_noalloc_max_scratch() -> int:
    return int(load().moe_dispatch_noalloc_max_scratch())


def _weights(w_gate_up, s_gate_up, w_down, s_down, phys_to_weight=None,
             w_f16=None) -> moe_expert_weights:
    """w_f16: None or the pair (w_gate_up_f16, w_down_f16) made by moe_weights_to_f16."""
    g16, d16 = w_f16 if w_f16 is not None else (None, None)
    return moe_expert_weights(_ptr(w_gate_up), _ptr(s_gate_up), _ptr(w_down), _ptr(s_down),
                              int(w_gate_up.shape[0]), _ptr(phys_to_weight), _ptr(g16), _ptr(d16))


def moe_weights_to_f16(src, dst=None, stream=None):
    """fp16 copy (exact) of an int8 device tensor, same shape; returns dst."""
    import torch
    if dst is None:
        dst = torch.empty(src.shape, dtype=torch.float16, device=src.device)
    if dst.numel() != src.numel():
        raise ValueError("moe_weights_to_f16: dst and src differ in size")
    _check("moe_weights_to_f16", load().moe_weights_to_f16(_ptr(src), src.numel(), _ptr(dst),
                                                           _stream(stream)))
    return dst


def moe_expert_ffn(shape: Shape, dispatch_buf, expert_offsets, expert_rows, w_gate_up, s_gate_up,
                   w_down, s_down, combine_buf, workspace, phys_to_weight=None, stream=None, w_f16=None):
    cs = shape.c()
    w = _weights(w_gate_up, s_gate_up, w_down, s_down, phys_to_weight, w_f16)
    _check("moe_expert_ffn", load().moe_expert_ffn(
        ctypes.byref(cs), _ptr(dispatch_buf), dispatch_buf.numel(), _ptr(expert_offsets),
        _ptr(expert_rows), ctypes.byref(w), _ptr(combine_buf), combine_buf.numel(),
        _ptr(workspace), workspace.numel(), _stream(stream)))


def moe_trampoline_bytes(shape: Shape) -> int:
    v = ctypes.c_int64(0)
    _check("moe_trampoline_bytes", load().moe_trampoline_bytes(ctypes.byref(shape.c()), ctypes.byref(v)))
    return v.value


def moe_dispatch_trampoline(shape: Shape, x, phys_idx, trampoline_buf, dispatch_buf, rank_counts,
                            expert_offsets, expert_rows, workspace, stream=None):
    cs = shape.c()
    _check("moe_dispatch_trampoline", load().moe_dispatch_trampoline(
        ctypes.byref(cs), _ptr(x), _ptr(phys_idx), _ptr(trampoline_buf), trampoline_buf.numel(),
        _ptr(dispatch_buf), dispatch_buf.numel(), _ptr(rank_counts), _ptr(expert_offsets),
        _ptr(expert_rows), _ptr(workspace), workspace.numel(), _stream(stream)))


def moe_expert_ffn_combine(shape: Shape, dispatch_buf, expert_offsets, expert_rows, w_gate_up,
                           s_gate_up, w_down, s_down, topk_w, combine_buf, out, workspace,
                           phys_to_weight=None, stream=None, w_f16=None):
    cs = shape.c()
    w = _weights(w_gate_up, s_gate_up, w_down, s_down, phys_to_weight, w_f16)
    _check("moe_expert_ffn_combine", load().moe_expert_ffn_combine(
        ctypes.byref(cs), _ptr(dispatch_buf), dispatch_buf.numel(), _ptr(expert_offsets),
        _ptr(expert_rows), ctypes.byref(w), _ptr(topk_w), _ptr(combine_buf), combine_buf.numel(),
        _ptr(out), _ptr(workspace), workspace.numel(), _stream(stream)))


def moe_expert_ffn_combine_ex(shape: Shape, dispatch_buf, expert_offsets, expert_rows, w_gate_up,
                              s_gate_up, w_down, s_down, topk_w, combine_buf, out, workspace,
                              expected: int, wait_ns: int, phys_to_weight=None, stream=None, w_f16=None):
    """moe_expert_ffn_combine with the combine's wait target and bound given."""
    cs = shape.c()
    w = _weights(w_gate_up, s_gate_up, w_down, s_down, phys_to_weight, w_f16)
    _check("moe_expert_ffn_combine_ex", load().moe_expert_ffn_combine_ex(
        ctypes.byref(cs), _ptr(dispatch_buf), dispatch_buf.numel(), _ptr(expert_offsets),
        _ptr(expert_rows), ctypes.byref(w), _ptr(topk_w), _ptr(combine_buf), combine_buf.numel(),
        _ptr(out), _ptr(workspace), workspace.numel(), int(expected), int(wait_ns), _stream(stream)))


def moe_combine(shape: Shape, combine_buf, topk_w, out, stream=None):
    cs = shape.c()
    _check("moe_combine", load().moe_combine(ctypes.byref(cs), _ptr(combine_buf),
                                             combine_buf.numel(), _ptr(topk_w), _ptr(out),
                                             _stream(stream)))


def moe_layer(shape: Shape, logits, x, w_gate_up, s_gate_up, w_down, s_down, routing: dict,
              dispatch_buf, combine_buf, workspace, out, rep_table=None, n_copies=None,
              phys_to_weight=None, stream=None, w_f16=None):
    cs = shape.c()
    w = _weights(w_gate_up, s_gate_up, w_down, s_down, phys_to_weight, w_f16)
    r = moe_routing(*[_ptr(routing[n]) for n, _ in moe_routing._fields_])
    mc = int(rep_table.shape[1]) if rep_table is not None else 0
    _check("moe_layer", load().moe_layer(
        ctypes.byref(cs), _ptr(logits), _ptr(x), _ptr(rep_table), _ptr(n_copies), mc,
        ctypes.byref(w), ctypes.byref(r), _ptr(dispatch_buf), dispatch_buf.numel(),
        _ptr(combine_buf), combine_buf.numel(), _ptr(workspace), workspace.numel(), _ptr(out),
        _stream(stream)))


def moe_layer_host(shape: Shape, h_logits, h_x, h_out, d_logits, d_x, w_gate_up, s_gate_up, w_down,
                   s_down, routing: dict, dispatch_buf, combine_buf, workspace, d_out, rep_table=None,
                   n_copies=None, phys_to_weight=None, stream=None, w_f16=None):
    """The whole layer from host tensors (page-locked CPU tensors: h_logits f32,
    h_x and h_out 16-bit) to host: the copies in, moe_layer and the copy out,
    all enqueued on `stream` by the library."""
    cs = shape.c()
    w = _weights(w_gate_up, s_gate_up, w_down, s_down, phys_to_weight, w_f16)
    r = moe_routing(*[_ptr(routing[n]) for n, _ in moe_routing._fields_])
    mc = int(rep_table.shape[1]) if rep_table is not None else 0
    _check("moe_layer_host", load().moe_layer_host(
        ctypes.byref(cs), _ptr(h_logits), _ptr(h_x), _ptr(h_out), _ptr(d_logits), _ptr(d_x),
        _ptr(rep_table), _ptr(n_copies), mc, ctypes.byref(w), ctypes.byref(r), _ptr(dispatch_buf),
        dispatch_buf.numel(), _ptr(combine_buf), combine_buf.numel(), _ptr(workspace),
        workspace.numel(), _ptr(d_out), _stream(stream)))


def moe_layer_graph_create(shape: Shape, logits, x, w_gate_up, s_gate_up, w_down, s_down,
                           routing: dict, dispatch_buf, combine_buf, workspace, out,
                           capture_stream, rep_table=None, n_copies=None, phys_to_weight=None,
                           w_f16=None) -> int:
    """Captures moe_layer with these arguments on capture_stream (a
    torch.cuda.Stream other than the legacy default stream); returns the
    graph handle for moe_graph_launch / moe_graph_destroy."""
    cs = shape.c()
    w = _weights(w_gate_up, s_gate_up, w_down, s_down, phys_to_weight, w_f16)
    r = moe_routing(*[_ptr(routing[n]) for n, _ in moe_routing._fields_])
    mc = int(rep_table.shape[1]) if rep_table is not None else 0
    h = ctypes.c_void_p(None)
    _check("moe_layer_graph_create", load().moe_layer_graph_create(
        ctypes.byref(cs), _ptr(logits), _ptr(x), _ptr(rep_table), _ptr(n_copies), mc,
        ctypes.byref(w), ctypes.byref(r), _ptr(dispatch_buf), dispatch_buf.numel(),
        _ptr(combine_buf), combine_buf.numel(), _ptr(workspace), workspace.numel(), _ptr(out),
        _stream(capture_stream), ctypes.byref(h)))
    return h.value


def moe_graph_launch(graph: int, stream=None) -> None:
    _check("moe_graph_launch", load().moe_graph_launch(graph, _stream(stream)))


def moe_graph_destroy(graph: int) -> None:
    _check("moe_graph_destroy", load().moe_graph_destroy(graph))


def moe_profile_enable(on: bool) -> None:
    _check("moe_profile_enable", load().moe_profile_enable(1 if on else 0))


def moe_profile_read(n: int = 2) -> tuple:
    """(gate/up GEMM ms, down GEMM ms, narrow-expert gate/up ms, narrow-expert
    down ms, then moe_layer's route, dispatch, FFN and combine ms), the first n
    of them, from the most recent calls; -1 for what did not run."""
    ms = (ctypes.c_float * n)()
    _check("moe_profile_read", load().moe_profile_read(ctypes.cast(ms, ctypes.c_void_p), n))
    return tuple(float(v) for v in ms)


def moe_launch_count() -> int:
    return int(load().moe_launch_count())


def moe_gemm_workspace_bytes(n_groups: int, max_rows: int, K: int) -> int:
    return int(load().moe_gemm_workspace_bytes(n_groups, max_rows, K))


def moe_device_status(workspace, stream=None) -> int:
    v = ctypes.c_int32(0)
    _check("moe_device_status", load().moe_device_status(_ptr(workspace), ctypes.byref(v),
                                                         _stream(stream)))
    return v.value


def moe_grouped_gemm_s8(offsets, max_rows: int, A, lda: int, B, C, workspace, row_index=None,
                        stream=None):
    """B: int8 [G, N, K]; C: int32 [M_total, N]."""
    G, N, K = (int(s) for s in B.shape)
    _check("moe_grouped_gemm_s8", load().moe_grouped_gemm_s8(
        G, _ptr(offsets), max_rows, _ptr(row_index), _ptr(A), lda, _ptr(B), N, K, _ptr(C),
        _ptr(workspace), workspace.numel(), _stream(stream)))
