"""CPU oracle for the decode-time MoE layer -- TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline leg import
this package.  The product (the CUDA library and its Python binding) never
loads, links or calls anything here, and nothing here loads the product.

The arithmetic lives in ``moe_oracle.c`` (plain C, one rounding per binary32
operation, binary64 where no integer depends on the result) and in
``eplb.py`` (the replica planner, plain Python).  This module compiles the C
file with gcc on first use and exposes numpy-friendly wrappers.

Parity status per function (what pins it; the tests under ``tests/`` hold
the pins):
  route          brute-force k-subset search; closed-form weight cases
  quantize       hand-worked vectors (tests/golden/quant_vectors.txt)
  exp_spec/silu  math.exp within 2 ulp; exact special values
  dispatch       naive re-derivation on tiny inputs + invariants
  expert_row     int32 accumulators vs numpy int64 matmul; one-hot weights;
                 the binary32 scale steps g, u, y by a hand-worked row with
                 distinct power-of-two scales (tests/golden/expert_scale_steps.txt)
                 and a float64 closed form on random distinct scales
  combine        identity experts reproduce the dequantised input
  buffer formula the page's worked example (225 MiB + 420 MiB)
  eplb           the page's [4, 256] rotation example; replica counts differ
                 by at most one; hand-checked greedy cases
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB_PATH = os.path.join(_BUILD, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into a shared library (gcc, OpenMP, no FP contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def load_library(path: str):
    """Load a compiled copy of moe_oracle.c and declare its functions (the
    tests also load copies with planted mistakes through this)."""
    lib = ctypes.CDLL(path)
    _declare(lib)
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        _lib = load_library(build())
        return _lib


def _declare(lib):
    P = ctypes.c_void_p
    i32, i64, f32, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_double
    lib.orc_exp_spec.argtypes = [f32]
    lib.orc_exp_spec.restype = f32
    lib.orc_silu.argtypes = [f32]
    lib.orc_silu.restype = f32
    lib.orc_round_f64_to_bf16.argtypes = [f64]
    lib.orc_round_f64_to_bf16.restype = ctypes.c_uint16
    lib.orc_round_f32_to_bf16.argtypes = [f32]
    lib.orc_round_f32_to_bf16.restype = ctypes.c_uint16
    lib.orc_quantize_row_f32.argtypes = [i32, P, P, P]
    lib.orc_quantize_row_f32.restype = None
    lib.orc_quantize_rows_bf16.argtypes = [i32, i32, P, P, P]
    lib.orc_quantize_rows_bf16.restype = None
    lib.orc_route.argtypes = [i32, i32, i32, i32, P, P, P, i32, P, P, P, P]
    lib.orc_route.restype = i32
    lib.orc_static_buffer_bytes.argtypes = [i64, i64, i64, i64, i64]
    lib.orc_static_buffer_bytes.restype = i64
    lib.orc_dispatch.argtypes = [i32] * 7 + [P] * 11
    lib.orc_dispatch.restype = i32
    lib.orc_expert_row.argtypes = [i32, i32, P, f32, P, P, P, P, i32, P, P,
                                   P, P, P, P, P]
    lib.orc_expert_row.restype = i32
    lib.orc_ffn_all.argtypes = [i32, i32, i32, i32, P, P, P, P, P, P, P, P,
                                i32, P, P]
    lib.orc_ffn_all.restype = i32
    lib.orc_combine.argtypes = [i32, i32, i32, i32, P, P, P, P]
    lib.orc_combine.restype = i32
    lib.orc_num_threads.argtypes = []
    lib.orc_num_threads.restype = i32
    lib.orc_set_num_threads.argtypes = [i32]
    lib.orc_set_num_threads.restype = None


def _p(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return _load().orc_num_threads()


def set_num_threads(n: int) -> None:
    """Threads of the oracle's parallel loops (results do not depend on it)."""
    _load().orc_set_num_threads(int(n))


# ------------------------------------------------------------------ scalars
def exp_spec(x: float) -> np.float32:
    return np.float32(_load().orc_exp_spec(float(np.float32(x))))


def silu(g: float) -> np.float32:
    return np.float32(_load().orc_silu(float(np.float32(g))))


def f64_to_bf16_bits(v: float) -> int:
    return int(_load().orc_round_f64_to_bf16(float(v)))


def f32_to_bf16_bits(v: float) -> int:
    return int(_load().orc_round_f32_to_bf16(float(np.float32(v))))


# ------------------------------------------------------------ quantisation
def quantize_f32(v) -> tuple[np.ndarray, np.float32]:
    v = np.ascontiguousarray(v, dtype=np.float32)
    q = np.empty(v.shape[-1], np.int8)
    s = np.zeros(1, np.float32)
    _load().orc_quantize_row_f32(v.shape[-1], _p(v), _p(q), _p(s))
    return q, s[0]


def quantize_bf16(x_bits: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """x_bits: uint16 [rows, H] bf16 bit patterns -> (int8 codes, f32 scales)."""
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    rows, H = x_bits.shape
    q = np.empty((rows, H), np.int8)
    s = np.empty(rows, np.float32)
    _load().orc_quantize_rows_bf16(rows, H, _p(x_bits), _p(q), _p(s))
    return q, s


# ------------------------------------------------------------------ route
def route(logits: np.ndarray, k: int, E_phys: int | None = None,
          rep_table: np.ndarray | None = None, n_copies: np.ndarray | None = None):
    """Returns (topk_idx i32[T,k], topk_w f32[T,k], phys_idx i32[T,k], counts i32[E_phys])."""
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = logits.shape
    E_phys = E if E_phys is None else E_phys
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float32)
    pidx = np.empty((T, k), np.int32)
    cnt = np.empty(E_phys, np.int32)
    maxc = 0
    if rep_table is not None:
        rep_table = np.ascontiguousarray(rep_table, dtype=np.int32)
        n_copies = np.ascontiguousarray(n_copies, dtype=np.int32)
        maxc = rep_table.shape[1]
    rc = _load().orc_route(T, E, E_phys, k, _p(logits), _p(rep_table), _p(n_copies),
                           maxc, _p(idx), _p(w), _p(pidx), _p(cnt))
    if rc:
        raise ValueError("oracle route: bad arguments")
    return idx, w, pidx, cnt


def static_buffer_bytes(rank_num, local_batch, topk, experts_per_rank, msg_size) -> int:
    return int(_load().orc_static_buffer_bytes(rank_num, local_batch, topk,
                                               experts_per_rank, msg_size))


# --------------------------------------------------------------- dispatch
def dispatch(x_bits: np.ndarray, phys_idx: np.ndarray, E_phys: int, R: int, S: int,
             fmt: int = 1, with_rows: bool = True) -> dict:
    """FusedDispatch layout and messages.  fmt 1 = INT8 codes, 0 = bf16 rows.
    with_rows=False skips the message rows (layout and metadata only)."""
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    phys_idx = np.ascontiguousarray(phys_idx, dtype=np.int32)
    T, H = x_bits.shape
    k = phys_idx.shape[1]
    lb, epr = T // S, E_phys // R
    mt = lb * min(k, epr)
    nslots = R * S * mt
    rowb = H if fmt == 1 else 2 * H
    rows = np.zeros((nslots, rowb), np.uint8) if with_rows else None
    ms = np.zeros(nslots, np.float32)
    msrc = np.full(nslots, -1, np.int32)
    mbs = np.full(nslots, -1, np.int32)
    mrs = np.full(nslots, -1, np.int32)
    rc_ = np.empty((R, S), np.int32)
    off = np.empty(E_phys + 1, np.int32)
    er = np.empty(T * k, np.int32)
    slot_of = np.empty((T, k), np.int32)
    rc = _load().orc_dispatch(T, H, E_phys, k, R, S, fmt, _p(x_bits), _p(phys_idx),
                              _p(rows), _p(ms), _p(msrc), _p(mbs), _p(mrs), _p(rc_),
                              _p(off), _p(er), _p(slot_of))
    if rc:
        raise ValueError("oracle dispatch: bad arguments or slot overflow")
    return dict(rows=rows, meta_scale=ms, meta_src=msrc, meta_bs=mbs, meta_rs=mrs,
                rank_counts=rc_, expert_offsets=off, expert_rows=er, slot_of=slot_of,
                mt=mt, lb=lb, epr=epr)


# ------------------------------------------------------------- expert FFN
def expert_row(xq: np.ndarray, xs: float, w_gu: np.ndarray, s_gu: np.ndarray,
               w_d: np.ndarray, s_d: np.ndarray, cfmt: int = 1, debug: bool = False, lib=None):
    """One routed row through one expert.  Returns (message, scale[, debug dict]).
    `lib` (optional) is another compiled copy of the oracle (load_library)."""
    H = xq.shape[0]
    I = w_d.shape[1]
    xq = np.ascontiguousarray(xq, dtype=np.int8)
    w_gu = np.ascontiguousarray(w_gu, dtype=np.int8)
    w_d = np.ascontiguousarray(w_d, dtype=np.int8)
    s_gu = np.ascontiguousarray(s_gu, dtype=np.float32)
    s_d = np.ascontiguousarray(s_d, dtype=np.float32)
    msg = np.empty(H, np.int8 if cfmt == 1 else np.uint16)
    sc = np.zeros(1, np.float32)
    dbg = None
    if debug:
        dbg = dict(acc_gu=np.empty(2 * I, np.int32), hq=np.empty(I, np.int8),
                   sh=np.zeros(1, np.float32), acc_d=np.empty(H, np.int32),
                   y=np.empty(H, np.float32))
    g = (lambda n: _p(dbg[n]) if dbg else None)
    (lib or _load()).orc_expert_row(H, I, _p(xq), float(xs), _p(w_gu), _p(s_gu), _p(w_d),
                           _p(s_d), cfmt, _p(msg), _p(sc), g("acc_gu"), g("hq"),
                           g("sh"), g("acc_d"), g("y"))
    if debug:
        dbg["sh"] = dbg["sh"][0]
        return msg, sc[0], dbg
    return msg, sc[0]


def ffn_all(xq: np.ndarray, xs: np.ndarray, phys_idx: np.ndarray, weights: dict,
            I: int, cfmt: int = 1, phys_to_logical: np.ndarray | None = None):
    """All (t, j) rows.  weights: {logical e: (w_gu, s_gu, w_d, s_d)} -- only
    the experts actually routed to need to be present.  Returns
    (cbuf [T,k,H] int8 or uint16 bf16 bits, cscale f32 [T,k])."""
    xq = np.ascontiguousarray(xq, dtype=np.int8)
    xs = np.ascontiguousarray(xs, dtype=np.float32)
    phys_idx = np.ascontiguousarray(phys_idx, dtype=np.int32)
    T, H = xq.shape
    k = phys_idx.shape[1]
    nlog = max(weights) + 1 if weights else 0
    if phys_to_logical is not None:
        phys_to_logical = np.ascontiguousarray(phys_to_logical, dtype=np.int32)
        nlog = max(nlog, int(phys_to_logical.max()) + 1)
    nlog = max(nlog, int(phys_idx.max()) + 1)
    PP = ctypes.c_void_p * nlog
    tabs = [PP(), PP(), PP(), PP()]
    keep = []
    for e, ws in weights.items():
        for n in range(4):
            a = np.ascontiguousarray(ws[n])
            keep.append(a)
            tabs[n][e] = a.ctypes.data
    cb = np.empty((T, k, H), np.int8 if cfmt == 1 else np.uint16)
    cs = np.zeros((T, k), np.float32)
    rc = _load().orc_ffn_all(T, H, I, k, _p(xq), _p(xs), _p(phys_idx),
                             _p(phys_to_logical), ctypes.cast(tabs[0], ctypes.c_void_p),
                             ctypes.cast(tabs[1], ctypes.c_void_p),
                             ctypes.cast(tabs[2], ctypes.c_void_p),
                             ctypes.cast(tabs[3], ctypes.c_void_p), cfmt, _p(cb), _p(cs))
    del keep
    if rc:
        raise ValueError("oracle ffn_all: weights missing for a routed expert")
    return cb, cs


# ---------------------------------------------------------------- combine
def combine(cbuf: np.ndarray, cscale: np.ndarray, topk_w: np.ndarray, cfmt: int = 1) -> np.ndarray:
    """Returns bf16 bit patterns uint16 [T, H]."""
    cbuf = np.ascontiguousarray(cbuf)
    cscale = np.ascontiguousarray(cscale, dtype=np.float32)
    topk_w = np.ascontiguousarray(topk_w, dtype=np.float32)
    T, k, H = cbuf.shape
    out = np.empty((T, H), np.uint16)
    _load().orc_combine(T, H, k, cfmt, _p(cbuf), _p(cscale), _p(topk_w), _p(out))
    return out


# ------------------------------------------------------------ whole layer
def layer(logits, x_bits, weights, E_phys, R, S, k, I, cfmt=1, rep_table=None,
          n_copies=None, phys_to_logical=None) -> dict:
    """Route -> quantise -> dispatch layout -> experts -> combine, all on CPU."""
    idx, w, pidx, cnt = route(logits, k, E_phys, rep_table, n_copies)
    xq, xs = quantize_bf16(x_bits)
    d = dispatch(x_bits, pidx, E_phys, R, S, fmt=1)
    cb, cs = ffn_all(xq, xs, pidx, weights, I, cfmt, phys_to_logical)
    out = combine(cb, cs, w, cfmt)
    return dict(topk_idx=idx, topk_w=w, phys_idx=pidx, counts=cnt, xq=xq, xs=xs,
                dispatch=d, cbuf=cb, cscale=cs, out=out)
