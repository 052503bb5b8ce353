"""C-ABI checks that need no GPU: the library builds, loads and exports every
entry point include/moe.h declares; host-only entry points (buffer formula,
layout, EPLB planner) match the oracle; argument validation rejects bad
input before anything is enqueued."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from oracle import eplb
from expert_dispatch_combine_gb300 import binding as B
from expert_dispatch_combine_gb300 import synth
from expert_dispatch_combine_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="module")
def lib():
    build()
    return B.load()


def _declared():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


def test_header_symbols_exported(lib):
    names = _declared()
    assert len(names) >= 14
    raw = ctypes.CDLL(B.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), n
    assert set(B.EXPORTED) <= set(names)


def test_status_strings(lib):
    assert B.moe_status_string(0) == "ok"
    assert "invalid" in B.moe_status_string(1)
    assert "index" in B.moe_status_string(B.MOE_ERR_INDEX)
    for code, text in B.STATUS.items():
        assert B.moe_status_string(code) != "unknown status", code
    assert B.moe_status_string(99) == "unknown status"


def test_buffer_formula_matches_page_example(lib):
    for line in open(os.path.join(GOLDEN, "buffer_formula.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        a = [int(x) for x in line.split()]
        assert B.moe_static_buffer_bytes(*a[:5]) == a[5]
    with pytest.raises(B.MoeError):
        B.moe_static_buffer_bytes(0, 96, 8, 1, 7680)
    with pytest.raises(B.MoeError):
        B.moe_static_buffer_bytes(1 << 40, 1 << 20, 8, 8, 1 << 20)  # overflow


@pytest.mark.parametrize("name", list(synth.WORKLOADS))
def test_layout_matches_formula(lib, name):
    w = synth.WORKLOADS[name]
    s = B.Shape(w.T, w.H, w.E_log, w.E_phys, w.k, w.I, w.R, w.S)
    L = B.moe_query_layout(s)
    assert L["max_tokens"] == w.lb * min(w.k, w.epr)
    per_rank = B.moe_static_buffer_bytes(w.S, w.lb, w.k, w.epr, w.H + 16)
    assert L["dispatch_bytes"] >= w.R * per_rank
    assert L["dispatch_bytes"] - w.R * per_rank < 1024
    assert L["dispatch_meta_offset"] % 256 == 0
    assert L["combine_scale_offset"] >= w.T * w.k * w.H
    assert L["workspace_bytes"] > 0


def test_expert_ffn_path_choice(lib):
    """The FFN kernel family follows the shape: dp4a GEMMs off the 64 grid,
    matrix-vector products for decode batches (at most 4 routed rows per
    physical expert, INT8 return messages, H and I multiples of 512), the
    tensor-core GEMMs otherwise."""
    def path(**kw):
        base = dict(T=64, H=256, E_log=16, E_phys=16, k=2, I=128, n_ranks=4, n_src_ranks=4)
        base.update(kw)
        return B.moe_expert_ffn_path(B.Shape(**base))
    assert path(H=48) == B.MOE_FFN_CUDA_CORE
    assert path() == B.MOE_FFN_TENSOR_CORE                     # H = 256: not a multiple of 512
    dec = dict(T=96, H=7168, E_log=256, E_phys=256, k=8, I=2048, n_ranks=32, n_src_ranks=32)
    assert path(**dec) == B.MOE_FFN_GEMV                        # 768 rows over 256 experts
    assert path(**dict(dec, T=128)) == B.MOE_FFN_GEMV           # exactly 4 rows per expert
    assert path(**dict(dec, T=160)) == B.MOE_FFN_TENSOR_CORE    # 5 rows per expert
    assert path(**dict(dec, combine_fmt=B.MOE_MSG_BF16)) == B.MOE_FFN_TENSOR_CORE
    with pytest.raises(B.MoeError):
        path(T=0)


def test_smoke_reaches_the_tensor_core_gemms(lib):
    """smoke()'s fp16-copy layer is above the decode size, so moe_layer runs
    its expert FFN on the tensor-core GEMMs (on the copies: CTA pairs), with
    no expert left to the matrix-vector kernels (H, I not multiples of 512)."""
    import __graft_entry__ as g
    w = synth.custom("smoke_f16", **g.SMOKE_F16)
    shape = B.Shape(w.T, w.H, w.E_log, w.E_phys, w.k, w.I, w.R, w.S)
    assert w.T * w.k > 32 * w.E_phys
    assert B.moe_expert_ffn_path(shape) == B.MOE_FFN_TENSOR_CORE
    assert B.moe_expert_ffn_narrow_rows(shape) == 0


@pytest.mark.parametrize("bad", [
    dict(T=0), dict(H=24), dict(I=8), dict(k=0), dict(k=17), dict(E_phys=8),
    dict(n_ranks=3), dict(n_src_ranks=5), dict(dispatch_fmt=2),
])
def test_shape_validation(lib, bad):
    base = dict(T=64, H=256, E_log=16, E_phys=16, k=2, I=128, n_ranks=4, n_src_ranks=4)
    base.update(bad)
    with pytest.raises(B.MoeError) as e:
        B.moe_query_layout(B.Shape(**base))
    assert e.value.code == 1


def test_entry_points_reject_before_enqueue(lib):
    """Null pointers, misaligned buffers and short buffers are refused on the
    host (the fake device pointers below are never dereferenced)."""
    s = B.Shape(64, 256, 16, 16, 2, 128, 4, 4).c()
    L = B.moe_query_layout(B.Shape(64, 256, 16, 16, 2, 128, 4, 4))
    P = ctypes.c_void_p
    fake = 1 << 40  # 256-aligned, never touched
    rc = lib.moe_dispatch(ctypes.byref(s), P(fake), P(fake), P(fake), L["dispatch_bytes"] - 256,
                          P(fake), P(fake), P(fake), P(fake), L["workspace_bytes"], None)
    assert rc == 2  # dispatch buffer too small
    rc = lib.moe_dispatch(ctypes.byref(s), P(fake), P(fake), P(fake + 8), L["dispatch_bytes"],
                          P(fake), P(fake), P(fake), P(fake), L["workspace_bytes"], None)
    assert rc == 1  # misaligned
    rc = lib.moe_dispatch(ctypes.byref(s), None, P(fake), P(fake), L["dispatch_bytes"],
                          P(fake), P(fake), P(fake), P(fake), L["workspace_bytes"], None)
    assert rc == 1  # null input
    rc = lib.moe_combine(ctypes.byref(s), P(fake), L["combine_bytes"] - 1, P(fake), P(fake), None)
    assert rc == 2
    # replicas require a map
    s2 = B.Shape(64, 256, 16, 24, 2, 128, 4, 4).c()
    rc = lib.moe_route(ctypes.byref(s2), P(fake), None, None, 0, P(fake), P(fake), P(fake),
                       P(fake), None)
    assert rc == 1
    # grouped GEMM: K not a multiple of 16, short workspace
    rc = lib.moe_grouped_gemm_s8(2, P(fake), 10, None, P(fake), 40, P(fake), 32, 40, P(fake),
                                 P(fake), 1 << 20, None)
    assert rc == 1
    rc = lib.moe_grouped_gemm_s8(2, P(fake), 10, None, P(fake), 64, P(fake), 32, 64, P(fake),
                                 P(fake), 16, None)
    assert rc == 2
    # graph capture: the legacy default stream cannot be captured; no handle is returned
    h = ctypes.c_void_p(12345)
    rc = lib.moe_layer_graph_create(ctypes.byref(s), P(fake), P(fake), None, None, 0, None, None,
                                    P(fake), L["dispatch_bytes"], P(fake), L["combine_bytes"],
                                    P(fake), L["workspace_bytes"], P(fake), None, ctypes.byref(h))
    assert rc == 1 and not h.value
    assert lib.moe_graph_destroy(None) == 0


@pytest.mark.parametrize("E,R,E_phys,slices,seed", [
    (16, 4, 24, 1, 0), (16, 4, 24, 3, 1), (256, 32, 288, 1, 2), (32, 8, 48, 4, 3), (8, 2, 8, 1, 4),
])
def test_eplb_planner_matches_oracle(lib, E, R, E_phys, slices, seed):
    rng = np.random.default_rng(seed)
    load = (rng.zipf(1.3, size=(slices, E)) * rng.integers(1, 50, size=(slices, E))).astype(np.float64)
    rep, nc, p2l = B.moe_eplb_plan(load, E_phys, R)
    rep_o, nc_o, p2l_o = eplb.plan(load, E_phys, R)
    assert (nc == nc_o).all()
    assert (p2l == p2l_o).all()
    assert (rep == rep_o[:, :rep.shape[1]]).all()


def test_eplb_planner_on_workload_counts(lib):
    w = synth.WORKLOADS["c3_eplb"]
    _, _, _, cnt = oracle.route(synth.logits(w), w.k)
    rep, nc, p2l = B.moe_eplb_plan(cnt.astype(np.float64), w.E_phys, w.R)
    rep_o, nc_o, p2l_o = eplb.plan(cnt[None, :].astype(np.float64), w.E_phys, w.R)
    assert (p2l == p2l_o).all() and (nc == nc_o).all()
    assert nc.sum() == w.E_phys
    # the hottest expert got the most copies
    assert nc[np.argmax(cnt)] == nc.max() > 1


def test_weight_copies_rejected_before_enqueue(lib):
    """moe_weights_to_f16 and the optional fp16 weight fields: argument errors
    are returned on the host (fake device pointers, never dereferenced)."""
    P = ctypes.c_void_p
    fake = 1 << 40
    assert lib.moe_weights_to_f16(None, 16, P(fake), None) == 1            # null source
    assert lib.moe_weights_to_f16(P(fake), 16, None, None) == 1            # null destination
    assert lib.moe_weights_to_f16(P(fake), -1, P(fake), None) == 1         # negative count
    assert lib.moe_weights_to_f16(P(fake + 8), 16, P(fake), None) == 1     # misaligned
    assert lib.moe_weights_to_f16(None, 0, None, None) == 0                # nothing to copy
    shape = B.Shape(64, 256, 16, 16, 2, 128, 4, 4)
    s = shape.c()
    L = B.moe_query_layout(shape)

    def ffn(w):
        return lib.moe_expert_ffn(ctypes.byref(s), P(fake), L["dispatch_bytes"], P(fake), P(fake),
                                  ctypes.byref(w), P(fake), L["combine_bytes"], P(fake),
                                  L["workspace_bytes"], None)

    def weights(g16, d16):
        return B.moe_expert_weights(fake, fake, fake, fake, 16, None, g16, d16)

    assert ffn(weights(fake, None)) == 1        # gate/up copy without the down copy
    assert ffn(weights(None, fake)) == 1        # down copy without the gate/up copy
    assert ffn(weights(fake + 8, fake)) == 1    # misaligned copy
    assert ffn(weights(fake, fake + 2)) == 1
