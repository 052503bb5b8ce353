"""Device-side index checks: corrupt caller data never makes a kernel address
memory outside the caller's buffers; the kernels skip the access and post a
code to the workspace status word instead.

Every buffer the library writes carries canary bytes after its end
(CanaryBuffers), checked after each call.  Inputs are corrupted on the host
before they are copied to the device; each index path was checked against its
buffer bounds on paper before these tests first ran.
"""
import numpy as np
import pytest
import torch

import oracle
from expert_dispatch_combine_gb300 import binding as B
from expert_dispatch_combine_gb300 import synth
from expert_dispatch_combine_gb300.layer import MoELayer

from gpu_util import CanaryBuffers, bits_to_bf16_tensor, lib, make_layer, shape_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib()


def _np(t):
    return t.detach().cpu().numpy()


def _route_bufs(T, k, E_phys, dev="cuda"):
    return (torch.empty((T, k), dtype=torch.int32, device=dev),
            torch.empty((T, k), dtype=torch.float32, device=dev),
            torch.empty((T, k), dtype=torch.int32, device=dev),
            torch.full((E_phys,), -7, dtype=torch.int32, device=dev))


# ------------------------------------------------------------------- route
def test_route_nan_logits_read_as_minus_inf():
    T, E, k = 57, 40, 6
    rng = np.random.default_rng(3)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    lg[rng.random((T, E)) < 0.2] = np.nan
    lg[5, :] = np.nan          # a row with no finite logit: ids by expert order
    lg[6, : E - 2] = np.nan    # fewer finite logits than k
    ref_in = np.where(np.isnan(lg), -np.inf, lg).astype(np.float32)
    idx, _, _, cnt = oracle.route(ref_in, k)
    shape = B.Shape(T, 16, E, E, k, 16, 1, 1)
    g_idx, g_w, g_p, g_c = _route_bufs(T, k, E)
    B.moe_route(shape, torch.from_numpy(lg).cuda(), g_idx, g_w, g_p, g_c)
    torch.cuda.synchronize()
    assert (_np(g_idx) == idx).all()
    assert (_np(g_p) == idx).all()
    assert (_np(g_c) == cnt).all()
    assert _np(g_idx)[5].tolist() == list(range(k))


@pytest.mark.parametrize("T,E,k", [(333, 1024, 8), (1000, 300, 7), (31, 1024, 32)])
def test_route_counts_wide_expert_sets(T, E, k):
    """Atomic-free counts (per-warp histograms, one 8-block cluster) at up to
    the largest expert count the ABI allows and id counts that fill no round."""
    lg = np.random.default_rng(T + E).standard_normal((T, E)).astype(np.float32)
    idx, wt, _, cnt = oracle.route(lg, k)
    shape = B.Shape(T, 16, E, E, k, 16, 1, 1)
    g_idx, g_w, g_p, g_c = _route_bufs(T, k, E)
    B.moe_route(shape, torch.from_numpy(lg).cuda(), g_idx, g_w, g_p, g_c)
    torch.cuda.synchronize()
    assert (_np(g_idx) == idx).all()
    assert (_np(g_c) == cnt).all()
    assert np.abs(_np(g_w) - wt).max() <= 2e-6


def test_route_invalid_replica_entries_give_minus_one():
    T, E_log, E_phys, k = 64, 8, 12, 2
    lg = np.random.default_rng(1).standard_normal((T, E_log)).astype(np.float32)
    rep = np.full((E_log, 3), -1, np.int32)
    rep[:, 0] = np.arange(E_log)
    nc = np.ones(E_log, np.int32)
    rep[1, 1] = 8
    nc[1] = 2
    rep[2, 1] = 99          # outside [0, E_phys): every other token of expert 2
    nc[2] = 2
    nc[3] = 0               # copy count outside [1, max_copies]
    nc[4] = 7
    idx, _, _, _ = oracle.route(lg, k)
    shape = B.Shape(T, 16, E_log, E_phys, k, 16, 1, 1)
    g_idx, g_w, g_p, g_c = _route_bufs(T, k, E_phys)
    B.moe_route(shape, torch.from_numpy(lg).cuda(), g_idx, g_w, g_p, g_c,
                torch.from_numpy(rep).cuda(), torch.from_numpy(nc).cuda())
    torch.cuda.synchronize()
    p = _np(g_p)
    t = np.arange(T)[:, None].repeat(k, 1)
    exp = idx.copy()
    exp[(idx == 1) & (t % 2 == 1)] = 8
    exp[(idx == 2) & (t % 2 == 1)] = -1
    exp[(idx == 3) | (idx == 4)] = -1
    assert (_np(g_idx) == idx).all()
    assert (p == exp).all()
    assert (_np(g_c) == np.bincount(exp[exp >= 0], minlength=E_phys)).all()


# ---------------------------------------------------------------- dispatch
def test_dispatch_drops_out_of_range_ids():
    w = synth.custom("bad_ids", seed=2, T=48, H=128, E_log=16, k=3, I=64, R=4, S=4)
    shape = shape_of(w)
    _, _, pidx, _ = oracle.route(synth.logits(w), w.k)
    bad = pidx.copy()
    bad[3, 1] = -5
    bad[17, 0] = w.E_phys + 3
    bad[40, 2] = 1 << 30
    buf = CanaryBuffers(shape)
    r = buf.routing
    x = bits_to_bf16_tensor(synth.hidden_bits(w))
    B.moe_dispatch(shape, x, torch.from_numpy(bad).cuda(), buf.dispatch, r["rank_counts"],
                   r["expert_offsets"], r["expert_rows"], buf.workspace)
    assert B.moe_device_status(buf.workspace) == B.MOE_ERR_INDEX
    buf.check()
    good = (bad >= 0) & (bad < w.E_phys)
    n = int(good.sum())
    assert int(_np(r["rank_counts"]).sum()) == n
    off = _np(r["expert_offsets"])
    assert off[-1] == n
    assert (np.diff(off) == np.bincount(bad[good], minlength=w.E_phys)).all()
    # the remaining messages sit where the oracle puts them when the bad routes are absent:
    # every listed slot holds one of them, each exactly once
    rows = _np(r["expert_rows"])[:n]
    meta = _np(buf.dispatch_meta())
    seen = set()
    for g in rows:
        t = meta[g, 1] * w.lb + meta[g, 2]
        j = meta[g, 3]
        assert good[t, j] and (t, j) not in seen
        seen.add((t, j))
    assert len(seen) == n


def test_dispatch_capacity_overflow_is_reported():
    """A replica table that maps four logical experts onto one physical slot
    (so a token sends four messages to a rank whose static area holds two per
    token) drops the extra messages and reports MOE_ERR_CAPACITY; every row
    list entry still names a written slot, and the whole layer stays inside
    its buffers."""
    T, H, E, k, I, R = 32, 128, 8, 4, 64, 4   # epr = 2 < k: max_tokens = 2 lb
    w = synth.custom("overflow", seed=4, T=T, H=H, E_log=E, k=k, I=I, R=R, S=4)
    shape = shape_of(w)
    lg = synth.logits(w)
    lg[:, :4] += 20.0                          # every token picks experts 0..3
    rep = np.arange(E, dtype=np.int32)[:, None].copy()
    rep[:4, 0] = 0                             # ... all mapped onto physical slot 0
    nc = np.ones(E, np.int32)
    w_gu, s_gu, w_d, s_d = synth.all_weights_torch(w, "cuda")
    layer = MoELayer(shape, w_gu, s_gu, w_d, s_d, rep_table=torch.from_numpy(rep).cuda(),
                     n_copies=torch.from_numpy(nc).cuda(), buffers=CanaryBuffers(shape))
    layer.forward(torch.from_numpy(lg).cuda(), bits_to_bf16_tensor(synth.hidden_bits(w)))
    b = layer.buf
    assert B.moe_device_status(b.workspace) == B.MOE_ERR_CAPACITY
    b.check()
    rc = _np(b.routing["rank_counts"])
    mt = b.layout["max_tokens"]
    assert rc.max() <= mt and (rc[0] == mt).all()
    rows = _np(b.routing["expert_rows"])
    meta = _np(b.dispatch_meta())
    assert ((rows >= 0) & (rows < R * 4 * mt)).all()
    assert (meta[rows, 1] < 4).all() and (meta[rows, 3] < k).all()


# -------------------------------------------------------------- expert FFN
FFN_CASES = {
    "tensor_core": dict(T=64, H=128, E_log=16, k=2, I=64, R=4, S=4),
    "gemv": dict(T=16, H=512, E_log=16, k=2, I=512, R=4, S=2),
    "cuda_core": dict(T=16, H=48, E_log=8, k=2, I=32, R=2, S=2),
}


def _ffn_after_valid_layer(name, corrupt):
    w = synth.custom("ffn_" + name, seed=9, **FFN_CASES[name])
    layer = make_layer(w)
    layer.forward(torch.from_numpy(synth.logits(w)).cuda(), bits_to_bf16_tensor(synth.hidden_bits(w)))
    b, r, s = layer.buf, layer.buf.routing, layer.shape
    assert B.moe_device_status(b.workspace) == 0
    offs, rows = r["expert_offsets"].clone(), r["expert_rows"].clone()
    corrupt(offs, rows)
    w_gu, s_gu, w_d, s_d = layer.w
    B.moe_expert_ffn(s, b.dispatch, offs, rows, w_gu, s_gu, w_d, s_d, b.combine, b.workspace)
    return b


@pytest.mark.parametrize("name", sorted(FFN_CASES))
def test_ffn_bad_row_list_entry(name):
    def corrupt(offs, rows):
        rows[1] = 1 << 30
        rows[-1] = -3
    b = _ffn_after_valid_layer(name, corrupt)
    assert B.moe_device_status(b.workspace) == B.MOE_ERR_INDEX
    b.check()


@pytest.mark.parametrize("name", sorted(FFN_CASES))
def test_ffn_bad_offsets(name):
    def corrupt(offs, rows):
        offs[3] = offs[5] + 7      # not a nondecreasing prefix
    b = _ffn_after_valid_layer(name, corrupt)
    assert B.moe_device_status(b.workspace) == B.MOE_ERR_INDEX
    b.check()


@pytest.mark.parametrize("name", sorted(FFN_CASES))
def test_ffn_offsets_beyond_rows(name):
    def corrupt(offs, rows):
        offs[-1] = offs[-1] + 1000  # more rows than the row list holds
    b = _ffn_after_valid_layer(name, corrupt)
    assert B.moe_device_status(b.workspace) == B.MOE_ERR_INDEX
    b.check()


def test_status_word_cleared_by_next_call():
    w = synth.custom("clear", seed=1, **FFN_CASES["tensor_core"])
    b = _ffn_after_valid_layer("tensor_core", lambda o, r: r.__setitem__(0, -1))
    assert B.moe_device_status(b.workspace) == B.MOE_ERR_INDEX
    layer = make_layer(w)
    layer.buf = b
    layer.forward(torch.from_numpy(synth.logits(w)).cuda(), bits_to_bf16_tensor(synth.hidden_bits(w)))
    assert B.moe_device_status(b.workspace) == 0
    b.check()
