"""Trampoline forward (two-hop FusedDispatch) against the one-hop dispatch:
every output (dispatch rows and meta, per-pair counts, expert offsets and
row lists) bit for bit, plus the contents of the trampolines' receive areas,
on small shapes with fewer source ranks than expert ranks (and equal), both
message formats, and at the full size of one 160-rank DP domain."""
import numpy as np
import pytest
import torch

import oracle
from expert_dispatch_combine_gb300 import binding as B
from expert_dispatch_combine_gb300 import synth
from expert_dispatch_combine_gb300.layer import LayerBuffers

from gpu_util import bits_to_bf16_tensor, eplb_map, lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib()


def _route(w, shape, buf, dev="cuda"):
    lg = torch.from_numpy(synth.logits(w)).to(dev)
    rep = nc = None
    if w.E_phys != w.E_log:
        r_, n_, _ = eplb_map(w)
        rep, nc = torch.from_numpy(r_).to(dev), torch.from_numpy(n_).to(dev)
    r = buf.routing
    B.moe_route(shape, lg, r["topk_idx"], r["topk_w"], r["phys_idx"], r["expert_counts"], rep, nc)
    return r


@pytest.mark.parametrize("fmt", [B.MOE_MSG_INT8, B.MOE_MSG_BF16])
@pytest.mark.parametrize("cfg", [
    dict(T=96, H=256, E_log=16, E_phys=24, k=2, I=64, R=12, S=8, zipf=1.2, plan_ranks=4),  # 8 -> 12 ranks
    dict(T=160, H=128, E_log=20, k=4, I=64, R=20, S=5),                     # 5 -> 20, epr = 1
    dict(T=64, H=256, E_log=16, k=3, I=64, R=4, S=4),                       # S = R
])
def test_trampoline_equals_direct_dispatch(cfg, fmt):
    w = synth.custom(seed=11, **cfg)
    shape = B.Shape(w.T, w.H, w.E_log, w.E_phys, w.k, w.I, w.R, w.S, fmt, B.MOE_MSG_INT8)
    buf = LayerBuffers(shape)
    r = _route(w, shape, buf)
    x = bits_to_bf16_tensor(synth.hidden_bits(w))
    buf.dispatch.zero_()
    B.moe_dispatch(shape, x, r["phys_idx"], buf.dispatch, r["rank_counts"], r["expert_offsets"],
                   r["expert_rows"], buf.workspace)
    torch.cuda.synchronize()
    ref = {n: r[n].clone() for n in ("rank_counts", "expert_offsets", "expert_rows")}
    ref_d = buf.dispatch.clone()
    buf.dispatch.zero_()
    for n in ref:
        r[n].fill_(-7)
    tbuf = torch.empty(B.moe_trampoline_bytes(shape), dtype=torch.uint8, device="cuda")
    B.moe_dispatch_trampoline(shape, x, r["phys_idx"], tbuf, buf.dispatch, r["rank_counts"],
                              r["expert_offsets"], r["expert_rows"], buf.workspace)
    torch.cuda.synchronize()
    assert torch.equal(buf.dispatch, ref_d)
    for n in ref:
        assert torch.equal(r[n], ref[n]), n
    # the trampolines' receive areas: each token once, with its scale and routes
    row_b = w.H if fmt == B.MOE_MSG_INT8 else 2 * w.H
    tb = tbuf.cpu().numpy()
    rows = tb[: w.T * row_b].reshape(w.T, row_b)
    meta_off = -(-w.T * row_b // 256) * 256
    meta = tb[meta_off: meta_off + 16 * w.T].view(np.int32).reshape(w.T, 4)
    routes_off = -(-(meta_off + 16 * w.T) // 256) * 256
    routes = tb[routes_off: routes_off + 4 * w.T * w.k].view(np.int32).reshape(w.T, w.k)
    pidx = r["phys_idx"].cpu().numpy()
    assert (routes == pidx).all()
    t = np.arange(w.T)
    assert (meta[:, 1] == t // w.lb).all() and (meta[:, 2] == t % w.lb).all() and (meta[:, 3] == w.k).all()
    if fmt == B.MOE_MSG_INT8:
        xq, xs = oracle.quantize_bf16(synth.hidden_bits(w))
        assert (rows.view(np.int8) == xq).all()
        assert (meta[:, 0].view(np.float32) == xs).all()
    else:
        assert (rows.view(np.uint16) == synth.hidden_bits(w)).all()


def test_trampoline_full_domain():
    """One DP domain of the pages' A2E configuration: 160 attention ranks x
    96 tokens to 288 expert ranks (k = 8, H = 7168)."""
    w = synth.WORKLOADS["tr_domain"]
    shape = B.Shape(w.T, w.H, w.E_log, w.E_phys, w.k, w.I, w.R, w.S, B.MOE_MSG_INT8, B.MOE_MSG_INT8)
    buf = LayerBuffers(shape)
    r = _route(w, shape, buf)
    x = bits_to_bf16_tensor(synth.hidden_bits(w))
    B.moe_dispatch(shape, x, r["phys_idx"], buf.dispatch, r["rank_counts"], r["expert_offsets"],
                   r["expert_rows"], buf.workspace)
    torch.cuda.synchronize()
    ref = {n: r[n].clone() for n in ("rank_counts", "expert_offsets", "expert_rows")}
    used = r["expert_rows"].long()
    ref_rows = buf.dispatch_rows()[used].clone()
    ref_meta = buf.dispatch_meta()[used].clone()
    buf.dispatch_rows()[used] = 0
    buf.dispatch_meta()[used] = 0
    for n in ref:
        r[n].fill_(-7)
    tbuf = torch.empty(B.moe_trampoline_bytes(shape), dtype=torch.uint8, device="cuda")
    B.moe_dispatch_trampoline(shape, x, r["phys_idx"], tbuf, buf.dispatch, r["rank_counts"],
                              r["expert_offsets"], r["expert_rows"], buf.workspace)
    torch.cuda.synchronize()
    for n in ref:
        assert torch.equal(r[n], ref[n]), n
    assert torch.equal(buf.dispatch_rows()[used], ref_rows)
    assert torch.equal(buf.dispatch_meta()[used], ref_meta)
    # and the layout is the oracle's
    d = oracle.dispatch(synth.hidden_bits(w), r["phys_idx"].cpu().numpy(), w.E_phys, w.R, w.S,
                        fmt=1, with_rows=False)
    assert (r["expert_rows"].cpu().numpy() == d["expert_rows"]).all()
    assert (r["rank_counts"].cpu().numpy() == d["rank_counts"]).all()
