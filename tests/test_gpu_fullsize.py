"""Full-size parity: the DeepSeek-V3-shaped workloads through moe_layer (the
launch configuration bench.py times, with and without the fp16 weight
copies), compared with the oracle

  - in full for every index array (routing, counts, dispatch layout, meta);
  - on sampled tokens for the INT8 codes of the dispatch messages, the return
    messages (codes + scales, bit-exact) and the layer output (tolerance),
    which the oracle computes one (token, route) at a time.
"""
import numpy as np
import pytest
import torch

import oracle
from expert_dispatch_combine_gb300 import binding as B
from expert_dispatch_combine_gb300 import synth

from gpu_util import (MAX_ABS, REL_L2, bf16_tensor_to_bits, bits_to_bf16_tensor, compare_bf16,
                      eplb_map, lib, make_layer)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib()


def _np(t):
    return t.detach().cpu().numpy()


def _sample(T, n=10, seed=0):
    rng = np.random.default_rng(seed)
    base = [0, 1, T // 2, T - 1]
    extra = rng.choice(T, size=min(T, n), replace=False).tolist()
    return sorted(set(base + extra))


@pytest.mark.parametrize("name,f16", [
    ("c1_decode", False), ("c2_decode_zipf", False), ("c3_eplb", False), ("c4_prefill", False),
    # the tensor-core GEMMs on the fp16 weight copies (bench.py's default form)
    ("c2_decode_zipf", True), ("c3_eplb", True), ("c4_prefill", True),
])
def test_fullsize_layer_sampled(name, f16):
    w = synth.WORKLOADS[name]
    layer = make_layer(w, f16_weights=f16)
    lg = synth.logits(w)
    xb = synth.hidden_bits(w)
    out = layer.forward(torch.from_numpy(lg).cuda(), bits_to_bf16_tensor(xb))
    torch.cuda.synchronize()
    b = layer.buf
    r = b.routing
    assert B.moe_device_status(b.workspace) == 0

    rep = nc = p2l = None
    if w.eplb:
        rep, nc, p2l = eplb_map(w)
    # ---- every index array in full
    idx, wt, pidx, cnt = oracle.route(lg, w.k, w.E_phys, rep, nc)
    assert (_np(r["topk_idx"]) == idx).all()
    assert (_np(r["phys_idx"]) == pidx).all()
    assert (_np(r["expert_counts"]) == cnt).all()
    assert np.abs(_np(r["topk_w"]) - wt).max() <= 2e-6
    d = oracle.dispatch(xb, pidx, w.E_phys, w.R, w.S, fmt=1, with_rows=False)
    assert (_np(r["rank_counts"]) == d["rank_counts"]).all()
    assert (_np(r["expert_offsets"]) == d["expert_offsets"]).all()
    assert (_np(r["expert_rows"]) == d["expert_rows"]).all()
    used = d["slot_of"].ravel()
    meta = _np(b.dispatch_meta()[torch.from_numpy(used.astype(np.int64)).cuda()])
    assert (meta[:, 0].view(np.float32) == d["meta_scale"][used]).all()
    assert (meta[:, 1] == d["meta_src"][used]).all()
    assert (meta[:, 2] == d["meta_bs"][used]).all()
    assert (meta[:, 3] == d["meta_rs"][used]).all()

    # ---- sampled tokens: codes, return messages, output
    toks = _sample(w.T, seed=w.seed)
    xq, xs = oracle.quantize_bf16(np.ascontiguousarray(xb[toks]))
    slots = d["slot_of"][toks]                       # [n, k]
    rows = _np(b.dispatch_rows()[torch.from_numpy(slots.ravel().astype(np.int64)).cuda()])
    rows = rows.reshape(len(toks), w.k, w.H).view(np.int8)
    assert (rows == xq[:, None, :]).all()
    need = sorted({int(p2l[p]) if p2l is not None else int(p) for p in pidx[toks].ravel()})
    weights = {e: synth.expert_weights_np(w, e) for e in need}
    cb, cs = oracle.ffn_all(xq, xs, np.ascontiguousarray(pidx[toks]), weights, w.I, 1, p2l)
    g_cb = _np(b.combine_rows()[torch.tensor(toks).cuda()]).view(np.int8)
    g_cs = _np(b.combine_scales()[torch.tensor(toks).cuda()])
    assert (g_cb == cb).all()
    assert (g_cs == cs).all()
    ref_out = oracle.combine(cb, cs, np.ascontiguousarray(wt[toks]), 1)
    max_abs, rel = compare_bf16(bf16_tensor_to_bits(out)[toks], ref_out)
    assert max_abs <= MAX_ABS and rel <= REL_L2, (max_abs, rel)
    del layer
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name,f16", [("c1_decode", False), ("c2_decode_zipf", True)])
def test_fullsize_repeat_is_bitwise_deterministic(name, f16):
    w = synth.WORKLOADS[name]
    layer = make_layer(w, f16_weights=f16)
    lg = torch.from_numpy(synth.logits(w)).cuda()
    x = bits_to_bf16_tensor(synth.hidden_bits(w))
    a = layer.forward(lg, x).clone()
    ca = layer.buf.combine.clone()
    for _ in range(3):
        bb = layer.forward(lg, x)
        assert torch.equal(a, bb)
        assert torch.equal(ca, layer.buf.combine)
