"""The CUDA paths that other tests compare with CUDA, here compared with the
CPU oracle directly:

  - FusedDispatch with bf16 (unquantised) messages against the oracle's
    dispatch with bf16 rows: every used row, every metadata record, the
    layout arrays (small shapes in full; the prefill-shaped workload,
    T = 16384, on sampled tokens with its layout in full);
  - the decode layer replayed from CUDA graphs: every replayed step's return
    messages and output against the oracle layer on that step's inputs;
  - moe_expert_ffn_combine (the combine done per token once its k return
    messages are in): messages bit for bit and the output within tolerance
    against the oracle layer.
"""
import numpy as np
import pytest
import torch

import oracle
from expert_dispatch_combine_gb300 import binding as B
from expert_dispatch_combine_gb300 import synth
from expert_dispatch_combine_gb300.layer import GraphedLayer

from gpu_util import (MAX_ABS, REL_L2, CanaryBuffers, bf16_tensor_to_bits, bits_to_bf16_tensor,
                      compare_bf16, eplb_map, lib, make_layer, shape_of)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib()


def _np(t):
    return t.detach().cpu().numpy()


def _layout_and_meta(buf, d, used):
    r = buf.routing
    assert (_np(r["rank_counts"]) == d["rank_counts"]).all()
    assert (_np(r["expert_offsets"]) == d["expert_offsets"]).all()
    assert (_np(r["expert_rows"]) == d["expert_rows"]).all()
    meta = _np(buf.dispatch_meta()[torch.from_numpy(used.astype(np.int64)).cuda()])
    assert (meta[:, 0].view(np.float32) == d["meta_scale"][used]).all()
    assert (meta[:, 1] == d["meta_src"][used]).all()
    assert (meta[:, 2] == d["meta_bs"][used]).all()
    assert (meta[:, 3] == d["meta_rs"][used]).all()


# ------------------------------------------------------ bf16 dispatch rows
@pytest.mark.parametrize("cfg", [
    dict(T=64, H=256, E_log=16, k=2, I=128, R=4, S=4),
    dict(T=40, H=1088, E_log=12, k=3, I=192, R=3, S=5),
    dict(T=130, H=128, E_log=16, k=2, I=64, R=16, S=2),   # epr = 1
    dict(T=31, H=48, E_log=8, k=8, I=32, R=2, S=1),       # k = E
])
@pytest.mark.parametrize("trampoline", [False, True], ids=["direct", "trampoline"])
def test_bf16_dispatch_vs_oracle(cfg, trampoline):
    w = synth.custom("bf16_dispatch", seed=11, **cfg)
    if trampoline and w.S > w.R:
        pytest.skip("the trampoline forward needs n_src_ranks <= n_ranks")
    shape = shape_of(w, B.MOE_MSG_BF16, B.MOE_MSG_BF16)
    xb = synth.hidden_bits(w)
    _, _, pidx, _ = oracle.route(synth.logits(w), w.k)
    d = oracle.dispatch(xb, pidx, w.E_phys, w.R, w.S, fmt=0)
    buf = CanaryBuffers(shape)
    r = buf.routing
    x = bits_to_bf16_tensor(xb)
    p = torch.from_numpy(pidx).cuda()
    if trampoline:
        tb = torch.empty(B.moe_trampoline_bytes(shape), dtype=torch.uint8, device="cuda")
        B.moe_dispatch_trampoline(shape, x, p, tb, buf.dispatch, r["rank_counts"],
                                  r["expert_offsets"], r["expert_rows"], buf.workspace)
    else:
        B.moe_dispatch(shape, x, p, buf.dispatch, r["rank_counts"], r["expert_offsets"],
                       r["expert_rows"], buf.workspace)
    torch.cuda.synchronize()
    used = d["slot_of"].ravel()
    _layout_and_meta(buf, d, used)
    rows = _np(buf.dispatch_rows())
    assert (rows[used] == d["rows"][used]).all()
    assert (d["meta_scale"][used] == 0).all()
    assert B.moe_device_status(buf.workspace) == 0
    buf.check()


def test_bf16_dispatch_prefill_sampled():
    """The prefill-shaped workload (T = 16384, H = 7168, top-8, 32 x 32 ranks),
    bf16 messages: the layout and every metadata record in full, the message
    rows of sampled tokens (the bf16 static area is 60 GB)."""
    w = synth.WORKLOADS["c4_prefill"]
    shape = shape_of(w, B.MOE_MSG_BF16, B.MOE_MSG_BF16)
    xb = synth.hidden_bits(w)
    _, _, pidx, _ = oracle.route(synth.logits(w), w.k)
    d = oracle.dispatch(xb, pidx, w.E_phys, w.R, w.S, fmt=0, with_rows=False)
    buf = CanaryBuffers(shape)
    r = buf.routing
    B.moe_dispatch(shape, bits_to_bf16_tensor(xb), torch.from_numpy(pidx).cuda(), buf.dispatch,
                   r["rank_counts"], r["expert_offsets"], r["expert_rows"], buf.workspace)
    torch.cuda.synchronize()
    _layout_and_meta(buf, d, d["slot_of"].ravel())
    rng = np.random.default_rng(4)
    toks = sorted(set([0, 1, w.T // 2, w.T - 1] + rng.choice(w.T, 12, replace=False).tolist()))
    slots = d["slot_of"][toks].ravel().astype(np.int64)
    rows = _np(buf.dispatch_rows()[torch.from_numpy(slots).cuda()]).view(np.uint16)
    rows = rows.reshape(len(toks), w.k, w.H)
    assert (rows == xb[toks][:, None, :]).all()
    assert B.moe_device_status(buf.workspace) == 0
    buf.check()
    del buf
    torch.cuda.empty_cache()


# --------------------------------------------------------- CUDA-graph replay
def _step_inputs(w, step):
    rng = np.random.default_rng(1000 + step)
    lg = (synth.logits(w) + rng.standard_normal((w.T, w.E_log)).astype(np.float32) * 0.5)
    xb = np.ascontiguousarray(synth.hidden_bits(w)[rng.permutation(w.T)])
    return lg.astype(np.float32), xb


def _oracle_layer(w, lg, xb, cfmt=B.MOE_MSG_INT8):
    rep = nc = p2l = None
    if w.eplb:
        rep, nc, p2l = eplb_map(w)
    weights = {e: synth.expert_weights_np(w, e) for e in range(w.E_log)}
    return oracle.layer(lg, xb, weights, w.E_phys, w.R, w.S, w.k, w.I, cfmt, rep, nc, p2l)


@pytest.mark.parametrize("w,f16", [
    (synth.WORKLOADS["c0_tiny"], False),
    (synth.custom("eplb_tiny", T=96, H=128, E_log=16, E_phys=24, k=2, I=64, R=8, seed=3,
                  zipf=1.2, eplb=True), False),
    # 1024 routed rows over 8 experts: the tensor-core GEMMs on the fp16 weight
    # copies, and the dispatch writing their input rows, inside the graph
    (synth.custom("graph_f16", T=512, H=256, E_log=8, k=2, I=128, R=4, seed=5, zipf=1.2), True),
], ids=["c0_tiny", "eplb_tiny", "f16_copies"])
def test_graph_replay_vs_oracle(w, f16):
    layer = make_layer(w, f16_weights=f16)
    gl = GraphedLayer(layer, n_sets=2)
    try:
        for step in range(4):
            lg, xb = _step_inputs(w, step)
            out = gl.step(torch.from_numpy(lg).cuda(), bits_to_bf16_tensor(xb))
            torch.cuda.synchronize()
            buf = gl.sets[step % 2][0]
            ref = _oracle_layer(w, lg, xb)
            assert (_np(buf.routing["topk_idx"]) == ref["topk_idx"]).all(), step
            assert (_np(buf.combine_rows()).view(np.int8) == ref["cbuf"]).all(), step
            assert (_np(buf.combine_scales()) == ref["cscale"]).all(), step
            max_abs, rel = compare_bf16(bf16_tensor_to_bits(out), ref["out"])
            assert max_abs <= MAX_ABS and rel <= REL_L2, (step, max_abs, rel)
            assert B.moe_device_status(buf.workspace) == 0
    finally:
        gl.close()


# ------------------------------------------------ fused FFN + combine path
@pytest.mark.parametrize("w", [
    synth.WORKLOADS["c0_tiny"],
    synth.custom(seed=6, T=300, H=256, E_log=4, k=4, I=128, R=2, S=3),
    synth.custom(seed=8, T=64, H=128, E_log=16, k=12, I=64, R=4, S=4),
], ids=["c0_tiny", "tc_300x256", "k12"])
def test_fused_ffn_combine_vs_oracle(w):
    layer = make_layer(w)
    lg, xb = synth.logits(w), synth.hidden_bits(w)
    layer.forward(torch.from_numpy(lg).cuda(), bits_to_bf16_tensor(xb))
    b, r, s = layer.buf, layer.buf.routing, layer.shape
    w_gu, s_gu, w_d, s_d = layer.w
    b.combine.zero_()
    out = torch.empty((w.T, w.H), dtype=torch.bfloat16, device="cuda")
    B.moe_expert_ffn_combine(s, b.dispatch, r["expert_offsets"], r["expert_rows"], w_gu, s_gu, w_d,
                             s_d, r["topk_w"], b.combine, out, b.workspace)
    torch.cuda.synchronize()
    ref = _oracle_layer(w, lg, xb)
    assert (_np(b.combine_rows()).view(np.int8) == ref["cbuf"]).all()
    assert (_np(b.combine_scales()) == ref["cscale"]).all()
    max_abs, rel = compare_bf16(bf16_tensor_to_bits(out), ref["out"])
    assert max_abs <= MAX_ABS and rel <= REL_L2, (max_abs, rel)
    assert B.moe_device_status(b.workspace) == 0
    b.check()
