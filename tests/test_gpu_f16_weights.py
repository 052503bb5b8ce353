"""The fp16 weight copies (moe_weights_to_f16) and the tensor-core GEMMs that
read them (batches above the decode size, both MMA operands from shared
memory): the copy is exact, and the layer on the copies equals the oracle
(and the int8-weight path) bit for bit in every return message.
"""
import numpy as np
import pytest
import torch

import oracle
from expert_dispatch_combine_gb300 import binding as B
from expert_dispatch_combine_gb300 import synth
from expert_dispatch_combine_gb300.layer import MoELayer

from gpu_util import (REL_L2, CanaryBuffers, bf16_tensor_to_bits, bits_to_bf16_tensor,
                      compare_bf16, lib, make_layer, shape_of)
from test_gpu_parity import _full_layer_check, _logits_for_counts, _special_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib()


def _np(t):
    return t.detach().cpu().numpy()


@pytest.mark.parametrize("n", [0, 5, 16, 4096 + 7, (1 << 20) + 3])
def test_weights_to_f16_exact(n):
    """Every int8 value, -128 and 127 included, becomes the fp16 of the same
    value (an 11-bit significand holds every 8-bit integer exactly)."""
    rng = np.random.default_rng(n)
    src = rng.integers(-128, 128, size=max(n, 1), dtype=np.int8)[:n].copy()
    if n >= 2:
        src[0], src[-1] = -128, 127
    d_src = torch.from_numpy(src).cuda()
    dst = torch.full((n,), float("nan"), dtype=torch.float16, device="cuda")
    B.moe_weights_to_f16(d_src, dst)
    torch.cuda.synchronize()
    assert (_np(dst).astype(np.float64) == src.astype(np.float64)).all()


# shapes with more than 32 routed rows per physical expert on average (the
# batches that read the copies)
F16_CASES = {
    "ragged_tiles": dict(T=300, H=256, E_log=4, k=4, I=128, R=2, S=3),          # 300 rows: 256 + 44
    "partial_block": dict(T=600, H=1088, E_log=8, k=2, I=192, R=2, S=4),        # 17 stages, 8.5 channel blocks
    "chunks": dict(T=520, H=2112, E_log=8, k=2, I=128, R=4, S=2),               # 33 stages: 3 exact chunks
    "zipf": dict(T=1024, H=512, E_log=16, k=4, I=256, R=8, S=4, zipf=1.3),      # hot experts, several tiles
    # tiles of at most 64 rows take two 64-K stages per ring slot; odd stage
    # counts (33 for gate/up, 3 for down) end on a zero-filled half slot
    "packed_odd": dict(T=200, H=2112, E_log=8, k=2, I=192, R=2, S=2, zipf=1.3),
}


@pytest.mark.parametrize("name", sorted(F16_CASES))
def test_layer_f16_weights_vs_oracle(name):
    w = synth.custom("f16_" + name, seed=21, **F16_CASES[name])
    assert w.T * w.k > 32 * w.E_phys
    _full_layer_check(w, B.MOE_MSG_INT8, f16_weights=True)


def test_layer_f16_weights_bf16_messages():
    w = synth.custom("f16_bf16msg", seed=22, **F16_CASES["partial_block"])
    _full_layer_check(w, B.MOE_MSG_BF16, f16_weights=True)


def test_layer_f16_weights_special_rows():
    w = synth.custom("f16_special", seed=23, T=256, H=256, E_log=8, k=2, I=128, R=4)
    _full_layer_check(w, B.MOE_MSG_INT8, xb=_special_rows(w), f16_weights=True)


def test_layer_f16_weights_eplb():
    w = synth.custom("f16_eplb", T=600, H=256, E_log=16, E_phys=24, k=2, I=128, R=8, seed=24,
                     zipf=1.2, eplb=True)
    _full_layer_check(w, B.MOE_MSG_INT8, f16_weights=True)


@pytest.mark.parametrize("counts", [
    [8, 9, 1, 2, 100, 16, 256, 120],   # narrow experts beside one- and two-tile experts
    [0, 3, 256, 15, 16, 0, 200, 22],
])
def test_layer_f16_weights_hybrid_narrow(counts):
    """Experts with 1..8 rows on the int8 matrix-vector kernels, the others on
    the fp16-copy GEMMs, in one layer."""
    T, E, k = 256, 8, 2
    w = synth.custom("f16_hybrid", seed=25, T=T, H=512, E_log=E, k=k, I=512, R=4, S=4)
    assert B.moe_expert_ffn_narrow_rows(shape_of(w)) == 8
    counts = np.array(counts)
    lg = _logits_for_counts(T, E, k, counts, seed=len(counts) + 1)
    _, _, _, cnt = oracle.route(lg, k)
    assert (cnt == counts).all()
    _full_layer_check(w, B.MOE_MSG_INT8, lg=lg, f16_weights=True)


def test_layer_f16_weights_sums_beyond_2p24():
    """Weights and activations near +127 everywhere: the gate/up sums reach
    about 2112 * 16129 = 3.4e7 > 2^24, so the exact 1024-K drains of the fp32
    accumulators decide every result; the oracle's sums are exact integers."""
    T, H, E, k, I = 300, 2112, 4, 2, 1088
    w = synth.custom("f16_big_sums", seed=26, T=T, H=H, E_log=E, k=k, I=I, R=2, S=2)
    rng = np.random.default_rng(26)
    f = np.ones((T, H), np.float32)
    m = rng.random((T, H)) < 0.05
    f[m] = rng.uniform(-1, 1, m.sum()).astype(np.float32)
    xb = synth.f32_to_bf16_bits(f)
    weights = {}
    for e in range(E):
        wgu = np.full((2 * I, H), 127, np.int8)
        m = rng.random(wgu.shape) < 0.1
        wgu[m] = rng.integers(-128, 128, m.sum()).astype(np.int8)
        wd = np.full((H, I), 127, np.int8)
        m = rng.random(wd.shape) < 0.2
        wd[m] = rng.integers(-128, 128, m.sum()).astype(np.int8)
        sgu = (rng.uniform(0.5, 1.5, 2 * I) * 1e-5).astype(np.float32)
        sd = (rng.uniform(0.5, 1.5, H) * 1e-5).astype(np.float32)
        weights[e] = (wgu, sgu, wd, sd)
    dev = torch.device("cuda")
    stack = [torch.from_numpy(np.stack([weights[e][n] for e in range(E)])).to(dev) for n in range(4)]
    shape = shape_of(w)
    layer = MoELayer(shape, *stack, buffers=CanaryBuffers(shape), f16_weights=True)
    lg = synth.logits(w)
    out = layer.forward(torch.from_numpy(lg).to(dev), bits_to_bf16_tensor(xb))
    torch.cuda.synchronize()
    ref = oracle.layer(lg, xb, weights, w.E_phys, w.R, w.S, w.k, w.I)
    b = layer.buf
    assert (_np(b.combine_rows()).view(np.int8) == ref["cbuf"]).all()
    assert (_np(b.combine_scales()) == ref["cscale"]).all()
    # the outputs here reach |y| ~ 8, beyond the absolute tolerance of the
    # standard workloads: against the oracle's combine (binary64 sum) on the
    # device's router weights, each output is within one bf16 ulp plus the
    # binary32 rounding of k products and sums
    wt = _np(b.routing["topk_w"])
    g = synth.bf16_bits_to_f32(bf16_tensor_to_bits(out)).astype(np.float64)
    r = synth.bf16_bits_to_f32(oracle.combine(ref["cbuf"], ref["cscale"], wt)).astype(np.float64)
    v = ref["cbuf"].astype(np.float64) * ref["cscale"][:, :, None].astype(np.float64)
    mag = np.abs(wt[:, :, None].astype(np.float64) * v).sum(axis=1)
    ulp = np.maximum(np.abs(r), np.abs(g)) * 2.0 ** -7
    assert (np.abs(g - r) <= ulp + 3 * k * 2.0 ** -24 * mag + 1e-38).all()
    max_abs, rel = compare_bf16(bf16_tensor_to_bits(out), ref["out"])
    assert rel <= REL_L2, (max_abs, rel)
    assert B.moe_device_status(b.workspace) == 0
    b.check()


def test_f16_copies_equal_int8_path_at_scale():
    """A larger batch (8192 rows, 512 per expert) on both weight forms: the
    return messages and the output agree bit for bit."""
    w = synth.custom("f16_vs_int8", seed=27, T=2048, H=1024, E_log=16, k=4, I=512, R=4, S=4,
                     zipf=1.1)
    lg = torch.from_numpy(synth.logits(w)).cuda()
    x = bits_to_bf16_tensor(synth.hidden_bits(w))
    res = []
    for f16 in (False, True):
        layer = make_layer(w, f16_weights=f16)
        out = layer.forward(lg, x).clone()
        torch.cuda.synchronize()
        res.append((out, layer.buf.combine_rows().clone(), layer.buf.combine_scales().clone()))
        assert B.moe_device_status(layer.buf.workspace) == 0
        layer.buf.check()
    assert torch.equal(res[0][1], res[1][1])
    assert torch.equal(res[0][2], res[1][2])
    assert torch.equal(res[0][0], res[1][0])


def test_f16_weights_fused_ffn_combine():
    """moe_expert_ffn_combine on the copies: same messages and output as the
    separate steps."""
    w = synth.custom("f16_fused", seed=28, **F16_CASES["ragged_tiles"])
    layer = make_layer(w, f16_weights=True)
    lg = torch.from_numpy(synth.logits(w)).cuda()
    x = bits_to_bf16_tensor(synth.hidden_bits(w))
    ref = layer.forward(lg, x).clone()
    ref_rows = layer.buf.combine_rows().clone()
    b, r, s = layer.buf, layer.buf.routing, layer.shape
    b.combine.zero_()
    out = torch.empty_like(ref)
    B.moe_expert_ffn_combine(s, b.dispatch, r["expert_offsets"], r["expert_rows"], *layer.w,
                             r["topk_w"], b.combine, out, b.workspace, w_f16=layer.w_f16)
    torch.cuda.synchronize()
    assert torch.equal(ref_rows, b.combine_rows())
    assert torch.equal(ref, out)
    assert B.moe_device_status(b.workspace) == 0
