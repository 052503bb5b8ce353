"""GPU parity: the CUDA library (through the C ABI) against the CPU oracle.

Integer results (indices, counts, offsets, slots, metadata, INT8 codes,
int32 accumulators) must match bit for bit; binary32 scales bit for bit;
routing weights within 2e-6; bf16 layer outputs within max-abs 2e-2 and
relative L2 1e-3.
"""
import numpy as np
import pytest
import torch

import oracle
from expert_dispatch_combine_gb300 import binding as B
from expert_dispatch_combine_gb300 import synth

from gpu_util import (MAX_ABS, REL_L2, LayerBuffers, bf16_tensor_to_bits, bits_to_bf16_tensor,
                      compare_bf16, eplb_map, lib, make_layer, shape_of)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib()


def _np(t):
    return t.detach().cpu().numpy()


# ------------------------------------------------------------------- route
@pytest.mark.parametrize("name", list(synth.WORKLOADS))
def test_route_parity(name):
    w = synth.WORKLOADS[name]
    lg = synth.logits(w)
    rep = nc = None
    if w.eplb:
        rep, nc, _ = eplb_map(w)
    idx, wt, pidx, cnt = oracle.route(lg, w.k, w.E_phys, rep, nc)
    shape = shape_of(w)
    dev = torch.device("cuda")
    g_idx = torch.empty((w.T, w.k), dtype=torch.int32, device=dev)
    g_w = torch.empty((w.T, w.k), dtype=torch.float32, device=dev)
    g_p = torch.empty((w.T, w.k), dtype=torch.int32, device=dev)
    g_c = torch.full((w.E_phys,), -7, dtype=torch.int32, device=dev)
    rep_d = torch.from_numpy(rep).to(dev) if rep is not None else None
    nc_d = torch.from_numpy(nc).to(dev) if nc is not None else None
    B.moe_route(shape, torch.from_numpy(lg).to(dev), g_idx, g_w, g_p, g_c, rep_d, nc_d)
    torch.cuda.synchronize()
    assert (_np(g_idx) == idx).all()
    assert (_np(g_p) == pidx).all()
    assert (_np(g_c) == cnt).all()
    assert np.abs(_np(g_w) - wt).max() <= 2e-6


def test_route_ties_and_k_equals_e():
    T, E = 33, 16
    lg = np.random.default_rng(0).integers(0, 3, size=(T, E)).astype(np.float32)
    for k in (1, 5, 16):
        idx, wt, _, cnt = oracle.route(lg, k)
        shape = B.Shape(T, 16, E, E, k, 16, 1, 1)
        dev = torch.device("cuda")
        g_idx = torch.empty((T, k), dtype=torch.int32, device=dev)
        g_w = torch.empty((T, k), dtype=torch.float32, device=dev)
        g_p = torch.empty((T, k), dtype=torch.int32, device=dev)
        g_c = torch.empty((E,), dtype=torch.int32, device=dev)
        B.moe_route(shape, torch.from_numpy(lg).to(dev), g_idx, g_w, g_p, g_c)
        torch.cuda.synchronize()
        assert (_np(g_idx) == idx).all()
        assert (_np(g_c) == cnt).all()
        assert np.abs(_np(g_w) - wt).max() <= 2e-6


# -------------------------------------------------------------- whole layer
def _full_layer_check(w, cfmt, xb=None, lg=None, f16_weights=False):
    """Every intermediate and the output of moe_layer against the oracle
    (hidden rows and logits from the workload's generator unless xb, bf16
    bits, or lg, f32 logits, is given; with f16_weights the layer also holds
    the fp16 weight copies)."""
    layer = make_layer(w, cfmt, f16_weights=f16_weights)
    if lg is None:
        lg = synth.logits(w)
    if xb is None:
        xb = synth.hidden_bits(w)
    out = layer.forward(torch.from_numpy(lg).cuda(), bits_to_bf16_tensor(xb))
    torch.cuda.synchronize()
    rep = nc = p2l = None
    if w.eplb:
        rep, nc, p2l = eplb_map(w)
    need = range(w.E_log)
    weights = {e: synth.expert_weights_np(w, e) for e in need}
    ref = oracle.layer(lg, xb, weights, w.E_phys, w.R, w.S, w.k, w.I, cfmt, rep, nc, p2l)
    b = layer.buf
    r = b.routing
    assert (_np(r["topk_idx"]) == ref["topk_idx"]).all()
    assert (_np(r["phys_idx"]) == ref["phys_idx"]).all()
    assert (_np(r["expert_counts"]) == ref["counts"]).all()
    assert np.abs(_np(r["topk_w"]) - ref["topk_w"]).max() <= 2e-6
    d = ref["dispatch"]
    assert (_np(r["rank_counts"]) == d["rank_counts"]).all()
    assert (_np(r["expert_offsets"]) == d["expert_offsets"]).all()
    assert (_np(r["expert_rows"]) == d["expert_rows"]).all()
    used = d["slot_of"].ravel()
    rows = _np(b.dispatch_rows())
    assert (rows[used] == d["rows"][used]).all()
    meta = _np(b.dispatch_meta())
    assert (meta[used, 0].view(np.float32) == d["meta_scale"][used]).all()
    assert (meta[used, 1] == d["meta_src"][used]).all()
    assert (meta[used, 2] == d["meta_bs"][used]).all()
    assert (meta[used, 3] == d["meta_rs"][used]).all()
    crow = _np(b.combine_rows())
    if cfmt == B.MOE_MSG_INT8:
        assert (crow.view(np.int8) == ref["cbuf"]).all()
        assert (_np(b.combine_scales()) == ref["cscale"]).all()
    else:
        assert (crow.view(np.uint16) == ref["cbuf"]).all()
    max_abs, rel = compare_bf16(bf16_tensor_to_bits(out), ref["out"])
    assert max_abs <= MAX_ABS and rel <= REL_L2, (max_abs, rel)
    assert B.moe_device_status(b.workspace) == 0
    b.check()  # no kernel wrote past any caller buffer


@pytest.mark.parametrize("cfmt", [B.MOE_MSG_INT8, B.MOE_MSG_BF16])
def test_layer_tiny_full(cfmt):
    _full_layer_check(synth.WORKLOADS["c0_tiny"], cfmt)


@pytest.mark.parametrize("cfg", [
    # tensor-core expert path (H, I multiples of 64)
    dict(T=130, H=128, E_log=16, k=2, I=64, R=16, S=2),   # epr = 1, ragged token tiles
    dict(T=40, H=1088, E_log=12, k=3, I=192, R=3, S=5),   # K = 17 stages (2 exact chunks), partial channel block
    dict(T=300, H=256, E_log=4, k=4, I=128, R=2, S=3),    # k = E: 300 rows per expert, 3 token tiles
    dict(T=512, H=256, E_log=64, k=4, I=128, R=8, S=4, zipf=1.5),  # decode tiles, hot experts span several
    # decode path: CUDA-core matrix-vector products (<= 4 rows per expert, H and I multiples of 512)
    dict(T=48, H=1024, E_log=32, k=2, I=512, R=8, S=4),   # 1-6 rows per expert, empty experts
    dict(T=40, H=512, E_log=64, k=4, I=1024, R=4, S=5, zipf=1.5),  # hot experts above 8 rows: several passes
    # CUDA-core expert path (H or I not a multiple of 64)
    dict(T=1, H=16, E_log=4, k=1, I=16, R=1),             # one token
    dict(T=31, H=48, E_log=8, k=8, I=32, R=2, S=1),       # k = E, ragged
    dict(T=40, H=64, E_log=12, k=3, I=48, R=3, S=5),      # epr = 4 > k
    dict(T=130, H=272, E_log=16, k=2, I=144, R=16, S=2),  # epr = 1, ragged tiles
])
def test_layer_edge_shapes(cfg):
    _full_layer_check(synth.custom(seed=5, **cfg), B.MOE_MSG_INT8)


def _special_rows(w):
    """Hidden rows for the degenerate cases of token-wise quantisation: +0 and
    -0 rows (scale 0, codes 0, and then h = 0 and y = 0 down the whole FFN),
    a single non-zero at the first index, the absmax at the last index,
    quotients on half-integers (round-half-even decides 62.5 -> 62, -2.5 -> -2),
    tiny and large magnitudes, a constant row (every code 127), and rows
    whose scales (of x, or of h further on) are binary32 subnormals."""
    xb = synth.hidden_bits(w).copy()
    f = synth.bf16_bits_to_f32(xb)
    H = w.H
    f[0] = 0.0
    f[2] = 0.0
    f[2, 0] = 3.0
    f[3, -1] = -8.0 * np.abs(f[3]).max()
    f[4] = 0.0
    f[4, :5] = [127.0, 62.5, -0.5, 1.5, -2.5]
    f[5] *= 1e-30
    f[6] *= 1e4
    f[7] = 0.75
    f[8] *= 1e-20   # h lands in the binary32 subnormals: subnormal scale s_h
    f[9] *= 1e-37   # subnormal dispatch scale absmax / 127
    xb = synth.f32_to_bf16_bits(f)
    xb[1] = 0x8000  # -0.0
    assert H >= 5
    return xb


@pytest.mark.parametrize("dims", [
    dict(T=64, H=256, E_log=16, k=2, I=128, R=4),            # tensor-core expert path
    dict(T=16, H=512, E_log=16, k=2, I=512, R=4, S=2),       # decode matrix-vector path
    dict(T=16, H=48, E_log=8, k=2, I=32, R=2),               # CUDA-core expert path
])
def test_layer_special_rows(dims):
    w = synth.custom("special_rows", seed=7, **dims)
    _full_layer_check(w, B.MOE_MSG_INT8, xb=_special_rows(w))


def _logits_for_counts(T, E, k, counts, seed):
    """Logits whose top-k routing gives each expert e exactly counts[e] rows
    (sum = T * k, each count at most T): the list in which expert e appears
    counts[e] times, expert by expert, fills slot j of token t at position
    j * T + t, so an expert's copies (fewer than T apart) never meet in one
    token; the chosen experts get large distinct logits."""
    rng = np.random.default_rng(seed)
    deck = np.repeat(np.arange(E), counts)
    assert len(deck) == T * k and max(counts) <= T
    lg = rng.standard_normal((T, E)).astype(np.float32)
    choice = deck.reshape(k, T).T
    for t in range(T):
        for j, e in enumerate(choice[t]):
            lg[t, e] = 20.0 - j
    return lg


@pytest.mark.parametrize("counts", [
    [8, 9, 1, 2, 60, 16, 120, 40],      # both sides of the 8-row threshold, one expert at 8
    [0, 3, 128, 15, 16, 0, 17, 77],     # empty experts, one in every token
])
def test_layer_hybrid_narrow_experts(counts):
    """Tensor-core path with the narrow experts (1..8 rows) on the
    matrix-vector kernels: H and I multiples of 512, INT8 return messages."""
    T, E, k = 128, 8, 2
    w = synth.custom("hybrid", seed=13, T=T, H=512, E_log=E, k=k, I=512, R=4, S=4)
    assert B.moe_expert_ffn_path(shape_of(w)) == B.MOE_FFN_TENSOR_CORE
    assert B.moe_expert_ffn_narrow_rows(shape_of(w)) == 8
    counts = np.array(counts)
    lg = _logits_for_counts(T, E, k, counts, seed=len(counts))
    _, _, _, cnt = oracle.route(lg, k)
    assert (cnt == counts).all()
    _full_layer_check(w, B.MOE_MSG_INT8, lg=lg)


def test_layer_eplb_tiny():
    w = synth.custom("eplb_tiny", T=96, H=128, E_log=16, E_phys=24, k=2, I=64, R=8, seed=3,
                     zipf=1.2, eplb=True)
    _full_layer_check(w, B.MOE_MSG_INT8)


def test_layer_eplb_decode_path():
    # replicas alias their logical expert's weights on the decode (matrix-vector) path
    w = synth.custom("eplb_decode", T=32, H=512, E_log=16, E_phys=24, k=2, I=512, R=8, seed=4,
                     zipf=1.2, eplb=True)
    _full_layer_check(w, B.MOE_MSG_INT8)


# ----------------------------------------------------------------- combine
@pytest.mark.parametrize("cfmt", [B.MOE_MSG_INT8, B.MOE_MSG_BF16])
def test_combine_on_synthetic_messages(cfmt):
    T, H, k, E = 77, 7168, 8, 256
    rng = np.random.default_rng(12)
    _, wt, _, _ = oracle.route(rng.standard_normal((T, E)).astype(np.float32), k)
    shape = B.Shape(T, H, E, E, k, 16, 32, 1, B.MOE_MSG_INT8, cfmt)
    buf = LayerBuffers(shape)
    if cfmt == B.MOE_MSG_INT8:
        cb = rng.integers(-127, 128, size=(T, k, H)).astype(np.int8)
        cs = rng.uniform(1e-4, 1e-2, size=(T, k)).astype(np.float32)
        buf.combine_rows().copy_(torch.from_numpy(cb.view(np.uint8)).cuda())
        buf.combine_scales().copy_(torch.from_numpy(cs).cuda())
    else:
        cb = synth.f32_to_bf16_bits(rng.standard_normal((T, k, H)).astype(np.float32))
        cs = np.zeros((T, k), np.float32)
        buf.combine_rows().copy_(torch.from_numpy(cb.view(np.uint8).reshape(T, k, 2 * H)).cuda())
    B.moe_combine(shape, buf.combine, torch.from_numpy(wt).cuda(), buf.out)
    torch.cuda.synchronize()
    ref = oracle.combine(cb, cs, wt, cfmt)
    max_abs, rel = compare_bf16(bf16_tensor_to_bits(buf.out), ref)
    assert max_abs <= MAX_ABS and rel <= REL_L2
    # binary32 accumulation vs binary64: the difference is bounded by one bf16
    # ulp of the result plus the binary32 rounding of k products and sums
    g = synth.bf16_bits_to_f32(bf16_tensor_to_bits(buf.out)).astype(np.float64)
    r = synth.bf16_bits_to_f32(ref).astype(np.float64)
    if cfmt == B.MOE_MSG_INT8:
        v = cb.astype(np.float64) * cs[:, :, None].astype(np.float64)
    else:
        v = synth.bf16_bits_to_f32(cb).astype(np.float64)
    mag = np.abs(wt[:, :, None].astype(np.float64) * v).sum(axis=1)
    ulp = np.maximum(np.abs(r), np.abs(g)) * 2.0 ** -7
    assert (np.abs(g - r) <= ulp + 3 * k * 2.0 ** -24 * mag + 1e-38).all()
    assert (g == r).mean() > 0.99


# ------------------------------------------------------ grouped int8 GEMM
@pytest.mark.parametrize("K,N", [(7168, 64), (2048, 256), (48, 32)])
def test_grouped_gemm_exact_worst_case(K, N):
    """|sum| up to K*127*127 (> 2^24 for K >= 1041): int32 must be exact."""
    rng = np.random.default_rng(K)
    G = 5
    sizes = np.array([0, 130, 1, 64, 257])
    offs = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    M = int(offs[-1])
    A = np.where(rng.random((M, K)) < 0.5, 127, -127).astype(np.int8)
    A[::7] = 127
    Bw = np.where(rng.random((G, N, K)) < 0.5, 127, -127).astype(np.int8)
    Bw[:, ::5] = 127
    Bw[:, 1::5] = -127
    ref = np.empty((M, N), np.int64)
    for g in range(G):
        a = A[offs[g]:offs[g + 1]].astype(np.int64)
        ref[offs[g]:offs[g + 1]] = a @ Bw[g].astype(np.int64).T
    ws = torch.empty(B.moe_gemm_workspace_bytes(G, M, K), dtype=torch.uint8, device="cuda")
    C = torch.empty((M, N), dtype=torch.int32, device="cuda")
    B.moe_grouped_gemm_s8(torch.from_numpy(offs).cuda(), M, torch.from_numpy(A).cuda(), K,
                          torch.from_numpy(Bw).cuda(), C, ws)
    torch.cuda.synchronize()
    assert (_np(C).astype(np.int64) == ref).all()
    assert B.moe_device_status(ws) == 0


@pytest.mark.parametrize("c", [18, 19, 36, 37, 73, 74, 127])
def test_grouped_gemm_sums_beyond_2p24(c):
    """Rows of codes with magnitude c, except c - 1 at every 16th element, and
    weights 127 * sign(code) on the even channels: every product is positive,
    the sums grow to 127 * sum |a| (up to 115 M at K = 7168, far beyond 2^24)
    and every 16-element block adds an odd amount, so no fp32 accumulator
    could hold the whole sum exactly; the drains every 1024 K keep the int32
    results exact."""
    K, N = 7168, 64
    rng = np.random.default_rng(c)
    G = 2
    sizes = np.array([130, 77])
    offs = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    M = int(offs[-1])
    mag = np.where(np.arange(K) % 16 == 0, c - 1, c)
    sign = np.where(rng.random((M, K)) < 0.5, 1, -1)
    A = (sign * mag).astype(np.int8)
    Bw = np.where(rng.random((G, N, K)) < 0.5, 127, -127).astype(np.int8)
    Bw[:, ::2] = (127 * sign[0]).astype(np.int8)   # even channels follow row 0's signs
    ref = np.empty((M, N), np.int64)
    for g in range(G):
        ref[offs[g]:offs[g + 1]] = A[offs[g]:offs[g + 1]].astype(np.int64) @ Bw[g].astype(np.int64).T
    assert np.abs(ref).max() == 127 * int(mag.sum())  # row 0 reaches the full sum
    ws = torch.empty(B.moe_gemm_workspace_bytes(G, M, K), dtype=torch.uint8, device="cuda")
    C = torch.empty((M, N), dtype=torch.int32, device="cuda")
    B.moe_grouped_gemm_s8(torch.from_numpy(offs).cuda(), M, torch.from_numpy(A).cuda(), K,
                          torch.from_numpy(Bw).cuda(), C, ws)
    torch.cuda.synchronize()
    assert (_np(C).astype(np.int64) == ref).all()
    assert B.moe_device_status(ws) == 0


@pytest.mark.parametrize("K", [64, 192, 320])
def test_grouped_gemm_odd_stage_counts_many_tiles(K):
    """1, 3 or 5 K stages of 64 per tile, and several tiles per CTA, so that
    stage pairs of one element follow each other across tiles."""
    rng = np.random.default_rng(K + 1)
    G, N = 4, 512
    sizes = np.array([6000, 5999, 6100, 5901])
    offs = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    M = int(offs[-1])
    A = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    Bw = rng.integers(-127, 128, size=(G, N, K)).astype(np.int8)
    ref = np.empty((M, N), np.int64)
    for g in range(G):
        ref[offs[g]:offs[g + 1]] = A[offs[g]:offs[g + 1]].astype(np.int64) @ Bw[g].astype(np.int64).T
    ws = torch.empty(B.moe_gemm_workspace_bytes(G, M, K), dtype=torch.uint8, device="cuda")
    C = torch.empty((M, N), dtype=torch.int32, device="cuda")
    B.moe_grouped_gemm_s8(torch.from_numpy(offs).cuda(), M, torch.from_numpy(A).cuda(), K,
                          torch.from_numpy(Bw).cuda(), C, ws)
    torch.cuda.synchronize()
    assert (_np(C).astype(np.int64) == ref).all()
    assert B.moe_device_status(ws) == 0


@pytest.mark.parametrize("N,K,lda", [(48, 96, 112), (144, 128, 160), (16, 1024, 1024)])
def test_grouped_gemm_gather_rows(N, K, lda):
    rng = np.random.default_rng(1)
    G = 3
    sizes = [5, 0, 9]
    offs = np.array([0, 5, 5, 14], np.int32)
    A = rng.integers(-127, 128, size=(40, lda)).astype(np.int8)
    ridx = rng.permutation(40)[:14].astype(np.int32)
    Bw = rng.integers(-127, 128, size=(G, N, K)).astype(np.int8)
    ref = np.empty((14, N), np.int64)
    for g in range(G):
        for r in range(offs[g], offs[g + 1]):
            ref[r] = Bw[g].astype(np.int64) @ A[ridx[r], :K].astype(np.int64)
    ws = torch.empty(B.moe_gemm_workspace_bytes(G, 14, K), dtype=torch.uint8, device="cuda")
    C = torch.empty((14, N), dtype=torch.int32, device="cuda")
    B.moe_grouped_gemm_s8(torch.from_numpy(offs).cuda(), 14, torch.from_numpy(A).cuda(), lda,
                          torch.from_numpy(Bw).cuda(), C, ws, row_index=torch.from_numpy(ridx).cuda())
    torch.cuda.synchronize()
    assert (_np(C).astype(np.int64) == ref).all()
    assert B.moe_device_status(ws) == 0


def test_weights_generated_on_device_equal_host():
    w = synth.WORKLOADS["c1_decode"]
    a = synth.int8_tensor_torch(w.seed, 17, synth.GATE_UP, (2 * w.I, w.H), device="cuda")
    b = synth.int8_tensor_np(w.seed, 17, synth.GATE_UP, (2 * w.I, w.H))
    assert (_np(a) == b).all()


@pytest.mark.parametrize("w", [
    synth.WORKLOADS["c0_tiny"],
    synth.custom(seed=6, T=300, H=256, E_log=4, k=4, I=128, R=2, S=3),
    synth.custom(seed=8, T=64, H=128, E_log=16, k=12, I=64, R=4, S=4),
    synth.WORKLOADS["c1_decode"],
], ids=["c0_tiny", "tc_300x256", "k12", "c1_decode"])
def test_fused_ffn_combine_equals_separate_steps(w):
    """moe_expert_ffn_combine (combine per token once its k messages are in,
    readiness counters) gives the messages and output of moe_expert_ffn
    followed by moe_combine, bit for bit."""
    layer = make_layer(w)
    lg = torch.from_numpy(synth.logits(w)).cuda()
    x = bits_to_bf16_tensor(synth.hidden_bits(w))
    ref = layer.forward(lg, x).clone()
    ref_rows = layer.buf.combine_rows().clone()
    ref_scales = layer.buf.combine_scales().clone()
    b, r, s = layer.buf, layer.buf.routing, layer.shape
    w_gu, s_gu, w_d, s_d = layer.w
    b.combine.zero_()
    out = torch.empty_like(ref)
    for _ in range(2):  # the readiness counters start from zero on every call
        B.moe_expert_ffn_combine(s, b.dispatch, r["expert_offsets"], r["expert_rows"], w_gu, s_gu,
                                 w_d, s_d, r["topk_w"], b.combine, out, b.workspace)
        torch.cuda.synchronize()
        assert torch.equal(ref_rows, b.combine_rows())
        assert torch.equal(ref_scales, b.combine_scales())
        assert torch.equal(ref, out)
