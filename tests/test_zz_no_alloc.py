"""moe_dispatch_noalloc: FusedDispatch for callers that cannot allocate a
workspace (an engine whose allocator owns all device memory, a decode loop
that must not synchronise on an allocation, a plug-in without its own device
memory).  Its scratch is a fixed device array inside the library.

Checked through the C ABI against moe_dispatch (the workspace entry point) on
two calls in a row with different inputs, so the second call runs on the
first call's leftover scratch.  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

from expert_dispatch_combine_gb300 import binding as B
from expert_dispatch_combine_gb300 import synth

from gpu_util import bits_to_bf16_tensor, lib

pytestmark = pytest.mark.gpu


def _route(shape, lg):
    dev = torch.device("cuda")
    T, k, E = shape.T, shape.k, shape.E_phys
    idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    w = torch.empty((T, k), dtype=torch.float32, device=dev)
    p = torch.empty((T, k), dtype=torch.int32, device=dev)
    c = torch.empty((E,), dtype=torch.int32, device=dev)
    B.moe_route(shape, torch.from_numpy(lg).to(dev), idx, w, p, c)
    return p


def _outputs(shape, L):
    dev = torch.device("cuda")
    return dict(
        dbuf=torch.zeros(L["dispatch_bytes"], dtype=torch.uint8, device=dev),
        rank_counts=torch.full((shape.n_ranks, shape.n_src_ranks), -1, dtype=torch.int32, device=dev),
        offsets=torch.full((shape.E_phys + 1,), -1, dtype=torch.int32, device=dev),
        rows=torch.full((shape.T * shape.k,), -1, dtype=torch.int32, device=dev),
    )


def _dispatch_both(shape, lg, xb):
    L = B.moe_query_layout(shape)
    pidx = _route(shape, lg)
    x = bits_to_bf16_tensor(xb)
    ref = _outputs(shape, L)
    ws = torch.empty(L["workspace_bytes"], dtype=torch.uint8, device="cuda")
    B.moe_dispatch(shape, x, pidx, ref["dbuf"], ref["rank_counts"], ref["offsets"], ref["rows"], ws)
    got = _outputs(shape, L)
    B.moe_dispatch_noalloc(shape, x, pidx, got["dbuf"], got["rank_counts"], got["offsets"],
                           got["rows"])
    torch.cuda.synchronize()
    for key in ("rank_counts", "offsets", "rows"):
        assert torch.equal(ref[key], got[key]), key
    # every message row and its metadata (the bytes of unused slots are not
    # written by either call; both buffers start zeroed)
    assert torch.equal(ref["dbuf"], got["dbuf"])


@pytest.mark.parametrize("name", ["c1_decode", "c4_prefill"])
def test_noalloc_dispatch_matches_workspace_dispatch_twice(name):
    lib()
    w = synth.WORKLOADS[name]
    shape = B.Shape(w.T, w.H, w.E_log, w.E_phys, w.k, w.I, w.R, w.S)
    lg = synth.logits(w)
    xb = synth.hidden_bits(w)
    _dispatch_both(shape, lg, xb)
    # second call in a row, different routing and hidden rows
    rng = np.random.default_rng(99)
    lg2 = rng.standard_normal(lg.shape).astype(np.float32)
    xb2 = synth.f32_to_bf16_bits(rng.standard_normal(xb.shape).astype(np.float32))
    _dispatch_both(shape, lg2, xb2)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    lib()
    cap = B.moe_dispatch_noalloc_max_scratch()
    assert cap == 4 << 20
    # 2^19 messages need 8 bytes of scratch each (4 MiB) plus the histograms:
    # just beyond the fixed array, while every buffer the caller passes is
    # large enough -- the rejection comes from the scratch limit, before any
    # launch
    shape = B.Shape(65536, 16, 16, 16, 8, 16, 16, 16)
    L = B.moe_query_layout(shape)
    dev = torch.device("cuda")
    x = torch.empty((65536, 16), dtype=torch.int16, device=dev)
    pidx = torch.zeros((65536, 8), dtype=torch.int32, device=dev)
    d = torch.empty((L["dispatch_bytes"],), dtype=torch.uint8, device=dev)
    rc = torch.empty((16, 16), dtype=torch.int32, device=dev)
    off = torch.empty((17,), dtype=torch.int32, device=dev)
    rows = torch.empty((65536 * 8,), dtype=torch.int32, device=dev)
    with pytest.raises(B.MoeError) as e:
        B.moe_dispatch_noalloc(shape, x, pidx, d, rc, off, rows)
    assert e.value.code == 2
