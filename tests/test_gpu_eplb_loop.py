"""The EPLB loop on the GPU: Collect against a host bincount, the re-planned
map against the oracle planner fed with the oracle's own per-slice loads,
and forwards after the switch against the oracle's routing and against a
layer built directly with the new map."""
import numpy as np
import pytest
import torch

import oracle
from oracle import eplb
from expert_dispatch_combine_gb300 import binding as B
from expert_dispatch_combine_gb300 import synth
from expert_dispatch_combine_gb300.eplb_loop import EplbLoop
from expert_dispatch_combine_gb300.layer import MoELayer

from gpu_util import bits_to_bf16_tensor, lib, shape_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib()


def test_collect_sums_physical_copies_per_logical_expert():
    rng = np.random.default_rng(7)
    E_log, E_phys = 16, 24
    p2l = np.concatenate([np.arange(E_log), rng.integers(0, E_log, E_phys - E_log)]).astype(np.int32)
    load = torch.zeros(E_log, dtype=torch.int64, device="cuda")
    want = np.zeros(E_log, np.int64)
    for _ in range(3):
        cnt = rng.integers(0, 1000, E_phys).astype(np.int32)
        B.moe_eplb_collect(torch.from_numpy(cnt).cuda(), load, torch.from_numpy(p2l).cuda())
        want += np.bincount(p2l, weights=cnt, minlength=E_log).astype(np.int64)
    torch.cuda.synchronize()
    assert (load.cpu().numpy() == want).all()
    # identity map
    load.zero_()
    cnt = rng.integers(0, 5, E_log).astype(np.int32)
    B.moe_eplb_collect(torch.from_numpy(cnt).cuda(), load)
    torch.cuda.synchronize()
    assert (load.cpu().numpy() == cnt).all()


def _step_inputs(w, step):
    """Zipf-skewed logits whose hot experts move with the step."""
    rng = np.random.default_rng(100 + step)
    lg = rng.standard_normal((w.T, w.E_log)).astype(np.float32)
    perm = np.roll(np.arange(w.E_log), 3 * (step // 4))  # hot set shifts every window
    lg += (-1.5 * np.log1p(np.arange(w.E_log, dtype=np.float32)))[perm][None, :]
    xb = synth.hidden_bits(w)
    return lg, xb


def test_loop_replans_from_collected_loads_and_routes_with_new_map():
    w = synth.custom("eplb_loop", T=256, H=128, E_log=16, E_phys=24, k=2, I=64, R=8, seed=9)
    shape = shape_of(w, B.MOE_MSG_INT8, B.MOE_MSG_INT8)
    W = synth.all_weights_torch(w, "cuda")
    layer = MoELayer(shape, *W)
    loop = EplbLoop(layer, n_slices=2, steps_per_slice=2)
    # the initial map is the plan of a uniform load
    rep0, nc0, p2l0 = eplb.plan(np.ones((1, w.E_log)), w.E_phys, w.R)
    assert (loop.plans[0][3] == p2l0).all()

    host_loads = np.zeros((2, w.E_log), np.float64)
    for step in range(6):
        lg, xb = _step_inputs(w, step)
        lg_t, x_t = torch.from_numpy(lg).cuda(), bits_to_bf16_tensor(xb)
        rep_now, nc_now, p2l_now = loop.plans[-1][1:]
        out = loop.step(lg_t, x_t).clone()
        torch.cuda.synchronize()
        # routing of this forward used the map in force before the step
        idx, wt, pidx, _ = oracle.route(lg, w.k, w.E_phys, rep_now, nc_now)
        assert (layer.buf.routing["phys_idx"].cpu().numpy() == pidx).all()
        if step < 4:
            host_loads[(step // 2) % 2] += np.bincount(idx.ravel(), minlength=w.E_log)
        # the output equals a layer built directly with that map
        ref_layer = MoELayer(shape, *W, rep_table=torch.from_numpy(rep_now).cuda(),
                             n_copies=torch.from_numpy(nc_now).cuda(),
                             phys_to_weight=torch.from_numpy(p2l_now).cuda())
        assert torch.equal(ref_layer.forward(lg_t, x_t), out)
        if step == 3:
            # window closed: the loop re-planned from its collected loads
            assert len(loop.plans) == 2
            loads, rep1, nc1, p2l1 = loop.plans[1]
            assert (loads == host_loads).all()
            r_o, n_o, p_o = eplb.plan(host_loads, w.E_phys, w.R)
            assert (p2l1 == p_o).all() and (nc1 == n_o).all()
            m = min(rep1.shape[1], r_o.shape[1])
            assert (rep1[:, :m] == r_o[:, :m]).all() and (rep1[:, m:] == -1).all()
            assert not (p2l1 == p2l0).all()  # the skew moved copies
    assert B.moe_device_status(layer.buf.workspace) == 0
