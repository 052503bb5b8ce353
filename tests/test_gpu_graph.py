"""The decode layer replayed from CUDA graphs over double-buffered static
buffers gives, step after step, the same outputs as eager moe_layer calls, and
a step's output stays intact while the next step runs in the other set."""
import numpy as np
import pytest
import torch

from expert_dispatch_combine_gb300 import synth
from expert_dispatch_combine_gb300.layer import GraphedLayer

from gpu_util import bits_to_bf16_tensor, lib, make_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib()


def _inputs(w, step):
    rng = np.random.default_rng(1000 + step)
    lg = synth.logits(w) + rng.standard_normal((w.T, w.E_log)).astype(np.float32) * 0.5
    xb = synth.hidden_bits(w)[rng.permutation(w.T)]
    return torch.from_numpy(lg).cuda(), bits_to_bf16_tensor(np.ascontiguousarray(xb))


@pytest.mark.parametrize("w", [
    synth.WORKLOADS["c0_tiny"],
    synth.custom(seed=5, T=300, H=256, E_log=4, k=4, I=128, R=2, S=3),
    synth.custom("eplb_tiny", T=96, H=128, E_log=16, E_phys=24, k=2, I=64, R=8, seed=3,
                 zipf=1.2, eplb=True),
    synth.WORKLOADS["c1_decode"],
], ids=["c0_tiny", "tc_300x256", "eplb_tiny", "c1_decode"])
def test_graph_replay_matches_eager(w):
    layer = make_layer(w)
    gl = GraphedLayer(layer, n_sets=2)
    prev = None
    for step in range(5):
        lg, x = _inputs(w, step)
        ref = layer.forward(lg, x).clone()
        out = gl.step(lg, x)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), step
        if prev is not None:  # the other buffer set still holds the previous step
            assert torch.equal(prev[0], prev[1])
        prev = (out, ref)
    gl.close()
