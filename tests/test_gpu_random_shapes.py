"""Seeded sweep of random layer shapes against the oracle: every intermediate
and the output of moe_layer (the same checks as the hand-picked shapes of
test_gpu_parity.py), on shapes nobody chose: hidden and intermediate sizes
that are multiples of 64 but not of the tiles (and, on two seeds, not of 64:
the CUDA-core path), decode-sized batches (the matrix-vector path), odd
expert counts, skewed routing, EPLB replicas, both weight forms and both
return formats.  Each
shape is printed in the test id, so a failure names the case to reproduce."""
import numpy as np
import pytest

from expert_dispatch_combine_gb300 import binding as B
from expert_dispatch_combine_gb300 import synth

from gpu_util import lib
from test_gpu_parity import _full_layer_check

pytestmark = pytest.mark.gpu


def _shape(seed: int) -> dict:
    rng = np.random.default_rng(1000 + seed)
    R = int(rng.choice([2, 4, 8]))
    S = int(rng.choice([1, 2, 4, 8]))
    # logical experts a multiple of R (the replica planner places the primary
    # experts evenly over the ranks); physical experts beyond them only with
    # EPLB, one redundant slot per rank, whose replica map and weight
    # aliasing give every physical expert its weights
    E_log = R * int(rng.integers(1, max(2, 32 // R) + 1))
    eplb = bool(rng.random() < 0.3)
    E_phys = E_log + (R if eplb else 0)
    k = int(rng.integers(1, min(8, E_log) + 1))
    lb = int(rng.integers(4, 97))
    T = S * lb
    # keep the oracle to about a second: at most ~2048 routed rows of H x I <= 1.2M
    while T * k > 2048 and lb > 4:
        lb = max(4, lb // 2)
        T = S * lb
    H = 64 * int(rng.integers(2, 34))
    I = 64 * int(rng.integers(1, 18))
    while H * I > 1_200_000:
        I = max(64, I - 64) if I > 64 else I
        H = H - 64 if H * I > 1_200_000 and H > 128 else H
    if seed % 8 == 6:
        # H or I not a multiple of 64: the CUDA-core path
        H, I = H - 48, I + 16
    zipf = float(rng.choice([0.0, 0.0, 1.1, 1.4]))
    f16 = bool(rng.random() < 0.5)
    cfmt = B.MOE_MSG_BF16 if seed % 4 == 3 else B.MOE_MSG_INT8
    if seed % 4 == 1:
        # a decode-sized batch (at most 4 routed rows per physical expert):
        # the matrix-vector path when H and I are multiples of 512, else the
        # CUDA-core path
        if seed % 8 == 1:
            H, I = 512 * int(rng.integers(1, 5)), 512 * int(rng.integers(1, 3))
        lb = max(1, (4 * E_phys) // (k * S))
        T = S * lb
    return dict(T=T, H=H, E_log=E_log, E_phys=E_phys, k=k, I=I, R=R, S=S, zipf=zipf, eplb=eplb,
                f16=f16, cfmt=cfmt)


SHAPES = [_shape(s) for s in range(16)]


def _id(c):
    return ("T{T}_H{H}_E{E_log}p{E_phys}_k{k}_I{I}_R{R}S{S}_z{zipf}{e}{f}{m}".format(
        e="_eplb" if c["eplb"] else "", f="_f16" if c["f16"] else "",
        m="_bf16msg" if c["cfmt"] == B.MOE_MSG_BF16 else "", **c))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib()


@pytest.mark.parametrize("c", SHAPES, ids=[_id(c) for c in SHAPES])
def test_random_shape_layer_vs_oracle(c):
    w = synth.custom("rand", seed=77, T=c["T"], H=c["H"], E_log=c["E_log"], E_phys=c["E_phys"],
                     k=c["k"], I=c["I"], R=c["R"], S=c["S"], zipf=c["zipf"], eplb=c["eplb"])
    _full_layer_check(w, c["cfmt"], f16_weights=c["f16"])


def _large(seed: int) -> dict:
    """Shapes with many token tiles per expert on the fp16 copies: 4096 to
    8192 routed rows over 8 or 16 experts, skewed so that the hottest ones
    span more than one raster band of 8 token tiles."""
    rng = np.random.default_rng(2000 + seed)
    R = 8
    E_log = int(rng.choice([8, 16]))
    k = int(rng.choice([2, 4]))
    T = 8 * int(rng.integers(512 // k, 1024 // k + 1))
    H = 64 * int(rng.integers(4, 17))
    I = 64 * int(rng.integers(2, 9))
    return dict(T=T, H=H, E_log=E_log, E_phys=E_log, k=k, I=I, R=R, S=8, zipf=float(rng.choice([1.2, 1.6])),
                eplb=False, f16=True, cfmt=B.MOE_MSG_INT8)


LARGE = [_large(s) for s in range(4)]


@pytest.mark.parametrize("c", LARGE, ids=[_id(c) for c in LARGE])
def test_random_large_shape_layer_vs_oracle(c):
    w = synth.custom("rand_large", seed=78, T=c["T"], H=c["H"], E_log=c["E_log"], E_phys=c["E_phys"],
                     k=c["k"], I=c["I"], R=c["R"], S=c["S"], zipf=c["zipf"], eplb=False)
    _full_layer_check(w, c["cfmt"], f16_weights=True)
