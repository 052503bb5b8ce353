"""Rate of the legacy warp-level INT8 tensor-core MMA (mma.sync m16n8k32
s8 x s8 -> s32) on this GPU, the second denominator for the expert FFN's
exact int8 contraction (the first is the fp16 tcgen05 rate: sm_103a has no
INT8 kind of tcgen05.mma).

The timed loop's accumulators must end at iters * 32 * a * b, so the number
printed comes from a loop that did its work.  Run with -s to see it:

    python -m pytest tests/test_gpu_mma_s8_rate.py -m gpu -s
"""
import ctypes
import os
import subprocess

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def rate_lib():
    out_dir = os.path.join(HERE, "_build")
    os.makedirs(out_dir, exist_ok=True)
    so = os.path.join(out_dir, "mma_s8_rate.so")
    subprocess.run([os.environ.get("NVCC", "nvcc"), "-O3", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
                    "-gencode", "arch=compute_103a,code=sm_103a",
                    os.path.join(HERE, "cuda", "mma_s8_rate.cu"), "-o", so], check=True)
    lib = ctypes.CDLL(so)
    lib.mma_s8_rate.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                ctypes.c_void_p, ctypes.POINTER(ctypes.c_float),
                                ctypes.POINTER(ctypes.c_double)]
    return lib


def test_mma_sync_s8_rate(rate_lib):
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    blocks, iters, a, b = 4 * sms, 8192, 3, -2
    out = torch.zeros(blocks * 256, dtype=torch.int32, device="cuda")
    ms, ops = ctypes.c_float(0), ctypes.c_double(0)
    assert rate_lib.mma_s8_rate(blocks, iters, 5, a, b, ctypes.c_void_p(out.data_ptr()),
                                ctypes.byref(ms), ctypes.byref(ops)) == 0
    want = iters * 32 * a * b
    assert bool((out == want).all()), f"accumulators differ from {want}"
    tops = ops.value / (ms.value / 1e3) / 1e12
    print(f"\nmma.sync m16n8k32 s8: {tops:.1f} TOPS ({blocks} blocks x 8 warps, {ms.value:.3f} ms per launch)")
    assert tops > 0
