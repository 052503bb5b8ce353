"""Failure detection without a GPU fault: the bounded mbarrier wait that
every wait of the tensor-core GEMM uses gives up after its limit on a barrier
nothing arrives on, records MOE_ERR_TIMEOUT in the status word and returns;
when another thread has already posted an error it gives up at once and
leaves that error in place.  The kernel ends normally in both cases."""
import ctypes
import os
import subprocess

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
PKG = os.path.join(ROOT, "expert_dispatch_combine_gb300", "csrc")
MOE_ERR_TIMEOUT = 5


@pytest.fixture(scope="module")
def helper():
    out_dir = os.path.join(HERE, "_build")
    os.makedirs(out_dir, exist_ok=True)
    so = os.path.join(out_dir, "wait_check.so")
    subprocess.run([os.environ.get("NVCC", "nvcc"), "-O3", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
                    "-gencode", "arch=compute_103a,code=sm_103a", "-I", PKG, "-I",
                    os.path.join(ROOT, "include"), os.path.join(HERE, "cuda", "wait_check.cu"),
                    "-o", so, "-lcuda"], check=True)
    lib = ctypes.CDLL(so)
    lib.wait_check.argtypes = [ctypes.c_ulonglong, ctypes.c_int, ctypes.c_void_p]
    return lib


def _run(helper, limit_ns, preset):
    out = (ctypes.c_longlong * 3)()
    assert helper.wait_check(limit_ns, preset, ctypes.cast(out, ctypes.c_void_p)) == 0
    return int(out[0]), int(out[1]), int(out[2])


def test_wait_times_out_and_records_status(helper):
    ok, status, ns = _run(helper, 1_000_000, 0)  # 1 ms limit
    assert ok == 0
    assert status == MOE_ERR_TIMEOUT
    assert 1_000_000 <= ns < 1_000_000_000


def test_wait_gives_up_on_posted_error(helper):
    ok, status, ns = _run(helper, 1_000_000_000, 3)  # 1 s limit, error already posted
    assert ok == 0
    assert status == 3  # left as posted
    assert ns < 100_000_000


# ------------------------------------------------ the combine's bounded wait
def test_combine_wait_runs_out_without_fault():
    """moe_expert_ffn_combine_ex with a target no token can reach (k + 1
    messages): the first token's wait runs out after its bound (20 ms), posts
    MOE_ERR_TIMEOUT and the other waits give up at once; the kernel ends, the
    return messages are still written (rows never wait), no token is combined,
    and the next call on the same context succeeds with status 0."""
    import time

    import numpy as np
    import torch

    from expert_dispatch_combine_gb300 import binding as B
    from expert_dispatch_combine_gb300 import synth

    import gpu_util

    gpu_util.lib()
    w = synth.WORKLOADS["c0_tiny"]
    layer = gpu_util.make_layer(w)
    lg = torch.from_numpy(synth.logits(w)).cuda()
    x = gpu_util.bits_to_bf16_tensor(synth.hidden_bits(w))
    ref = layer.forward(lg, x).clone()
    ref_rows = layer.buf.combine_rows().clone()
    b, r, s = layer.buf, layer.buf.routing, layer.shape
    w_gu, s_gu, w_d, s_d = layer.w
    sentinel = torch.full_like(ref, 7.0)
    out = sentinel.clone()
    b.combine.zero_()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    B.moe_expert_ffn_combine_ex(s, b.dispatch, r["expert_offsets"], r["expert_rows"], w_gu, s_gu,
                                w_d, s_d, r["topk_w"], b.combine, out, b.workspace,
                                expected=w.k + 1, wait_ns=20_000_000)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert B.moe_device_status(b.workspace) == MOE_ERR_TIMEOUT
    assert dt < 10.0
    assert torch.equal(b.combine_rows(), ref_rows)   # every return message was written
    assert torch.equal(out, sentinel)                # no token was combined
    b.check()
    # the context is intact: the same call with the right target completes normally
    B.moe_expert_ffn_combine_ex(s, b.dispatch, r["expert_offsets"], r["expert_rows"], w_gu, s_gu,
                                w_d, s_d, r["topk_w"], b.combine, out, b.workspace,
                                expected=w.k, wait_ns=2_000_000_000)
    torch.cuda.synchronize()
    assert B.moe_device_status(b.workspace) == 0
    assert torch.equal(out, ref)
