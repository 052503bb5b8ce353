"""Device arithmetic of the library against its straightforward forms:

- the SiLU of the requantisation row kernel (branch-free, FMA-based division)
  against the IEEE-division form on every binary32 input, and both, with the
  exp behind them, against the oracle on a strided sample plus special values;
- the token-wise INT8 code of the dispatch and row kernels (the quotient
  from the reciprocal by Markstein's correction) against the IEEE-division
  form on 2^30 random (row absmax, value) pairs, half of them next to a
  half-integer quotient, and in groups of 16 on 2^26 rows."""
import ctypes
import os
import subprocess

import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(ROOT, "expert_dispatch_combine_gb300", "csrc")


@pytest.fixture(scope="module")
def helper():
    out_dir = os.path.join(HERE, "_build")
    os.makedirs(out_dir, exist_ok=True)
    so = os.path.join(out_dir, "device_math_check.so")
    subprocess.run([os.environ.get("NVCC", "nvcc"), "-O3", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
                    "-gencode", "arch=compute_103a,code=sm_103a", "-I", CSRC,
                    os.path.join(HERE, "cuda", "device_math_check.cu"), "-o", so], check=True)
    lib = ctypes.CDLL(so)
    P = ctypes.c_void_p
    lib.silu_check_all.argtypes = [ctypes.POINTER(ctypes.c_ulonglong), ctypes.POINTER(ctypes.c_uint)]
    lib.silu_eval.argtypes = [P, P, P, P, ctypes.c_int]
    U64P = ctypes.POINTER(ctypes.c_ulonglong)
    lib.quant_check.argtypes = [ctypes.c_ulonglong, U64P, U64P, ctypes.POINTER(ctypes.c_uint)]
    lib.quant_rows_check.argtypes = [ctypes.c_ulonglong, U64P, U64P, ctypes.POINTER(ctypes.c_uint)]
    return lib


def test_fast_silu_equals_ieee_division_form_on_all_inputs(helper):
    m = ctypes.c_ulonglong(0)
    first = ctypes.c_uint(0)
    assert helper.silu_check_all(ctypes.byref(m), ctypes.byref(first)) == 0
    assert m.value == 0, f"{m.value} mismatches, first at bit pattern {first.value:#010x}"


def test_device_silu_and_exp_match_oracle_sample(helper):
    bits = np.arange(0, 1 << 32, 16381, dtype=np.uint64).astype(np.uint32)
    specials = np.array([0.0, -0.0, 1.0, -1.0, 87.0, -87.0, 88.0, -88.0, 88.5, -88.5, 44.36, -44.36,
                         1e-45, -1e-45, 3e38, -3e38, np.inf, -np.inf], dtype=np.float32).view(np.uint32)
    bits = np.concatenate([bits, specials])
    x = bits.view(np.float32)
    n = len(x)
    spec = np.empty(n, np.float32)
    fast = np.empty(n, np.float32)
    ex = np.empty(n, np.float32)
    ptr = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    assert helper.silu_eval(ptr(x), ptr(spec), ptr(fast), ptr(ex), n) == 0
    ref_s = np.array([oracle.silu(v) for v in x], dtype=np.float32)
    ref_e = np.array([oracle.exp_spec(v) for v in x], dtype=np.float32)

    def same(a, b):
        return (a.view(np.uint32) == b.view(np.uint32)) | (np.isnan(a) & np.isnan(b))

    assert same(spec, ref_s).all()
    assert same(fast, ref_s).all()
    assert same(ex, ref_e).all()


def test_reciprocal_quantisation_equals_division_form(helper):
    m = ctypes.c_ulonglong(0)
    nh = ctypes.c_ulonglong(0)
    first = ctypes.c_uint(0)
    n = 1 << 30
    assert helper.quant_check(n, ctypes.byref(m), ctypes.byref(nh), ctypes.byref(first)) == 0
    assert nh.value > n // 4  # the near-half-integer draws happened
    assert m.value == 0, f"{m.value} mismatches, first at draw {first.value}"


def test_group_quantisation_equals_division_form(helper):
    """The 16-value group form of the row kernels (the correctly rounded
    quotient from the reciprocal by Markstein's correction, no division and no
    branch per value) on 2^26 rows of 16 values, most of them holding a value
    next to a half-integer quotient."""
    n = 1 << 26
    m, nr = ctypes.c_ulonglong(0), ctypes.c_ulonglong(0)
    first = ctypes.c_uint(0)
    assert helper.quant_rows_check(n, ctypes.byref(m), ctypes.byref(nr), ctypes.byref(first)) == 0
    assert nr.value > n // 2  # most rows hold a value next to a half-integer quotient
    assert m.value == 0, f"{m.value} rows differ, first at row {first.value}"
