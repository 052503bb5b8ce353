"""Seeded synthetic inputs for the MoE layer workloads.

This module holds no arithmetic of the method itself: it only draws inputs
(gate logits, hidden states, INT8 expert weights and their scales) and is the
one piece shared by the CUDA path's tests/benchmark and by the CPU oracle.

Workloads (DeepSeek-V3/R1 MoE-layer shapes):
  c0_tiny        T=64,    H=256,  E=16,        k=2, I=128,  4 ranks
  c1_decode      T=96,    H=7168, E=256,       k=8, I=2048, 32 ranks
  c2_decode_zipf T=12288, H=7168, E=256,       k=8, I=2048, 32 ranks, Zipf 1.1
  c3_eplb        T=4608,  H=7168, E=256(+32),  k=8, I=2048, 32 ranks, Zipf 1.2
  c4_prefill     T=16384, H=7168, E=256,       k=8, I=2048, 32 ranks

Recipe:
  logits  N(0,1) binary32 (numpy PCG64 stream [seed, 1]); skewed workloads
          add -s*ln(pi(e)+1) with pi a seeded permutation (stream [seed, 2]);
  hidden  N(0,1) binary32 (stream [seed, 3]) rounded to bfloat16 (RNE);
  weights int8 uniform on [-127, 127] from a counter hash (below), so that
          the same values can be drawn on the host or directly on the GPU;
  scales  U[0.5, 1.5) / (127 sqrt(fan_in)) binary32 (stream [seed, 1000+e]),
          fan_in = H for gate/up, I for down.

Counter hash for weights: for 32-bit words,
  mix(x) = x ^= x>>16; x = (x * 0x7FEB352D) mod 2^32; x ^= x>>15;
           x = (x * 0x1B873593) mod 2^32; x ^= x>>16
  key(seed, e, tensor) = mix(mix(seed + 0x68E31DA4) ^ (4*e + tensor + 1))
  w[i] = (mix((key + i * 0x9E3779B9) mod 2^32) mod 255) - 127,
  i = flat element index (< 2^31).
Both mix multipliers are below 2^31 and i * 0x9E3779B9 < 2^63, so every
intermediate fits in a signed 64-bit integer and the same code runs exactly
in numpy and torch.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

M32 = 0xFFFFFFFF


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    E_log: int
    E_phys: int
    k: int
    I: int
    R: int
    S: int
    seed: int
    zipf: float = 0.0
    eplb: bool = False
    plan_ranks: int = 0  # ranks the replica planner places over (0: R)
    msg_formats: bool = False  # also time dispatch/combine alone with bf16 and INT8 messages

    @property
    def placement_ranks(self) -> int:
        return self.plan_ranks or self.R

    @property
    def lb(self) -> int:
        return self.T // self.S

    @property
    def epr(self) -> int:
        return self.E_phys // self.R

    @property
    def mt(self) -> int:
        return self.lb * min(self.k, self.epr)


WORKLOADS = {
    "c0_tiny": Workload("c0_tiny", 64, 256, 16, 16, 2, 128, 4, 4, 0),
    "c1_decode": Workload("c1_decode", 96, 7168, 256, 256, 8, 2048, 32, 32, 1),
    "c2_decode_zipf": Workload("c2_decode_zipf", 12288, 7168, 256, 256, 8, 2048, 32, 32, 2, zipf=1.1),
    "c3_eplb": Workload("c3_eplb", 4608, 7168, 256, 288, 8, 2048, 32, 32, 3, zipf=1.2, eplb=True),
    "c4_prefill": Workload("c4_prefill", 16384, 7168, 256, 256, 8, 2048, 32, 32, 4, msg_formats=True),
    # profiling case: the DeepSeek-V3 expert shape with 32 experts (1.4 GB of
    # weights, about 3.5 GB on the device in total) and 1024 rows per expert
    "prof_e32": Workload("prof_e32", 4096, 7168, 32, 32, 8, 2048, 32, 32, 5),
    # profiling case of the decode matrix-vector path: the same expert shape,
    # 32 experts (1.4 GB of weights), 16 tokens x top-8 = 4 rows per expert
    "prof_decode_e32": Workload("prof_decode_e32", 16, 7168, 32, 32, 8, 2048, 32, 16, 6),
    # trampoline forward ("xDeepServe", P044-P047): one DP domain of 160
    # attention ranks x 96 tokens (the pages' global batch 46,080 is three such
    # domains) sent to 288 expert ranks, one physical expert each (256 routed
    # experts + 32 redundant copies, placed over 32 groups of 9 slots)
    "tr_domain": Workload("tr_domain", 15360, 7168, 256, 288, 8, 2048, 288, 160, 10, zipf=1.2,
                          eplb=True, plan_ranks=32),
}


def custom(name="custom", T=64, H=256, E_log=16, E_phys=None, k=2, I=128, R=4, S=None,
           seed=0, zipf=0.0, eplb=False, plan_ranks=0) -> Workload:
    return Workload(name, T, H, E_log, E_phys if E_phys else E_log, k, I, R,
                    S if S else R, seed, zipf, eplb, plan_ranks)


# ------------------------------------------------------------------ floats
def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """binary32 -> bfloat16 bit patterns, round to nearest even (finite input)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def zipf_bias(w: Workload) -> np.ndarray:
    if w.zipf == 0.0:
        return np.zeros(w.E_log, np.float64)
    perm = np.random.default_rng([w.seed, 2]).permutation(w.E_log)
    return -w.zipf * np.log(perm.astype(np.float64) + 1.0)


def logits(w: Workload, rows: slice | None = None) -> np.ndarray:
    z = np.random.default_rng([w.seed, 1]).standard_normal((w.T, w.E_log), dtype=np.float32)
    out = (z.astype(np.float64) + zipf_bias(w)[None, :]).astype(np.float32)
    return out if rows is None else np.ascontiguousarray(out[rows])


def hidden_bits(w: Workload) -> np.ndarray:
    """uint16 [T, H] bf16 bit patterns."""
    z = np.random.default_rng([w.seed, 3]).standard_normal((w.T, w.H), dtype=np.float32)
    return f32_to_bf16_bits(z)


# ------------------------------------------------------------- int weights
def _mix_np(x: np.ndarray) -> np.ndarray:
    x = x ^ (x >> 16)
    x = (x * 0x7FEB352D) & M32
    x = x ^ (x >> 15)
    x = (x * 0x1B873593) & M32
    x = x ^ (x >> 16)
    return x


def _key(seed: int, e: int, tensor: int) -> int:
    k0 = int(_mix_np(np.array([(seed + 0x68E31DA4) & M32], np.int64))[0])
    return int(_mix_np(np.array([k0 ^ ((4 * e + tensor + 1) & M32)], np.int64))[0])


def _mix_u32(x: np.ndarray) -> np.ndarray:
    """mix() on a uint32 array, in place (uint32 products wrap mod 2^32)."""
    x ^= x >> np.uint32(16)
    x *= np.uint32(0x7FEB352D)
    x ^= x >> np.uint32(15)
    x *= np.uint32(0x1B873593)
    x ^= x >> np.uint32(16)
    return x


def int8_tensor_np(seed: int, e: int, tensor: int, shape) -> np.ndarray:
    """Host draw of one int8 weight tensor (threaded over chunks)."""
    import concurrent.futures
    import os

    n = int(np.prod(shape))
    key = np.uint32(_key(seed, e, tensor))
    out = np.empty(n, np.int8)
    step = 1 << 21

    def work(st):
        m = min(step, n - st)
        i = np.arange(st, st + m, dtype=np.uint32)
        i *= np.uint32(0x9E3779B9)
        i += key
        v = _mix_u32(i)
        v %= np.uint32(255)
        out[st:st + m] = (v.astype(np.int16) - 127).astype(np.int8)

    starts = range(0, n, step)
    if n <= step:
        for st in starts:
            work(st)
    else:
        with concurrent.futures.ThreadPoolExecutor(min(32, os.cpu_count() or 1)) as ex:
            list(ex.map(work, starts))
    return out.reshape(shape)


def int8_tensor_torch(seed: int, e: int, tensor: int, shape, device="cpu", out=None):
    """Same values as int8_tensor_np, computed with torch on any device.
    If `out` (int8, contiguous, numel == prod(shape)) is given it is filled in
    chunks to bound temporary memory."""
    import torch

    n = int(np.prod(shape))
    key = _key(seed, e, tensor)

    def mix(x):
        x = x ^ (x >> 16)
        x = (x * 0x7FEB352D) & M32
        x = x ^ (x >> 15)
        x = (x * 0x1B873593) & M32
        x = x ^ (x >> 16)
        return x

    if out is None:
        out = torch.empty(n, dtype=torch.int8, device=device)
    flat = out.view(-1)
    step = 1 << 24
    for s in range(0, n, step):
        m = min(step, n - s)
        i = torch.arange(s, s + m, dtype=torch.int64, device=flat.device)
        v = mix((i * 0x9E3779B9 + key) & M32) % 255 - 127
        flat[s:s + m] = v.to(torch.int8)
    return out.view(*shape)


GATE_UP, DOWN = 0, 1


def expert_scales(w: Workload, e: int) -> tuple[np.ndarray, np.ndarray]:
    rng = np.random.default_rng([w.seed, 1000 + e])
    s_gu = (rng.uniform(0.5, 1.5, 2 * w.I) / (127.0 * math.sqrt(w.H))).astype(np.float32)
    s_d = (rng.uniform(0.5, 1.5, w.H) / (127.0 * math.sqrt(w.I))).astype(np.float32)
    return s_gu, s_d


def expert_weights_np(w: Workload, e: int):
    """(w_gu int8 [2I, H], s_gu f32 [2I], w_d int8 [H, I], s_d f32 [H]) of logical expert e."""
    s_gu, s_d = expert_scales(w, e)
    return (int8_tensor_np(w.seed, e, GATE_UP, (2 * w.I, w.H)), s_gu,
            int8_tensor_np(w.seed, e, DOWN, (w.H, w.I)), s_d)


def all_weights_torch(w: Workload, device="cuda"):
    """All logical experts' weights on `device`:
    (w_gu int8 [E, 2I, H], s_gu f32 [E, 2I], w_d int8 [E, H, I], s_d f32 [E, H])."""
    import torch

    E = w.E_log
    w_gu = torch.empty((E, 2 * w.I, w.H), dtype=torch.int8, device=device)
    w_d = torch.empty((E, w.H, w.I), dtype=torch.int8, device=device)
    s_gu = np.empty((E, 2 * w.I), np.float32)
    s_d = np.empty((E, w.H), np.float32)
    for e in range(E):
        int8_tensor_torch(w.seed, e, GATE_UP, (2 * w.I, w.H), out=w_gu[e])
        int8_tensor_torch(w.seed, e, DOWN, (w.H, w.I), out=w_d[e])
        s_gu[e], s_d[e] = expert_scales(w, e)
    return (w_gu, torch.from_numpy(s_gu).to(device), w_d, torch.from_numpy(s_d).to(device))
