"""Pins of the oracle's binary32 scale steps inside one expert row.

The expert FFN scales each exact integer contraction by the token's scale and
by the output channel's weight scale ("xDeepServe on CloudMatrix384", section
"DeepSeek INT8 量化", P085 equation y_ij ~ s_i s^w_j sum_k q(x_ik) q(w_jk)):

    g_i = (acc_g[i] * xs) * sg[i]      gate channel i   (weight row i)
    u_i = (acc_u[i] * xs) * su[i]      up channel i     (weight row I + i, P088)
    y_c = (acc_d[c] * s_h) * sd[c]     down channel c   (s_h: token scale of h)

Two pins, each with distinct per-channel scales:
  * a hand-worked row (tests/golden/expert_scale_steps.txt) in which every
    scale is a power of two and every gate sits where SiLU is exact, so each
    intermediate value is exact and was derived by hand;
  * a float64 closed form on random rows and scales, within the binary32
    roundings of each step.
A third test plants, one at a time, the mistakes these pins exist to catch
(up channel scaled by the gate's scale, gate and up scales swapped, down
scales mis-indexed, token scale or s_h dropped) in compiled copies of the
oracle and checks that each copy fails a pin.
"""
import math
import os
import subprocess

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "expert_scale_steps.txt")


def _golden():
    kv = {}
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, val = (s.strip() for s in line.split("=", 1))
        kv[key] = [float(v) for v in val.split()]
    H, I = len(kv["xq"]), len(kv["hq"])
    g = dict(
        xq=np.array(kv["xq"], np.int8), xs=np.float32(kv["xs"][0]),
        w_gu=np.array([kv[f"w_gu_row{r}"] for r in range(2 * I)], np.int8),
        s_gu=np.array(kv["s_gu"], np.float32),
        w_d=np.array([kv[f"w_d_row{c}"] for c in range(H)], np.int8),
        s_d=np.array(kv["s_d"], np.float32),
        acc_gu=np.array(kv["acc_gu"], np.int64), s_h=np.float32(kv["s_h"][0]),
        hq=np.array(kv["hq"], np.int64), acc_d=np.array(kv["acc_d"], np.int64),
        y=np.array(kv["y"], np.float32), msg_scale=np.float32(kv["msg_scale"][0]),
        msg_codes=np.array(kv["msg_codes"], np.int64))
    assert g["w_gu"].shape == (2 * I, H) and g["w_d"].shape == (H, I)
    return g


def check_hand_worked(expert_row):
    g = _golden()
    msg, sc, dbg = expert_row(g["xq"], g["xs"], g["w_gu"], g["s_gu"], g["w_d"], g["s_d"],
                              cfmt=1, debug=True)
    assert (dbg["acc_gu"] == g["acc_gu"]).all()
    assert dbg["sh"] == g["s_h"], (dbg["sh"], g["s_h"])
    assert (dbg["hq"] == g["hq"]).all(), dbg["hq"]
    assert (dbg["acc_d"] == g["acc_d"]).all(), dbg["acc_d"]
    assert (dbg["y"] == g["y"]).all(), dbg["y"]
    assert sc == g["msg_scale"], sc
    assert (msg.astype(np.int64) == g["msg_codes"]).all(), msg
    # bf16 return message: every y of the row is exact in bf16
    msg16, _ = expert_row(g["xq"], g["xs"], g["w_gu"], g["s_gu"], g["w_d"], g["s_d"], cfmt=0)
    y_bits = (g["y"].view(np.uint32) >> 16).astype(np.uint16)
    assert (g["y"].view(np.uint32) & 0xFFFF == 0).all()
    assert (msg16 == y_bits).all()


def _closed_form_case(seed):
    """A random row: codes, token scale and per-channel scales drawn so that the
    SwiGLU gates span SiLU's nonlinear range."""
    rng = np.random.default_rng(seed)
    H, I = 96, 40
    xq = rng.integers(-127, 128, H).astype(np.int8)
    xs = np.float32(rng.uniform(0.5, 2.0) * 2.0 ** rng.integers(-8, -3))
    w_gu = rng.integers(-127, 128, (2 * I, H)).astype(np.int8)
    w_d = rng.integers(-127, 128, (H, I)).astype(np.int8)
    s_gu = (rng.uniform(0.05, 4.0, 2 * I) / (127 * math.sqrt(H))).astype(np.float32)
    s_d = (rng.uniform(0.05, 4.0, H) / (127 * math.sqrt(I))).astype(np.float32)
    return xq, xs, w_gu, s_gu, w_d, s_d


def check_closed_form(expert_row, seeds=range(6)):
    """Float64 closed form of every scale step.  Tolerances: g and u carry two
    binary32 roundings, SiLU a few more (exp within 2 ulp, one add, one
    divide), h one; s_h = absmax/127 then agrees within 16 ulp.  y carries two
    roundings of exact operands (acc_d is exact, s_h is the oracle's own)."""
    eps = 2.0 ** -24
    for seed in seeds:
        xq, xs, w_gu, s_gu, w_d, s_d = _closed_form_case(seed)
        I = w_d.shape[1]
        _, _, dbg = expert_row(xq, xs, w_gu, s_gu, w_d, s_d, cfmt=1, debug=True)
        acc = w_gu.astype(np.int64) @ xq.astype(np.int64)
        assert (dbg["acc_gu"] == acc).all()
        g = acc[:I] * float(xs) * s_gu[:I].astype(np.float64)
        u = acc[I:] * float(xs) * s_gu[I:].astype(np.float64)
        h = g / (1.0 + np.exp(-g)) * u
        sh_ref = np.abs(h).max() / 127.0
        assert abs(float(dbg["sh"]) - sh_ref) <= 16 * eps * sh_ref, (seed, dbg["sh"], sh_ref)
        codes_ref = h / sh_ref
        diff = np.abs(dbg["hq"].astype(np.float64) - codes_ref)
        assert diff.max() <= 0.5 + 1e-3, (seed, diff.max())
        # the codes equal round(h / s_h) except within a few ulp of a half-integer
        near_tie = np.abs(np.abs(codes_ref - np.floor(codes_ref)) - 0.5) < 1e-4
        assert (dbg["hq"] == np.rint(codes_ref))[~near_tie].all(), seed
        acc_d = w_d.astype(np.int64) @ dbg["hq"].astype(np.int64)
        assert (dbg["acc_d"] == acc_d).all()
        y_ref = acc_d * float(dbg["sh"]) * s_d.astype(np.float64)
        err = np.abs(dbg["y"].astype(np.float64) - y_ref)
        assert (err <= 2.0 * eps * np.abs(y_ref) + 1e-45).all(), (seed, (err / np.abs(y_ref)).max())


def test_expert_scale_steps_hand_worked():
    check_hand_worked(oracle.expert_row)


def test_expert_scale_steps_closed_form():
    check_closed_form(oracle.expert_row)


# ---------------------------------------------- planted mistakes must fail
_SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "oracle", "moe_oracle.c")

MUTANTS = {
    # the up channel scaled by its gate channel's scale (wrong row index)
    "up_uses_gate_scale": [("u = u * s_gu[I + i];", "u = u * s_gu[i];")],
    # gate and up scales swapped
    "gate_up_scales_swapped": [("g = g * s_gu[i];", "g = g * s_gu[I + i];"),
                               ("u = u * s_gu[I + i];", "u = u * s_gu[i];")],
    # down scale of the wrong output channel
    "down_scale_shifted": [("v = v * s_d[c];", "v = v * s_d[(c + 1) % H];")],
    "down_scale_first": [("v = v * s_d[c];", "v = v * s_d[0];")],
    # token scale dropped from the gate, from both projections, or s_h dropped
    "gate_token_scale_dropped": [("g = g * xs;", "g = g * 1.0f;")],
    "token_scale_dropped": [("g = g * xs;", "g = g * 1.0f;"), ("u = u * xs;", "u = u * 1.0f;")],
    "h_scale_dropped": [("v = v * sh;", "v = v * 1.0f;")],
}


def _build_mutant(name, edits, tmpdir):
    src = open(_SRC).read()
    for old, new in edits:
        assert src.count(old) == 1, (name, old)
        src = src.replace(old, new)
    c = os.path.join(tmpdir, f"mut_{name}.c")
    so = os.path.join(tmpdir, f"libmut_{name}.so")
    open(c, "w").write(src)
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                    "-fno-fast-math", "-o", so, c, "-lm"], check=True)
    return oracle.load_library(so)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_scale_mistakes_fail_a_pin(name, tmp_path):
    lib = _build_mutant(name, MUTANTS[name], str(tmp_path))

    def row(*a, **kw):
        return oracle.expert_row(*a, lib=lib, **kw)

    failed = []
    for check in (check_hand_worked, check_closed_form):
        try:
            check(row)
        except AssertionError:
            failed.append(check.__name__)
    assert failed, f"planted mistake {name!r} passed every scale pin"
