"""Host logic of bench.py (no GPU): the DRAM-traffic figure is only reported
when the committed ncu summary was taken on the current kernel source, the
message byte counts of the two bookkeeping helpers agree, and both arms'
`config` objects carry the same keys."""
import hashlib
import os
import shutil

import pytest

import bench
from expert_dispatch_combine_gb300 import synth


@pytest.mark.parametrize("kind", sorted(bench.TRAFFIC_PROFILES))
def test_traffic_scales_the_committed_ratio(kind):
    name, src = bench.TRAFFIC_PROFILES[kind]
    txt = open(os.path.join(bench.ROOT, "profiles", name)).read()
    kv = dict(l.split(":", 1) for l in txt.splitlines()
              if l.startswith(("source_sha1:", "traffic_bytes_per_launch:", "algorithmic_bytes_per_launch:")))
    src_sha = hashlib.sha1(open(src, "rb").read()).hexdigest()
    got = bench.measured_traffic(10 ** 9, kind)
    if kv["source_sha1"].strip() != src_sha:
        assert got is None  # a summary of another kernel source is never used
        return
    ratio = int(kv["traffic_bytes_per_launch"]) / int(kv["algorithmic_bytes_per_launch"])
    assert got == int(round(ratio * 10 ** 9))
    assert 0.5 < ratio < 2.0


def test_traffic_is_null_for_a_changed_source(tmp_path, monkeypatch):
    name, src = bench.TRAFFIC_PROFILES["tc_f16"]
    changed = tmp_path / "ffn_tc.cu"
    shutil.copy(src, changed)
    with open(changed, "a") as f:
        f.write("\n// changed\n")
    monkeypatch.setitem(bench.TRAFFIC_PROFILES, "tc_f16", (name, str(changed)))
    assert bench.measured_traffic(10 ** 9, "tc_f16") is None


def test_traffic_is_null_without_a_summary(monkeypatch):
    _, src = bench.TRAFFIC_PROFILES["tc"]
    monkeypatch.setitem(bench.TRAFFIC_PROFILES, "tc", ("no_such_summary.md", src))
    assert bench.measured_traffic(10 ** 9, "tc") is None


@pytest.mark.parametrize("name", ["c1_decode", "c2_decode_zipf", "c4_prefill"])
def test_int8_message_bytes_agree(name):
    """The layer's dispatch/combine bytes (INT8 messages) and the standalone
    message-format bookkeeping count the same bytes; bf16 rows add H bytes
    per message and drop the 4-byte scale of the combine."""
    w = synth.WORKLOADS[name]
    alg = bench.algorithmic(w)
    d8, c8 = bench.message_bytes(w, bf16=False)
    d16, c16 = bench.message_bytes(w, bf16=True)
    assert (d8, c8) == (alg["dispatch_bytes"], alg["combine_bytes"])
    m = w.T * w.k
    assert d16 - d8 == m * w.H
    assert c16 - c8 == m * w.H - m * 4
    assert alg["ffn_ops"] == alg["gate_up_ops"] + alg["down_ops"] == m * 6 * w.H * w.I


def test_config_keys_and_l2_statement():
    big = bench.config_of(synth.WORKLOADS["c2_decode_zipf"], 1)
    small = bench.config_of(synth.WORKLOADS["c0_tiny"], 1)
    ref = bench.config_of(synth.WORKLOADS["c2_decode_zipf"], 1, weights="int8")
    assert set(big) == set(small) == set(ref)
    assert big["workload"] == "c2_decode_zipf" and big["parallelism"] == "replicas x1"
    assert big["l2"].startswith("inputs larger than L2")
    assert small["l2"].startswith("inputs fit in L2")


def test_single_replica_aggregate():
    ms, value = bench.replica_aggregate(8.0, 12288, 1)
    assert ms == 8.0
    assert value == pytest.approx(12288 / 0.008)
