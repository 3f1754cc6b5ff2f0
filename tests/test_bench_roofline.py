"""The bench's roofline object and traffic records (CPU).

* a committed ncu record is used only while its hash is the current decode sources' hash (else the bench
  line carries `traffic` null), and a used record is consistent (bytes, no re-reads);
* a record marked "alu" turns the roofline into the issue roofline (warp-instructions per second against
  152 SMs x 4 schedulers x 1 per clock x 2070 MHz) with the HBM figures alongside; without a record the
  roofline is the HBM one against the measured copy peak and `traffic` is null;
* runs with a switch (value side, shapes, gate, bypass, meter off) never reuse the plain kernel's record.
"""
import argparse
import json
import os

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _result(layer_ms=0.5, traffic=None):
    return {"traffic": traffic, "layer_ms_mean": layer_ms, "achieved": 1000.0, "peak": 6788.3, "peak_kind": "measured",
            "per_step_bytes": 28 * 500_000_000, "call_ms_mean": 0.51}


def _args():
    return argparse.Namespace(layers=0)


def test_committed_records_are_used_only_for_the_sources_they_describe():
    with open(os.path.join(ROOT, "profiles", "decode_traffic.json")) as f:
        recs = json.load(f)
    h = bench.kernel_hash()
    for name in ("qwen3_8b_cartridge", "int8_7b_certified"):
        rec = bench.traffic_record(name)
        if recs[name]["kernel_hash"] != h:
            assert rec is None, name     # counters of an older kernel: the bench line carries traffic null
            continue
        assert rec is not None
        assert rec["bytes_per_launch"] == rec["dram_bytes_read"] + rec["dram_bytes_write"]
        # no re-reads: DRAM reads within 1 % of the algorithmic bytes
        assert abs(rec["dram_bytes_read"] / rec["algorithmic_bytes_per_launch"] - 1) < 0.01
    assert recs["int8_7b_certified"]["bound"] == "alu"


def test_switches_never_reuse_the_plain_record():
    assert bench.traffic_record("qwen3_8b_cartridge", variant=True) is None


def test_hbm_roofline_without_a_record():
    w = bench.W.WORKLOADS["int8_7b_certified"]
    r = bench.roofline_of(_result(), w, _args())
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["traffic"] is None
    assert r["frac"] == pytest.approx(1000.0 / 6788.3)
    assert r["algorithmic_bytes_per_launch"] == 500_000_000


def test_issue_roofline_with_an_alu_record():
    w = bench.W.WORKLOADS["int8_7b_certified"]
    rec = {"bound": "alu", "warp_inst_per_launch": 600_000_000, "bytes_per_launch": 510_000_000}
    r = bench.roofline_of(_result(layer_ms=0.5, traffic=rec), w, _args())
    assert r["bound"] == "alu" and r["unit"] == "warp-instructions/s"
    assert r["achieved"] == pytest.approx(600_000_000 / 0.5e-3)
    assert r["peak"] == pytest.approx(152 * 4 * 2070e6)
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"])
    assert r["traffic"] == 510_000_000
    assert r["hbm_achieved_gbs"] == 1000.0 and r["hbm_frac"] == pytest.approx(1000.0 / 6788.3)


def test_every_switch_counts_as_a_variant():
    base = dict(value_side=False, shapes=False, gate=False, meter_off=False, int8_groups=False)
    w = bench.W.WORKLOADS["qwen3_8b_cartridge"]
    assert not bench.runs_a_variant(argparse.Namespace(**base), w)
    for k in base:
        assert bench.runs_a_variant(argparse.Namespace(**{**base, k: True}), w), k
    # the --bypass switch turns the INT8 workload into one with a fixed-channel key bypass
    x = bench.W.reduced(bench.W.WORKLOADS["int8_7b_certified"], massive_pairs=4, massive_scale=30.0, bypass_pairs=4)
    assert bench.runs_a_variant(argparse.Namespace(**base), x)


def test_kernel_fingerprint_ignores_comments_only():
    code = "int f(int x) {\n  return x + 1;  // one\n}\n"
    assert bench.code_only(code) == bench.code_only("/* header\n spanning lines */\n" + code.replace("// one", "// two"))
    assert bench.code_only(code) == bench.code_only(code.replace("\n}", "\n\n   \n}"))
    assert bench.code_only(code) != bench.code_only(code.replace("x + 1", "x + 2"))
    texts = {f: open(os.path.join(ROOT, f), encoding="utf-8").read() for f in bench.KERNEL_SOURCES}
    assert bench.kernel_hash(lambda f: texts[f]) == bench.kernel_hash()
    f0 = bench.KERNEL_SOURCES[0]
    edited = dict(texts, **{f0: texts[f0] + "\n// a trailing comment\n"})
    assert bench.kernel_hash(lambda f: edited[f]) == bench.kernel_hash()
    edited = dict(texts, **{f0: texts[f0] + "\nstatic int kvq_unused_probe;\n"})
    assert bench.kernel_hash(lambda f: edited[f]) != bench.kernel_hash()
