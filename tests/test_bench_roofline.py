"""The bench's roofline object and traffic records (CPU).

* a committed ncu record is used only while its hash is the current decode sources' hash (else the bench
  line carries `traffic` null), and a used record is consistent (bytes, no re-reads);
* a record marked "alu" turns the roofline into the issue roofline (warp-instructions per second against
  the device's SMs x 4 schedulers x 1 per clock x its maximum SM clock) with the HBM figures alongside;
  without a record the roofline is the HBM one against the measured copy peak and `traffic` is null;
* the default run carries the second target workload; N ranks shard a global batch of N x B sequences;
* runs with a switch (value side, shapes, gate, bypass, meter off) never reuse the plain kernel's record.
"""
import argparse
import json
import os

import numpy as np
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
    # no device figures in the result: the GB300 fallback (or the measured maximum clock) is named
    assert r["peak"] == pytest.approx(152 * 4 * bench.max_sm_mhz(None)[0] * 1e6)
    assert "fallback" in r["peak_source"]
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"])
    assert r["traffic"] == 510_000_000
    assert r["hbm_achieved_gbs"] == 1000.0 and r["hbm_frac"] == pytest.approx(1000.0 / 6788.3)


def test_issue_peak_uses_the_device_sm_count_and_sampled_clock():
    w = bench.W.WORKLOADS["int8_7b_certified"]
    rec = {"bound": "alu", "warp_inst_per_launch": 600_000_000, "bytes_per_launch": 510_000_000}
    res = dict(_result(layer_ms=0.5, traffic=rec), sms=148, clocks={"sm_mhz": 1800.0, "sm_max_mhz": 1965.0})
    r = bench.roofline_of(res, w, _args())
    assert r["peak"] == pytest.approx(148 * 4 * 1965e6)
    assert "148 SMs (the device's SM count)" in r["peak_source"] and "clocks.max.sm" in r["peak_source"]


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


def _fake_run(w, traffic, e2e=True):
    per_step = bench.step_bytes(w, bench.W.seq_lengths(w))
    r = {"value": per_step / 5e-3 / 1e9, "ms_step": 5.0, "achieved": 6000.0, "graph": True, "layer_ms_mean": 0.14,
         "call_ms_mean": 0.15, "layer_ms_median": 0.14, "peak": 6788.3, "peak_kind": "measured", "traffic": traffic,
         "clocks": {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}, "launches": 3 * 36 * 10 + 10,
         "attended": 1.0e9, "per_step_bytes": per_step, "world": 1, "rank": 0, "counts": [0, 0, 0, 0],
         "resident": w.n_layers}
    if e2e:
        r["e2e"] = {"value": 0.97 * r["value"], "unit": "GB/s", "h2d_bytes_per_step": 123, "d2h_bytes_per_step": 45}
    return r


def test_bench_line_carries_the_contract_keys(monkeypatch):
    import sys

    monkeypatch.setattr(sys, "argv", ["bench.py", "--steps", "10", "--warmup", "3", "--no-cpu-baseline"])
    args = bench.parse()
    w = bench.W.WORKLOADS[args.workload]
    rec = bench.traffic_record(w.name)
    line = bench.bench_line(args, w, _fake_run(w, rec))
    json.dumps(line)   # serialisable
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "roofline", "clocks", "gpu_launches", "e2e"):
        assert k in line, k
    assert line["n_gpus"] == 1 and line["steps"] == 10 and line["warmup"] == 3 and line["higher_is_better"] is True
    assert line["scaling"] == "weak" and line["vs_baseline"] is None and line["data"] == "synthetic"
    assert line["config"]["workload"] == "qwen3_8b_cartridge" and "l2" in line["config"]
    ro = line["roofline"]
    for k in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert k in ro, k
    assert ro["frac"] == pytest.approx(ro["achieved"] / ro["peak"])
    assert ro["traffic"] == (rec["bytes_per_launch"] if rec else None)
    assert set(line["e2e"]) >= {"value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"}
    assert set(line["clocks"]) >= {"sm_mhz", "sm_max_mhz", "reasons"}
    assert line["gpu_launches"] > 0 and "note" not in line and "cpu_baseline" not in line


def test_bench_line_of_a_switch_and_a_profiling_run(monkeypatch):
    import sys

    monkeypatch.setattr(sys, "argv", ["bench.py", "--workload", "int8_7b_certified", "--int8-groups", "--layers", "2",
                                      "--no-cpu-baseline", "--no-e2e"])
    args = bench.parse()
    w = bench.W.reduced(bench.W.WORKLOADS["int8_7b_certified"], k_fmt="int8g32", v_fmt="int8g32")
    line = bench.bench_line(args, w, _fake_run(w, bench.traffic_record(w.name, variant=bench.runs_a_variant(args, w)),
                                               e2e=False))
    assert line["roofline"]["traffic"] is None and line["roofline"]["bound"] == "hbm"
    assert "not a bench line" in line["note"] and line["config"]["layout"] == "K int8g32 / V int8g32"


def test_cpu_baseline_object():
    w = bench.W.reduced(bench.W.WORKLOADS["tiny"], seq_len=256)
    cb = bench.cpu_baseline(w, budget_s=0.2)
    assert cb["kind"] == "oracle" and cb["unit"] == "GB/s" and cb["value"] > 0
    assert cb["cores"] == os.cpu_count() and cb["blas_threads"] >= 1
    assert "units of layer 0 at full context" in cb["sample"]


def test_default_run_carries_the_second_target_workload(monkeypatch):
    import sys

    monkeypatch.setattr(sys, "argv", ["bench.py", "--steps", "10", "--warmup", "3", "--no-cpu-baseline"])
    args = bench.parse()
    assert bench.times_second_workload(args)
    w2 = bench.W.WORKLOADS[bench.SECOND_WORKLOAD]
    rec = {"bound": "alu", "warp_inst_per_launch": 500_000_000, "bytes_per_launch": 2_456_000_000}
    obj = bench.second_object(args, w2, dict(_fake_run(w2, rec), sms=152))
    json.dumps(obj)
    for k in ("value", "unit", "ms_per_step", "roofline", "clocks", "e2e", "config"):
        assert k in obj, k
    assert obj["config"]["workload"] == "int8_7b_certified" and obj["config"]["meter"] == "tier A + tier B"
    assert obj["roofline"]["bound"] == "alu" and "hbm_frac" in obj["roofline"]
    # a switch, a profiling shape or another workload times only what was asked for
    for extra in (["--value-side"], ["--layers", "2"], ["--batch", "4"], ["--workload", "tiny"], ["--no-second"],
                  ["--eager"], ["--separate-append"]):
        monkeypatch.setattr(sys, "argv", ["bench.py", *extra])
        assert not bench.times_second_workload(bench.parse()), extra


@pytest.mark.parametrize("name", ["qwen3_8b_cartridge", "ragged_paged"])
def test_rank_shares_partition_the_global_batch(name):
    w = bench.W.WORKLOADS[name]
    w1, lens1, idx1 = bench.rank_share(w, 0, 1)
    assert w1 is w and np.array_equal(lens1, bench.W.seq_lengths(w)) and np.array_equal(idx1, np.arange(w.batch))
    for world in (2, 4):
        lens_g = bench.W.seq_lengths(bench.W.reduced(w, batch=w.batch * world))
        shares = [bench.rank_share(w, r, world) for r in range(world)]
        allidx = np.sort(np.concatenate([s[2] for s in shares]))
        assert np.array_equal(allidx, np.arange(w.batch * world))           # every sequence on exactly one rank
        for wr, lens, idx in shares:
            assert wr.batch == len(idx) and np.array_equal(lens, lens_g[idx])
        if name == "qwen3_8b_cartridge":
            assert all(s[0].batch == w.batch for s in shares)                # fixed lengths: equal shares
        cfg = bench.workload_config(w, world)
        assert cfg["batch"] == w.batch * world and cfg["batch_per_gpu"] == w.batch and "dp" in cfg["parallelism"]


def test_bench_line_cpu_baseline_branch(monkeypatch):
    import sys

    monkeypatch.setattr(sys, "argv", ["bench.py", "--value-side"])
    monkeypatch.setattr(bench, "cpu_baseline", lambda w: {"value": 0.03, "unit": "GB/s", "cores": 16, "kind": "oracle",
                                                          "sample": "s"})
    args = bench.parse()
    w = bench.W.WORKLOADS[args.workload]
    line = bench.bench_line(args, w, _fake_run(w, None))
    assert line["cpu_baseline"]["kind"] == "oracle" and "value side" in line["cpu_baseline"]["sample"]
    assert "value side" in line["config"]["meter"]
