"""GPU parity of the alternative bound shapes (WitCert Sec. 4.3 Proposition 1; det-tanh) via the C ABI.

With KVQ_TIER_S the decode also keeps, per (sequence, query head), the largest Tier A radius max_t c_t
(merged over the splits by max) and 1 - A^- = sum_t p~_t (1 - e^{-c_t}) (merged with the softmax
weights, like A); kvq_meter turns them into the two-sided meter min(meter, 1/2 (A/A^- - A^-/A)) and the
det-tanh bound tanh(max_t c_t).  Bars: max radius and 1 - A^- within 1e-4 relative of the oracle, both
bounds within 1e-4 relative and never below the exact TV, and nothing else changes.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import workloads as W  # noqa: E402
from tests.parity import make_inputs, reference_case, run_case_gpu  # noqa: E402

CASES = {
    "tiny": lambda: W.reduced(W.WORKLOADS["tiny"], seq_len=300),
    "cartridge": lambda: W.reduced(W.WORKLOADS["qwen3_8b_cartridge"], batch=2, seq_len=150),
    "int8": lambda: W.reduced(W.WORKLOADS["int8_7b_certified"], batch=2, seq_len=333),
    "fp8raw": lambda: W.reduced(W.WORKLOADS["fp8_raw_stress"], batch=2, seq_len=200),
    "ragged": lambda: W.reduced(W.WORKLOADS["ragged_paged"], batch=4, ragged=(40, 700)),
}


@pytest.fixture(scope="module")
def kvq():
    import quantized_kv_cache_kvq_gb300 as m

    m.load()
    return m


def _rel(a, b):
    return np.abs(a - b) / np.maximum(np.abs(b), 1e-30)


@pytest.mark.parametrize("name", list(CASES))
def test_shapes_parity_and_soundness(kvq, name):
    w = CASES[name]()
    inp = make_inputs(w)
    ref = reference_case(w, inputs=inp)
    value = name == "cartridge"  # the value side and the shapes together in one case
    gpu = run_case_gpu(w, inputs=inp, shapes=True, value=value)
    assert gpu["err"] == 0
    assert _rel(gpu["c_max"], ref["c_max"]).max() <= 1e-4
    assert _rel(gpu["om"], ref["om"]).max() <= 1e-4
    B, Hq = w.batch, w.n_q_heads
    outs = {k: torch.empty((1, B, Hq), device="cuda") for k in ("ma", "ra", "ts", "th")}
    counts = torch.zeros(4, dtype=torch.int32, device="cuda")
    kvq.meter(gpu["ms_dev"].view(1, B, Hq, 8), 1, B, Hq, gpu["mp"], outs["ma"], outs["ra"], counts,
              two_sided=outs["ts"], det_tanh=outs["th"])
    ts = outs["ts"].cpu().numpy()[0].astype(np.float64)
    th = outs["th"].cpu().numpy()[0].astype(np.float64)
    ma = outs["ma"].cpu().numpy()[0].astype(np.float64)
    assert _rel(ts, ref["meter_2s"]).max() <= 1e-4
    assert _rel(th, ref["meter_tanh"]).max() <= 1e-4
    assert np.all(ts <= ma) and np.all(ts >= ref["tv"]) and np.all(th >= ref["tv"])
    if value:
        assert _rel(gpu["value_r"], ref["value_r"]).max() <= 2e-3


def test_shapes_change_nothing_else(kvq):
    w = CASES["int8"]()
    inp = make_inputs(w)
    on = run_case_gpu(w, inputs=inp, shapes=True)
    off = run_case_gpu(w, inputs=inp)
    assert np.array_equal(on["out"], off["out"])
    assert np.array_equal(on["state"][..., :6], off["state"][..., :6], equal_nan=True)
    assert np.all(np.isnan(off["state"][..., 6:8]))
