"""GPU parity of the value side of the output-error bound (WitCert Sec. 3) via the C ABI.

||y - y_hat|| <= 2 TV max_t ||v_t|| + sum_t p~_t rho^v_t.  kvq_append stores the value witness
(rho^v_t, ||v_t||) as fp16 rounded up; the decode accumulates R = sum_t p~_t rho^v_t with the
softmax weights and Vmax = max_t ||v_t||, merges both over the splits, and kvq_meter turns them
into the bound 2 meter Vmax + R.  Bars:
* stored value witness: bit-exact with the oracle (each the exact norm rounded up to fp16), so never
  below the exact norms;
* R within 2e-3 relative of the oracle (fp32 accumulation), Vmax the oracle's exactly;
* the bound from kvq_meter within 2e-3 relative of the oracle's and never below the exact output
  error ||y - y_hat|| (exact keys and values, float64);
* the value side changes nothing else: out and the Tier A / B state are bit-identical with it off.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import workloads as W  # noqa: E402
from tests.parity import make_inputs, oracle_cache_rows, reference_case, run_case_gpu  # noqa: E402

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


@pytest.mark.parametrize("k_fmt,v_fmt", [("bf16", "e4m3s"), ("bf16", "bf16"), ("int8", "int8"), ("e4m3", "e4m3"),
                                         ("e4m3s", "e4m3s")])
def test_append_value_witness(kvq, k_fmt, v_fmt):
    from oracle.encoders import fp16_value
    from quantized_kv_cache_kvq_gb300 import layout as L

    n, hkv, pages = 500, 4, 48
    rng = np.random.default_rng(11)
    k = rng.standard_normal((n, hkv, 128)).astype(np.float32)
    v = (rng.standard_normal((n, hkv, 128)) * rng.uniform(0.05, 20.0, (n, hkv, 1))).astype(np.float32)
    slots = rng.permutation(pages * 16)[:n].astype(np.int32)
    seed, layer = 0x1234, 3
    cache = kvq.PagedCache(k_fmt, v_fmt, hkv, pages, layer=layer, seed=seed, value_witness=True)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.append(cache, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), torch.from_numpy(slots).cuda(), err)
    torch.cuda.synchronize()
    assert err.item() == 0
    ref = oracle_cache_rows(k, v, slots, k_fmt, v_fmt, seed, layer)
    pg, t = slots // 16, slots % 16
    got = L.unpack_vw(cache.v_witness.cpu().numpy(), hkv)[pg, :, t]     # [n, hkv, 2] fp16 bits
    r = ref["vh"] - v.astype(np.float64)
    exact = np.stack([np.sqrt((r * r).sum(-1)), np.sqrt((v.astype(np.float64) ** 2).sum(-1))], axis=-1)
    assert np.all(fp16_value(got) >= exact)                               # sound
    assert np.array_equal(got, ref["vw16"])                               # bit-exact


@pytest.mark.parametrize("name", list(CASES))
def test_value_side_parity_and_soundness(kvq, name):
    w = CASES[name]()
    inp = make_inputs(w)
    ref = reference_case(w, inputs=inp)
    gpu = run_case_gpu(w, inputs=inp, value=True)
    assert gpu["err"] == 0
    B, Hq = w.batch, w.n_q_heads
    rel = np.abs(gpu["value_r"] - ref["value_r"]) / np.maximum(ref["value_r"], 1e-30)
    assert rel.max() <= 2e-3, rel.max()
    vm, vr = gpu["value_vmax"], ref["value_vmax"]
    assert np.array_equal(vm, vr)
    # the bound through kvq_meter
    ma = torch.empty((1, B, Hq), device="cuda")
    ra = torch.empty((1, B, Hq), device="cuda")
    ob = torch.empty((1, B, Hq), device="cuda")
    counts = torch.zeros(4, dtype=torch.int32, device="cuda")
    kvq.meter(gpu["ms_dev"].view(1, B, Hq, 8), 1, B, Hq, gpu["mp"], ma, ra, counts, out_bound=ob)
    bound = ob.cpu().numpy()[0].astype(np.float64)
    meter = ma.cpu().numpy()[0].astype(np.float64)
    assert np.allclose(bound, 2 * meter * vm + gpu["value_r"], rtol=1e-6)
    rel_b = np.abs(bound - ref["out_bound"]) / np.maximum(ref["out_bound"], 1e-30)
    assert rel_b.max() <= 2e-3, rel_b.max()
    assert np.all(bound >= ref["out_err"]), (bound - ref["out_err"]).min()


def test_value_side_changes_nothing_else(kvq):
    w = CASES["cartridge"]()
    inp = make_inputs(w)
    on = run_case_gpu(w, inputs=inp, value=True)
    off = run_case_gpu(w, inputs=inp, value=False)
    assert np.array_equal(on["out"], off["out"])
    assert np.array_equal(on["state"][..., :4], off["state"][..., :4], equal_nan=True)
    assert np.all(np.isnan(off["state"][..., 4:6]))


def test_value_side_needs_the_value_witness(kvq):
    w = W.reduced(W.WORKLOADS["tiny"], seq_len=64)
    inp = make_inputs(w)
    dev = torch.device("cuda")
    cache = kvq.PagedCache(w.k_fmt, w.v_fmt, w.n_kv_heads, inp["num_pages"], device=dev)  # no value witness
    q = torch.zeros((1, w.n_q_heads, 128), dtype=torch.float32, device=dev)
    out = torch.empty((1, w.n_q_heads, 128), device=dev)
    ms = torch.empty((1, w.n_q_heads, 8), device=dev)
    ws = torch.empty(kvq.decode_workspace_size(1, w.n_kv_heads, w.n_q_heads), dtype=torch.uint8, device=dev)
    mp = kvq.meter_params(kvq.TIER_A | kvq.TIER_V, 1, w.n_q_heads)
    with pytest.raises(kvq.KvqError) as e:
        kvq.decode_attn(cache, q, torch.from_numpy(inp["bt"]).to(dev), torch.tensor([64], dtype=torch.int32, device=dev),
                        out, ws, meter=mp, meter_state=ms)
    assert e.value.status == 1  # KVQ_ERR_INVALID_ARG
