"""GPU parity of the fixed-channel key outlier bypass (WitCert Sec. 6.2.5) via the C ABI.

INT8-dithered keys with m RoPE pairs per (layer, kv head) stored in fp16 and left out of the INT8
amax.  Bars: codes, scales and the fp16 outlier values bit-exact with the oracle (bypassed codes 0);
witness bit-exact (the exact band norm rounded up to fp16); decode output within 2e-3 and both
meters' ln(A - 1) within 1e-4 of the oracle (Tier B with the deterministic fp16 term of the bypassed
channels), meter >= exact TV; and the page's Table 5 effect on the GPU: the same massive-pair
workload meters far lower with the bypass than without.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import workloads as W  # noqa: E402
from tests.parity import make_inputs, oracle_cache_rows, reference_case, run_case_gpu  # noqa: E402


def _wl(m, q_dtype="bf16", bypass=True):
    base = W.WORKLOADS["int8_7b_certified"]
    return W.reduced(base, batch=2, seq_len=333, massive_pairs=m, massive_scale=30.0, bypass_pairs=m if bypass else 0,
                     q_dtype=q_dtype)


@pytest.fixture(scope="module")
def kvq():
    import quantized_kv_cache_kvq_gb300 as m

    m.load()
    return m


@pytest.mark.parametrize("m", [4, 8])
def test_append_bypass_bit_exact(kvq, m):
    from oracle.encoders import fp16_value
    from oracle.quant import band_norms
    from quantized_kv_cache_kvq_gb300 import layout as L

    n, hkv, pages = 400, 4, 32
    rng = np.random.default_rng(21)
    pairs = np.stack([np.sort(rng.choice(64, m, replace=False)) for _ in range(hkv)]).astype(np.int32)
    k = rng.standard_normal((n, hkv, 128))
    for h in range(hkv):
        k[:, h, np.concatenate([pairs[h], pairs[h] + 64])] *= 40.0
    k = k.astype(np.float32)
    v = rng.standard_normal((n, hkv, 128)).astype(np.float32)
    slots = rng.permutation(pages * 16)[:n].astype(np.int32)
    seed, layer = 0xABCDEF, 2
    cache = kvq.PagedCache("int8", "int8", hkv, pages, layer=layer, seed=seed,
                           outlier_pairs=torch.from_numpy(pairs).cuda())
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.append(cache, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), torch.from_numpy(slots).cuda(), err)
    torch.cuda.synchronize()
    assert err.item() == 0
    ref = oracle_cache_rows(k, v, slots, "int8", "int8", seed, layer, pairs=pairs)
    pg, t = slots // 16, slots % 16
    kc = L.unpack_k(cache.k.cpu().numpy(), "int8", hkv)[pg, :, t]
    assert np.array_equal(kc.view(np.int8), ref["kc"])
    assert np.array_equal(L.unpack_s(cache.k_scale.cpu().numpy(), hkv)[pg, :, t], ref["ksb"])
    ko = L.unpack_ko(cache.k_outlier.cpu().numpy(), hkv, m)[pg, :, t]
    assert np.array_equal(ko, ref["kob"])
    w = L.unpack_w(cache.witness.cpu().numpy(), hkv)[pg, :, t]
    exact = band_norms(ref["kh"] - k.astype(np.float64))
    assert np.all(fp16_value(w) >= exact)
    assert np.array_equal(w, ref["w16"])


@pytest.mark.parametrize("m,q_dtype", [(4, "bf16"), (8, "bf16"), (4, "f32")])
def test_decode_bypass_parity(kvq, m, q_dtype):
    w = _wl(m, q_dtype)
    inp = make_inputs(w)
    ref = reference_case(w, inputs=inp)
    gpu = run_case_gpu(w, inputs=inp)
    assert gpu["err"] == 0
    rel = np.linalg.norm(gpu["out"] - ref["out"], axis=-1) / np.linalg.norm(ref["out"], axis=-1)
    assert rel.max() <= 2e-3, rel.max()
    assert np.max(np.abs(gpu["log_am1"] - ref["log_am1"])) <= 1e-4
    assert np.max(np.abs(gpu["log_am1_b"] - ref["log_am1_b"])) <= 1e-4
    assert np.all(gpu["meter"] >= ref["tv"])


def test_table5_effect_on_gpu(kvq):
    w_on, w_off = _wl(4, bypass=True), _wl(4, bypass=False)
    on = run_case_gpu(w_on, inputs=make_inputs(w_on))
    off = run_case_gpu(w_off, inputs=make_inputs(w_off))
    assert on["err"] == 0 and off["err"] == 0
    raw_on = np.exp(on["log_am1"]) * (np.exp(on["log_am1"]) + 2) / 2   # 1/2 (A^2 - 1)
    raw_off = np.exp(off["log_am1"]) * (np.exp(off["log_am1"]) + 2) / 2
    assert np.median(raw_off) >= 1.0
    assert np.median(raw_on) <= np.median(raw_off) / 10 and raw_on.max() < 0.2


def test_bypass_needs_int8_keys_and_valid_pairs(kvq):
    pairs = torch.tensor([[1, 2, 3, 4]] * 2, dtype=torch.int32, device="cuda")
    bad = kvq.PagedCache("bf16", "e4m3s", 2, 4, outlier_pairs=pairs)
    k = torch.randn((4, 2, 128), device="cuda")
    slots = torch.arange(4, dtype=torch.int32, device="cuda")
    with pytest.raises(kvq.KvqError) as e:
        kvq.append(bad, k, k.clone(), slots)
    assert e.value.status == 2  # KVQ_ERR_UNSUPPORTED_LAYOUT
    out_of_range = kvq.PagedCache("int8", "int8", 2, 4, outlier_pairs=torch.tensor([[1, 70]] * 2, dtype=torch.int32,
                                                                                  device="cuda"))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.append(out_of_range, k, k.clone(), slots, err)
    torch.cuda.synchronize()
    assert err.item() == 5  # KVQ_ERR_DEVICE_BOUNDS
