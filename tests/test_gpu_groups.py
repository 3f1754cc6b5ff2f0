"""GPU parity of the group-scaled INT8 layout (one fp16 scale per token per 32-channel group, WitCert §6.2.3,
Table 4's default G_c = 32) through the C ABI.

Bar: codes, group scales and the witness as in the per-token INT8 layout (codes, scales and the
witness bit-exact); decode output within 2e-3 relative, ln(A - 1)
of Tier A and Tier B within 1e-4, the meter never below the exact TV, for bf16 and fp32 queries, GQA groups
of 7 and 4, partial last pages, and keys whose groups have very different scales (massive channels in some
groups only).  Meter off and the value side leave the output bit-identical.  Mixed layouts are refused.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import workloads as W  # noqa: E402
from tests.parity import make_inputs, oracle_cache_rows, reference_case, run_case_gpu  # noqa: E402

G32 = dict(k_fmt="int8g32", v_fmt="int8g32")
CASES = {
    # 7 query heads per kv head, Tier B; massive RoPE pairs put a few channels of some groups far above the rest
    "int8g32": W.reduced(W.WORKLOADS["int8_7b_certified"], batch=3, seq_len=517, massive_pairs=4,
                         massive_scale=30.0, **G32),
    # 4 query heads per kv head, ragged lengths with a random page permutation
    "int8g32_ragged": W.reduced(W.WORKLOADS["ragged_paged"], batch=5, ragged=(17, 900), tier_b=True,
                                delta_req=1e-3, **G32),
}


@pytest.fixture(scope="module")
def kvq():
    import quantized_kv_cache_kvq_gb300 as m

    assert torch.cuda.is_available()
    m.load()
    return m


def _check(w, gpu, ref):
    assert gpu["err"] == 0
    on = np.linalg.norm(ref["out"], axis=-1)
    rel = np.linalg.norm(gpu["out"] - ref["out"], axis=-1) / on
    assert rel.max() <= 2e-3, rel.max()
    la_g, la_r = gpu["log_am1"], ref["log_am1"]
    both_inf = np.isneginf(la_g) & np.isneginf(la_r)
    assert np.all(np.abs(la_g - la_r)[~both_inf] <= 1e-4), np.nanmax(np.abs(la_g - la_r)[~both_inf])
    assert np.all(gpu["meter"] >= ref["tv"])
    assert np.allclose(gpu["lse"], ref["lse"], rtol=0, atol=2e-4)
    if w.tier_b:
        d = np.abs(gpu["log_am1_b"] - ref["log_am1_b"])
        assert d.max() <= 1e-4, d.max()


def test_append_group_scales_bit_exact(kvq):
    from oracle.encoders import fp16_value
    from oracle.quant import band_norms
    from quantized_kv_cache_kvq_gb300 import layout as L

    n, hkv, pages = 700, 4, 64
    rng = np.random.default_rng(11)
    k = rng.standard_normal((n, hkv, 128))
    k[:, :, [3, 70]] *= 40          # groups 0 and 2 carry massive channels, groups 1 and 3 do not
    v = rng.standard_normal((n, hkv, 128)) * 3
    v[:, :, 100] *= 25
    k, v = k.astype(np.float32), v.astype(np.float32)
    slots = rng.permutation(pages * 16)[:n].astype(np.int32)
    seed, layer = 0x0123456789ABCDEF, 5
    cache = kvq.PagedCache("int8g32", "int8g32", hkv, pages, layer=layer, seed=seed)
    assert cache.k_scale.shape[1] == 128 and cache.v_scale.shape[1] == 128
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.append(cache, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), torch.from_numpy(slots).cuda(), err)
    torch.cuda.synchronize()
    assert err.item() == 0
    ref = oracle_cache_rows(k, v, slots, "int8g32", "int8g32", seed, layer)
    pg, t = slots // 16, slots % 16
    kc = L.unpack_k(cache.k.cpu().numpy(), "int8g32", hkv)[pg, :, t]
    vc = L.unpack_v(cache.v.cpu().numpy(), "int8g32", hkv)[pg, :, t]
    assert np.array_equal(kc.view(np.int8), ref["kc"])
    assert np.array_equal(vc.view(np.int8), ref["vc"])
    ks = L.unpack_gs(cache.k_scale.cpu().numpy(), hkv)[pg, :, t]       # [n, hkv, 4]
    vs = L.unpack_gs(cache.v_scale.cpu().numpy(), hkv)[pg, :, t]
    assert np.array_equal(ks, ref["ksb"]) and np.array_equal(vs, ref["vsb"])
    # the groups really differ: massive-channel groups carry scales far above the others
    kv = fp16_value(ks)
    assert np.median(kv[..., 0] / kv[..., 1]) > 5
    w = L.unpack_w(cache.witness.cpu().numpy(), hkv)[pg, :, t]
    exact = band_norms(ref["kh"] - k.astype(np.float64))
    assert np.all(fp16_value(w) >= exact)
    assert np.array_equal(w, ref["w16"])


@pytest.mark.parametrize("name", list(CASES))
def test_decode_group_scales_parity(kvq, name):
    w = CASES[name]
    inp = make_inputs(w, layer=1)
    _check(w, run_case_gpu(w, layer=1, inputs=inp), reference_case(w, layer=1, inputs=inp))


def test_decode_group_scales_fp32_query(kvq):
    # the key products add the query's low part; the dither products and each group's 9/2 sum start value use
    # the high part
    w = W.reduced(CASES["int8g32"], q_dtype="f32", seq_len=300)
    inp = make_inputs(w)
    _check(w, run_case_gpu(w, inputs=inp), reference_case(w, inputs=inp))


def test_group_scales_meter_off_and_value_side(kvq):
    w = W.reduced(CASES["int8g32"], seq_len=200)
    inp = make_inputs(w)
    on = run_case_gpu(w, inputs=inp, meter=True)
    off = run_case_gpu(w, inputs=inp, meter=False)
    val = run_case_gpu(w, inputs=inp, meter=True, value=True)
    assert np.array_equal(on["out"], off["out"]) and np.array_equal(on["out"], val["out"])
    ref = reference_case(w, inputs=inp)
    rel = np.abs(val["value_r"] - ref["value_r"]) / np.maximum(ref["value_r"], 1e-30)
    assert rel.max() <= 2e-3, rel.max()
    vm, vr = val["value_vmax"], ref["value_vmax"]
    assert np.all(vm >= vr) and np.all(vm <= vr * (1 + 2.0 ** -10) + 1e-30)


def test_group_scales_fewer_tokens_than_a_page(kvq):
    w = W.reduced(CASES["int8g32"], batch=2, seq_len=5)
    inp = make_inputs(w)
    _check(w, run_case_gpu(w, inputs=inp), reference_case(w, inputs=inp))


def test_mixed_layouts_refused(kvq):
    dev = torch.device("cuda")
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    k = torch.zeros((1, 2, 128), device=dev)
    slots = torch.zeros(1, dtype=torch.int32, device=dev)
    for kf, vf in (("int8g32", "int8"), ("int8", "int8g32"), ("bf16", "int8g32")):
        cache = kvq.PagedCache(kf, vf, 2, 4, device=dev)
        with pytest.raises(RuntimeError, match="UNSUPPORTED_LAYOUT"):
            kvq.append(cache, k, k, slots, err)
    pairs = torch.tensor([[1, 2], [3, 4]], dtype=torch.int32)
    cache = kvq.PagedCache("int8g32", "int8g32", 2, 4, device=dev, outlier_pairs=pairs)
    with pytest.raises(RuntimeError, match="UNSUPPORTED_LAYOUT"):
        kvq.append(cache, k, k, slots, err)
    torch.cuda.synchronize()
    assert err.item() == 0
