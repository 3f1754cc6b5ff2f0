"""GPU parity on the method's edge cases, through the C ABI, against the oracle.

* Identity quantizer (WitCert §3, Theorem 1 with w = 0): keys that are already bfloat16 values stored in
  the BF16 layout have an exactly zero residual, so every witness byte is 0, ln(A - 1) is -inf and the
  meter is exactly 0 (and so is the oracle's exact TV).
* All-zero rows (WitCert §4.2 quantizer, amax = 0): E4M3-scaled values, INT8 keys and values, and one
  all-zero 32-channel group of the group-scaled INT8 layout store scale 0 and code 0, bit for bit; the
  decode over those rows matches the oracle.
* Exact half-ties of rint(fp32(fp32(x / s) + xi)) (the 0.5-tie disagreement of WitCert §6.2.1's
  acceptance list): inputs built so that y + xi = k + 1/2 exactly for the row's own dither; both sides
  round half to even.
* E4M3 saturation: the raw cast of values at and beyond +-448 (and of inf), ties between E4M3 values,
  E4M3 subnormals, and the scaled path where the fp16 scale rounds down so that x / s exceeds 448.
* The per-request risk ranking of the FP8 raw-cast workload from a real decode of every layer, against
  the oracle's ranking of the oracle's own raw scores, up to float64 near-ties.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import workloads as W  # noqa: E402
from tests.parity import make_inputs, oracle_cache_rows, reference_case, run_case_gpu  # noqa: E402


@pytest.fixture(scope="module")
def kvq():
    import quantized_kv_cache_kvq_gb300 as m

    assert torch.cuda.is_available()
    m.load()
    return m


def _decode_ok(w, gpu, ref):
    assert gpu["err"] == 0
    on = np.linalg.norm(ref["out"], axis=-1)
    rel = np.linalg.norm(gpu["out"] - ref["out"], axis=-1) / np.maximum(on, 1e-30)
    assert rel.max() <= 2e-3, rel.max()
    la_g, la_r = gpu["log_am1"], ref["log_am1"]
    both = np.isneginf(la_g) & np.isneginf(la_r)
    assert np.all(np.abs(la_g[~both] - la_r[~both]) <= 1e-4)
    assert np.all(gpu["meter"] >= ref["tv"])
    if w.tier_b:
        assert np.max(np.abs(gpu["log_am1_b"] - ref["log_am1_b"])) <= 1e-4


def _stored_rows(cache, w, slots):
    """Codes, scales and witness bits the GPU stored at ``slots`` (all kv heads)."""
    from quantized_kv_cache_kvq_gb300 import layout as L

    hkv = w.n_kv_heads
    pg, t = slots // 16, slots % 16
    out = {"kc": L.unpack_k(cache.k.cpu().numpy(), w.k_fmt, hkv)[pg, :, t],
           "vc": L.unpack_v(cache.v.cpu().numpy(), w.v_fmt, hkv)[pg, :, t],
           "w16": L.unpack_w(cache.witness.cpu().numpy(), hkv)[pg, :, t]}
    for side, fmt in (("k", w.k_fmt), ("v", w.v_fmt)):
        sc = getattr(cache, f"{side}_scale")
        if sc is None:
            out[f"{side}sb"] = None
        elif fmt == "int8g32":
            out[f"{side}sb"] = L.unpack_gs(sc.cpu().numpy(), hkv)[pg, :, t]
        else:
            out[f"{side}sb"] = L.unpack_s(sc.cpu().numpy(), hkv)[pg, :, t]
    return out


def _same_rows(got, ref):
    for key in ("kc", "vc", "w16", "ksb", "vsb"):
        if ref[key] is None:
            assert got[key] is None, key
            continue
        r = ref[key] if ref[key].dtype == got[key].dtype else ref[key].view(got[key].dtype)
        assert np.array_equal(got[key], r), key


def test_identity_quantizer_meters_exactly_zero(kvq):
    w = W.reduced(W.WORKLOADS["tiny"], seq_len=300)          # K bf16 / V e4m3 scaled, fp32 query
    inp = make_inputs(w)
    inp["seqs"] = [(W.round_bf16_input(k), v, q) for k, v, q in inp["seqs"]]
    ref = reference_case(w, inputs=inp)
    gpu = run_case_gpu(w, inputs=inp)
    assert gpu["err"] == 0
    assert not np.any(gpu["cache"].witness.cpu().numpy())     # every witness byte 0
    assert np.all(np.isneginf(gpu["log_am1"])) and np.all(gpu["meter"] == 0.0)
    assert np.all(np.isneginf(ref["log_am1"])) and np.all(ref["tv"] == 0.0)
    _decode_ok(w, gpu, ref)
    # and kvq_meter turns -inf into meter 0 and raw score -inf
    B, Hq = w.batch, w.n_q_heads
    ma, ra = torch.empty((1, B, Hq), device="cuda"), torch.empty((1, B, Hq), device="cuda")
    counts = torch.zeros(4, dtype=torch.int32, device="cuda")
    kvq.meter(gpu["ms_dev"].view(1, B, Hq, 8), 1, B, Hq, gpu["mp"], ma, ra, counts)
    assert np.all(ma.cpu().numpy() == 0.0) and np.all(np.isneginf(ra.cpu().numpy()))
    assert counts.cpu().tolist()[0] == B * Hq


ZERO_LAYOUTS = {
    "e4m3s_values": dict(k_fmt="bf16", v_fmt="e4m3s"),
    "int8": dict(k_fmt="int8", v_fmt="int8", tier_b=True, delta_req=1e-3),
    "int8g32": dict(k_fmt="int8g32", v_fmt="int8g32", tier_b=True, delta_req=1e-3),
}


@pytest.mark.parametrize("name", list(ZERO_LAYOUTS))
def test_all_zero_rows_store_scale_zero_and_decode(kvq, name):
    w = W.reduced(W.WORKLOADS["tiny"], batch=2, n_q_heads=28, n_kv_heads=4, seq_len=250, **ZERO_LAYOUTS[name])
    inp = make_inputs(w)
    seqs = []
    for s, (k, v, q) in enumerate(inp["seqs"]):
        k, v = k.copy(), v.copy()
        k[3::7] = 0.0                      # whole key rows
        v[5::6] = 0.0                      # whole value rows
        if w.k_fmt == "int8g32":           # one zero group per row for some tokens: group 1 of K, group 2 of V
            k[2::4, :, 32:64] = 0.0
            v[2::3, :, 64:96] = 0.0
        seqs.append((k, v, q))
    inp["seqs"] = seqs
    ref = reference_case(w, inputs=inp)
    gpu = run_case_gpu(w, inputs=inp)
    _decode_ok(w, gpu, ref)
    for s, (slots, rows) in enumerate(ref["rows"]):
        got = _stored_rows(gpu["cache"], w, slots)
        _same_rows(got, rows)
        k, v, _ = inp["seqs"][s]
        zk = np.all(k == 0, axis=-1)                               # [n, hkv]
        zv = np.all(v == 0, axis=-1)
        assert zk.any() and zv.any()
        if w.k_fmt != "int8g32":
            if got["ksb"] is not None:
                assert np.all(got["ksb"][zk] == 0)
            assert np.all(got["vsb"][zv] == 0)
            assert np.all(got["vc"][zv].astype(np.int64) == 0)
        else:
            assert np.all(got["ksb"][..., 1][np.all(k[..., 32:64] == 0, axis=-1)] == 0)
            assert np.all(got["vsb"][..., 2][np.all(v[..., 64:96] == 0, axis=-1)] == 0)
        if w.k_fmt.startswith("int8"):
            assert np.all(got["kc"][zk] == 0)


def test_int8_exact_half_ties_round_to_even(kvq):
    """Rows whose every channel c > 0 lands on y + xi = k_c + 1/2 exactly (channel 0 carries the amax that
    fixes s = 2^-6): the codes must be the even neighbours on both sides."""
    from oracle.philox import dither
    from quantized_kv_cache_kvq_gb300 import layout as L

    n, hkv, pages = 96, 2, 8
    seed, layer = 0x7E57_0001, 4
    rng = np.random.default_rng(21)
    slots = rng.permutation(pages * 16)[:n].astype(np.int32)
    xi = dither(seed, layer, np.arange(hkv)[None, :, None], slots[:, None, None], np.arange(128)[None, None, :])
    kint = rng.integers(-120, 120, (n, hkv, 128))
    # x = (k + 1/2 - xi) / 64: exact in binary32 (xi on the 2^-10 grid), x / s = x * 64 exactly
    x = ((kint + 0.5 - xi) / 64.0).astype(np.float32)
    x[..., 0] = np.float32(126.5 / 64.0)           # amax: s = fp16(amax / 126.5) = 2^-6 exactly
    assert np.all(np.abs(x[..., 1:]) < x[..., :1])
    y2 = x[..., 1:].astype(np.float64) * 64.0 + xi[..., 1:]
    assert np.all(y2 - np.floor(y2) == 0.5)        # every such channel is an exact tie
    cache = kvq.PagedCache("int8", "int8", hkv, pages, layer=layer, seed=seed)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    xt = torch.from_numpy(x).cuda()
    kvq.append(cache, xt, xt, torch.from_numpy(slots).cuda(), err)
    torch.cuda.synchronize()
    assert err.item() == 0
    ref = oracle_cache_rows(x, x, slots, "int8", "int8", seed, layer)
    pg, t = slots // 16, slots % 16
    kc = L.unpack_k(cache.k.cpu().numpy(), "int8", hkv)[pg, :, t]
    vc = L.unpack_v(cache.v.cpu().numpy(), "int8", hkv)[pg, :, t]
    assert np.array_equal(kc, ref["kc"]) and np.array_equal(vc, ref["vc"])
    assert np.all(kc[..., 1:].astype(np.int64) % 2 == 0)            # half to even
    assert np.array_equal(L.unpack_s(cache.k_scale.cpu().numpy(), hkv)[pg, :, t], ref["ksb"])
    assert np.array_equal(L.unpack_w(cache.witness.cpu().numpy(), hkv)[pg, :, t], ref["w16"])


def test_e4m3_saturation_ties_and_subnormals(kvq):
    from quantized_kv_cache_kvq_gb300 import layout as L

    special = np.array([448.0, 449.0, 463.9, 464.0, 464.1, 479.0, 480.0, 500.0, 1e6, 3.0e38, np.inf,
                        2.0 ** -10, 3 * 2.0 ** -11, 2.0 ** -9, 1.5 * 2.0 ** -9, 2.0 ** -12, 1e-30,
                        0.0, 1.0 + 2.0 ** -4, 1.0 + 3 * 2.0 ** -4, 240.0, 232.0, 248.0], dtype=np.float64)
    vals = np.concatenate([special, -special])
    hkv, pages = 2, 4
    n = 8
    rng = np.random.default_rng(22)
    x = rng.standard_normal((n, hkv, 128)).astype(np.float32)
    x[:, :, :vals.size] = vals.astype(np.float32)
    k = x.copy()
    k[~np.isfinite(k)] = 0.0                      # keys stay finite (a non-finite key is flagged)
    v = x.copy()
    v[~np.isfinite(v)] = 0.0
    slots = np.arange(n, dtype=np.int32)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    cache = kvq.PagedCache("e4m3", "e4m3", hkv, pages)
    kvq.append(cache, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), torch.from_numpy(slots).cuda(), err)
    torch.cuda.synchronize()
    assert err.item() == 0
    ref = oracle_cache_rows(k, v, slots, "e4m3", "e4m3", 0, 0)
    kc = L.unpack_k(cache.k.cpu().numpy(), "e4m3", hkv)[slots // 16, :, slots % 16]
    assert np.array_equal(kc, ref["kc"])
    assert np.all(kc[..., :8] == ref["kc"][..., :8]) and np.all((kc[0, 0, 1:10] & 0x7F) == 0x7E)  # saturated to 448
    # the device conversion of the infinities and of the largest binary32 values, against the oracle's encoder
    from oracle.encoders import e4m3_bits_rne_satfinite

    big = np.array([np.inf, -np.inf, 3.4e38, -3.4e38, 464.0, -464.0], dtype=np.float32)
    out = torch.empty(big.size, dtype=torch.uint8, device="cuda")
    kvq.debug_encode(1, torch.from_numpy(big).cuda(), out)
    assert np.array_equal(out.cpu().numpy(), e4m3_bits_rne_satfinite(big))
    # scaled values: amax / 448 = 1 + 2^-12 rounds down to the fp16 scale 1.0, so the amax channel's
    # x / s = 448.11 saturates to 448
    vs = rng.standard_normal((n, hkv, 128)).astype(np.float32)
    vs[:, :, 7] = np.float32(448.0 * (1 + 2.0 ** -12))
    cache2 = kvq.PagedCache("bf16", "e4m3s", hkv, pages)
    kvq.append(cache2, torch.from_numpy(k).cuda(), torch.from_numpy(vs).cuda(), torch.from_numpy(slots).cuda(), err)
    torch.cuda.synchronize()
    assert err.item() == 0
    ref2 = oracle_cache_rows(k, vs, slots, "bf16", "e4m3s", 0, 0)
    vc = L.unpack_v(cache2.v.cpu().numpy(), "e4m3s", hkv)[slots // 16, :, slots % 16]
    assert np.array_equal(vc, ref2["vc"]) and np.all(vc[..., 7] == 0x7E)
    assert np.array_equal(L.unpack_s(cache2.v_scale.cpu().numpy(), hkv)[slots // 16, :, slots % 16], ref2["vsb"])
    assert np.all(ref2["vsb"] == np.float16(1.0).view(np.uint16))


def test_fp8_raw_ranking_from_a_real_decode(kvq):
    """Config 4's gating output: kvq_meter ranks (layer, head) cells per request from the decode's own meter
    states; the order must follow the oracle's float64 raw scores (ties within 1e-4 may swap)."""
    from oracle import meter as OM

    w = W.reduced(W.WORKLOADS["fp8_raw_stress"], batch=3, n_layers=4, seq_len=700)
    L_, B, Hq = w.n_layers, w.batch, w.n_q_heads
    states, raw_ref = [], []
    for layer in range(L_):
        inp = make_inputs(w, layer)
        gpu = run_case_gpu(w, layer=layer, inputs=inp)
        ref = reference_case(w, layer=layer, inputs=inp)
        _decode_ok(w, gpu, ref)
        states.append(gpu["ms_dev"])
        raw_ref.append(ref["raw"])
        mp = gpu["mp"]
    st = torch.stack(states).contiguous()                                   # [L, B, H, 8]
    ma = torch.empty((L_, B, Hq), device="cuda")
    ra = torch.empty((L_, B, Hq), device="cuda")
    counts = torch.zeros(4, dtype=torch.int32, device="cuda")
    rank = torch.empty((B, L_ * Hq), dtype=torch.int32, device="cuda")
    kvq.meter(st, L_, B, Hq, mp, ma, ra, counts, ranking=rank)
    torch.cuda.synchronize()
    rk = rank.cpu().numpy().astype(np.int64)
    raw = np.stack(raw_ref).transpose(1, 0, 2).reshape(B, -1)             # oracle raw [B, L*H]
    ref_rank = OM.rank_cells(np.stack(raw_ref).transpose(1, 0, 2))
    assert np.isfinite(raw).all() and raw.std() > 0.1                     # informative, varied scores
    for b in range(B):
        assert sorted(rk[b].tolist()) == list(range(L_ * Hq))              # a permutation
        s = raw[b][rk[b]]
        assert np.all(np.diff(s) <= 1e-4 * np.maximum(1.0, np.abs(s[1:])))  # non-increasing up to near-ties
        # where the oracle's scores are separated by more than the tolerance, the positions agree
        sep = np.abs(np.diff(raw[b][ref_rank[b]])) > 1e-4 * np.maximum(1.0, np.abs(raw[b][ref_rank[b]][1:]))
        pos_g = np.argsort(rk[b])
        pos_r = np.argsort(ref_rank[b])
        isolated = np.ones(L_ * Hq, bool)
        isolated[ref_rank[b][1:][~sep]] = False
        isolated[ref_rank[b][:-1][~sep]] = False
        assert np.array_equal(pos_g[isolated], pos_r[isolated])
