"""GPU parity of the quantize-on-append kernel and the conversion / dither hooks, via the C ABI.

Bar: codes, scales, dither and witness bit-exact with the oracle; the witness is
the exact band norm rounded up to fp16 (so also never below the exact norm).
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def kvq():
    import quantized_kv_cache_kvq_gb300 as m

    assert torch.cuda.is_available()
    m.load()
    return m


LAYOUTS = [("bf16", "e4m3s"), ("bf16", "bf16"), ("int8", "int8"), ("e4m3", "e4m3"), ("e4m3s", "e4m3s"),
           ("e4m3", "bf16"), ("bf16", "e4m3"), ("int8", "e4m3s")]


def _rows(n, hkv, seed, scale=1.0, outlier=False):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n, hkv, 128)) * scale
    if outlier:
        x[:, :, [3, 70]] *= 20
    return x.astype(np.float32)


@pytest.mark.parametrize("k_fmt,v_fmt", LAYOUTS)
def test_append_bit_exact(kvq, k_fmt, v_fmt):
    from oracle.encoders import fp16_value
    from oracle.quant import band_norms
    from quantized_kv_cache_kvq_gb300 import layout as L
    from tests.parity import oracle_cache_rows

    n, hkv, pages = 700, 4, 64
    k = _rows(n, hkv, 1, outlier=True)
    v = _rows(n, hkv, 2, scale=3.0)
    rng = np.random.default_rng(3)
    slots = rng.permutation(pages * 16)[:n].astype(np.int32)
    seed, layer = 0x0123456789ABCDEF, 5
    cache = kvq.PagedCache(k_fmt, v_fmt, hkv, pages, layer=layer, seed=seed)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.append(cache, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), torch.from_numpy(slots).cuda(), err)
    torch.cuda.synchronize()
    assert err.item() == 0
    ref = oracle_cache_rows(k, v, slots, k_fmt, v_fmt, seed, layer)
    pg, t = slots // 16, slots % 16
    kc = L.unpack_k(cache.k.cpu().numpy(), k_fmt, hkv)[pg, :, t]      # [n, hkv, 128]
    vc = L.unpack_v(cache.v.cpu().numpy(), v_fmt, hkv)[pg, :, t]
    assert np.array_equal(kc, ref["kc"].view(kc.dtype) if ref["kc"].dtype != kc.dtype else ref["kc"])
    assert np.array_equal(vc, ref["vc"].view(vc.dtype) if ref["vc"].dtype != vc.dtype else ref["vc"])
    if cache.k_scale is not None:
        assert np.array_equal(L.unpack_s(cache.k_scale.cpu().numpy(), hkv)[pg, :, t], ref["ksb"])
    if cache.v_scale is not None:
        assert np.array_equal(L.unpack_s(cache.v_scale.cpu().numpy(), hkv)[pg, :, t], ref["vsb"])
    w = L.unpack_w(cache.witness.cpu().numpy(), hkv)[pg, :, t]       # [n, hkv, 16]
    exact = band_norms(ref["kh"] - k.astype(np.float64))
    wv = fp16_value(w)
    assert np.all(wv >= exact)                                          # sound
    assert np.array_equal(w, ref["w16"])                                # bit-exact


def test_dither_hook_matches_oracle(kvq):
    from oracle.philox import dither

    slots = np.random.default_rng(4).integers(0, 2**31 - 1, 5000).astype(np.int32)
    out = torch.empty((5000, 128), dtype=torch.float32, device="cuda")
    for seed, layer, head in [(0, 0, 0), (0xFFFFFFFFFFFFFFFF, 27, 3), (123456789123, 11, 7)]:
        kvq.debug_dither(seed, layer, head, torch.from_numpy(slots).cuda(), out)
        ref = dither(seed, layer, head, slots[:, None], np.arange(128)[None, :])
        assert np.array_equal(out.cpu().numpy().astype(np.float64), ref)


@pytest.mark.parametrize("kind", [0, 1, 2, 3])
def test_device_encoders_match_oracle(kvq, kind):
    from oracle.encoders import bf16_bits_rne, e4m3_bits_rne_satfinite, fp16_bits

    rng = np.random.default_rng(10 + kind)
    bits = rng.integers(0, 2**32, 1 << 22, dtype=np.uint64).astype(np.uint32)
    # dense coverage of the e4m3 / fp16 ranges: exponents near zero with all low mantissa patterns
    dense = (np.arange(1 << 20, dtype=np.uint32) << 3) + np.uint32(0x3A000000)
    x = np.concatenate([bits.view(np.float32), dense.view(np.float32), -dense.view(np.float32)])
    x = x[np.isfinite(x)] if kind != 0 else x
    xt = torch.from_numpy(x.copy()).cuda()
    if kind == 1:
        out = torch.empty(x.size, dtype=torch.uint8, device="cuda")
    else:
        out = torch.empty(x.size, dtype=torch.int16, device="cuda")
    kvq.debug_encode(kind, xt, out)
    got = out.cpu().numpy()
    if kind == 0:
        ref = bf16_bits_rne(x)
        nan = np.isnan(x)
        assert np.array_equal(got.view(np.uint16)[~nan], ref[~nan])
    elif kind == 1:
        assert np.array_equal(got, e4m3_bits_rne_satfinite(x))
    else:
        ref = fp16_bits(x.astype(np.float64), "rne" if kind == 2 else "ru")
        assert np.array_equal(got.view(np.uint16), ref)


def test_append_device_errors(kvq):
    hkv, pages = 2, 4
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    cache = kvq.PagedCache("int8", "e4m3s", hkv, pages)
    k = torch.randn(3, hkv, 128, device="cuda")
    v = torch.randn(3, hkv, 128, device="cuda")
    # a slot beyond the cache
    kvq.append(cache, k, v, torch.tensor([0, 1, pages * 16 + 5], dtype=torch.int32, device="cuda"), err)
    torch.cuda.synchronize()
    assert err.item() == 5  # KVQ_ERR_DEVICE_BOUNDS
    # a non-finite key
    err.zero_()
    k2 = k.clone()
    k2[1, 0, 7] = float("nan")
    kvq.append(cache, k2, v, torch.tensor([0, 1, 2], dtype=torch.int32, device="cuda"), err)
    torch.cuda.synchronize()
    assert err.item() == 6  # KVQ_ERR_NONFINITE_INPUT
    # a value scale above the decode range
    err.zero_()
    v2 = v.clone()
    v2[2, 1, 0] = 2.0e5
    kvq.append(cache, k, v2, torch.tensor([0, 1, 2], dtype=torch.int32, device="cuda"), err)
    torch.cuda.synchronize()
    assert err.item() == 7  # KVQ_ERR_RANGE
    # negative slots are skipped silently
    err.zero_()
    kvq.append(cache, k, v, torch.tensor([-1, -1, 3], dtype=torch.int32, device="cuda"), err)
    torch.cuda.synchronize()
    assert err.item() == 0
