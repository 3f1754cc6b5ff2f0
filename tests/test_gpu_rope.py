"""GPU parity of RoPE-on-append (kvq_append_rope) via the C ABI.

Keys arrive pre-RoPE with their positions and the caller's binary32 cos/sin table; the oracle rotates
them in binary32 step by step (oracle.rope) and quantizes the result.  Bars: codes and scales
bit-exact with the oracle on four layouts (a rotation computed differently, e.g. with fused
multiply-adds, moves some codes), the witness bit-exact;
position 0 equals kvq_append of the same keys byte for byte; a position outside the table is
reported and its token skipped.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

LAYOUTS = [("bf16", "e4m3s"), ("int8", "int8"), ("e4m3", "e4m3"), ("bf16", "bf16")]


@pytest.fixture(scope="module")
def kvq():
    import quantized_kv_cache_kvq_gb300 as m

    m.load()
    return m


def _planes(cache):
    return [p.clone() for p in (cache.k, cache.v, cache.witness, cache.k_scale, cache.v_scale) if p is not None]


@pytest.mark.parametrize("k_fmt,v_fmt", LAYOUTS)
def test_append_rope_bit_exact(kvq, k_fmt, v_fmt):
    from oracle.encoders import fp16_value
    from oracle.quant import band_norms
    from oracle.rope import cos_sin_table, rope_fp32
    from quantized_kv_cache_kvq_gb300 import layout as L
    from tests.parity import oracle_cache_rows

    n, hkv, pages, max_pos = 600, 4, 64, 8192
    rng = np.random.default_rng(11)
    k = (rng.standard_normal((n, hkv, 128)) * 3).astype(np.float32)
    v = rng.standard_normal((n, hkv, 128)).astype(np.float32)
    pos = rng.integers(0, max_pos, n).astype(np.int32)
    slots = rng.permutation(pages * 16)[:n].astype(np.int32)
    table = cos_sin_table(max_pos)
    seed, layer = 0x5EED, 3
    cache = kvq.PagedCache(k_fmt, v_fmt, hkv, pages, layer=layer, seed=seed)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.append_rope(cache, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), torch.from_numpy(pos).cuda(),
                    torch.from_numpy(table).cuda(), torch.from_numpy(slots).cuda(), err)
    torch.cuda.synchronize()
    assert err.item() == 0
    k_rot = rope_fp32(k, pos, table)
    ref = oracle_cache_rows(k_rot, v, slots, k_fmt, v_fmt, seed, layer)
    pg, t = slots // 16, slots % 16
    kc = L.unpack_k(cache.k.cpu().numpy(), k_fmt, hkv)[pg, :, t]
    vc = L.unpack_v(cache.v.cpu().numpy(), v_fmt, hkv)[pg, :, t]
    assert np.array_equal(kc, ref["kc"].view(kc.dtype) if ref["kc"].dtype != kc.dtype else ref["kc"])
    assert np.array_equal(vc, ref["vc"].view(vc.dtype) if ref["vc"].dtype != vc.dtype else ref["vc"])
    if cache.k_scale is not None:
        assert np.array_equal(L.unpack_s(cache.k_scale.cpu().numpy(), hkv)[pg, :, t], ref["ksb"])
    if cache.v_scale is not None:
        assert np.array_equal(L.unpack_s(cache.v_scale.cpu().numpy(), hkv)[pg, :, t], ref["vsb"])
    w = L.unpack_w(cache.witness.cpu().numpy(), hkv)[pg, :, t]
    assert np.all(fp16_value(w) >= band_norms(ref["kh"] - k_rot.astype(np.float64)))   # sound
    assert np.array_equal(w, ref["w16"])


def test_position_zero_is_plain_append_and_bad_positions_are_reported(kvq):
    from oracle.rope import cos_sin_table

    n, hkv, pages = 96, 2, 8
    rng = np.random.default_rng(12)
    k = torch.from_numpy(rng.standard_normal((n, hkv, 128)).astype(np.float32)).cuda()
    v = torch.from_numpy(rng.standard_normal((n, hkv, 128)).astype(np.float32)).cuda()
    slots = torch.from_numpy(rng.permutation(pages * 16)[:n].astype(np.int32)).cuda()
    table = torch.from_numpy(cos_sin_table(16)).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    a = kvq.PagedCache("int8", "e4m3s", hkv, pages, seed=7)
    b = kvq.PagedCache("int8", "e4m3s", hkv, pages, seed=7)
    kvq.append_rope(a, k, v, torch.zeros(n, dtype=torch.int32, device="cuda"), table, slots, err)
    kvq.append(b, k, v, slots, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert all(torch.equal(x, y) for x, y in zip(_planes(a), _planes(b)))
    # token 5 at a position past the table: reported, and its slot left as it was
    c = kvq.PagedCache("int8", "e4m3s", hkv, pages, seed=7)
    before = _planes(c)
    bad = torch.zeros(n, dtype=torch.int32, device="cuda")
    bad[5] = 16
    kvq.append_rope(c, k[5:6].contiguous(), v[5:6].contiguous(), bad[5:6].contiguous(), table,
                    slots[5:6].contiguous(), err)
    torch.cuda.synchronize()
    assert err.item() == 5   # KVQ_ERR_DEVICE_BOUNDS
    assert all(torch.equal(x, y) for x, y in zip(_planes(c), before))
