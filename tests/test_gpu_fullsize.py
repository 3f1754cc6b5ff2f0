"""Full-size parity: one layer of every workload at its full shape, in the launch configuration the
benchmark times (same grid, same persistent split plan, same workspace), checked on sampled
(sequence, kv head) units that the oracle recomputes one by one from the same binary32 inputs.

Sampled units include the first and last sequence, the longest and the shortest (ragged), so the
prefix/suffix boundary, partial last pages and random page permutations are all exercised.  Bar: the
append's K and V codes, K and V scales and witness of the sampled units are bit-exact (the shared
prefix's too); outputs within 2e-3 relative; ln(A - 1) (Tier A, and Tier B where enabled) within 1e-4;
meter never below the exact TV.
"""
import math

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import workloads as W  # noqa: E402
from oracle import attention as OA  # noqa: E402
from oracle.encoders import fp16_value  # noqa: E402
from tests.parity import SM_SCALE, oracle_cache_rows  # noqa: E402


def _host_planes(cache):
    return {n: (getattr(cache, n).cpu().numpy() if getattr(cache, n) is not None else None)
            for n in ("k", "v", "k_scale", "v_scale", "witness")}


def _check_stored(planes, num_pages, hkv, h, slots, k_fmt, v_fmt, rows):
    """Codes, scales and witness the GPU stored for kv head h at ``slots`` equal the oracle's ``rows``."""
    from quantized_kv_cache_kvq_gb300 import layout as L

    pg, t = slots // 16, slots % 16

    def head_tiles(plane, head_major):
        tiles = plane.reshape(hkv, num_pages, -1)[h] if head_major else plane.reshape(num_pages, hkv, -1)[:, h]
        return tiles.reshape(num_pages, -1)

    kc = L.unpack_k(head_tiles(planes["k"], False), k_fmt, 1)[pg, 0, t]
    vc = L.unpack_v(head_tiles(planes["v"], False), v_fmt, 1)[pg, 0, t]
    for got, ref in ((kc, rows["kc"][:, 0]), (vc, rows["vc"][:, 0])):
        assert np.array_equal(got, ref.view(got.dtype) if ref.dtype != got.dtype else ref)
    w16 = L.unpack_w(head_tiles(planes["witness"], False), 1)[pg, 0, t]
    assert np.array_equal(w16, rows["w16"][:, 0])
    for side, fmt in (("k", k_fmt), ("v", v_fmt)):
        ref = rows[f"{side}sb"]
        if ref is None:
            continue
        tiles = head_tiles(planes[f"{side}_scale"], True)
        got = (L.unpack_gs if fmt == "int8g32" else L.unpack_s)(tiles, 1)[pg, 0, t]
        assert np.array_equal(got, ref[:, 0])


def _sample_units(w, lens):
    B, H = w.batch, w.n_kv_heads
    seqs = {0, B - 1, int(np.argmax(lens)), int(np.argmin(lens))}
    return sorted({(s, (3 * s + 1) % H) for s in seqs})


@pytest.mark.parametrize("name", ["tiny", "qwen3_8b_cartridge", "int8_7b_certified", "fp8_raw_stress", "ragged_paged"])
def test_fullsize_sampled_parity(name):
    import quantized_kv_cache_kvq_gb300 as kvq
    from quantized_kv_cache_kvq_gb300 import layout as L

    kvq.load()
    w = W.WORKLOADS[name]
    dev = torch.device("cuda")
    layer = 3 if w.n_layers > 3 else 0
    lens = W.seq_lengths(w)
    bt = W.block_table_for(w, lens, layer)
    B, Hkv, Hq, G = w.batch, w.n_kv_heads, w.n_q_heads, w.group
    num_pages = int(((lens + 15) // 16).sum())
    seed = 0xBEEF0000 + 31 * w.wid + layer
    cache = kvq.PagedCache(w.k_fmt, w.v_fmt, Hkv, num_pages, layer=layer, seed=seed, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    g = torch.Generator(device=dev)
    g.manual_seed(W.unit_seed(w, 700_000 + layer))
    units = _sample_units(w, lens)
    keep = {s: None for s, _ in units}
    starts = np.concatenate([[0], np.cumsum(lens)])
    for s in range(B):
        n = int(lens[s])
        pos = torch.arange(w.prefix_len, w.prefix_len + n, device=dev)
        k, v = W.gen_tokens_gpu(w, layer, pos, g, dev)
        slots = W.slot_mapping(bt, s, np.arange(n))
        kvq.append(cache, k, v, torch.from_numpy(slots).to(dev), err)
        if s in keep:
            keep[s] = (k.cpu().numpy(), v.cpu().numpy(), slots)
        del k, v
    prefix = None
    pre = None
    if w.prefix_len:
        pseed = seed ^ 0x5A5A
        prefix = kvq.PagedCache(w.prefix_k_fmt, w.prefix_v_fmt, Hkv, (w.prefix_len + 15) // 16, layer=layer,
                                seed=pseed, device=dev)
        pk, pv = W.gen_tokens_gpu(w, layer, torch.arange(w.prefix_len, device=dev), g, dev, sink=True)
        kvq.append(prefix, pk, pv, torch.arange(w.prefix_len, dtype=torch.int32, device=dev), err)
        pre = (pk.cpu().numpy(), pv.cpu().numpy(), pseed)
    qd = torch.bfloat16 if w.q_dtype == "bf16" else torch.float32
    q = torch.randn((B, Hq, 128), generator=g, device=dev).to(qd).contiguous()
    out = torch.empty((B, Hq, 128), device=dev)
    ms = torch.empty((B, Hq, 8), device=dev)
    ws = torch.empty(kvq.decode_workspace_size(B, Hkv, Hq), dtype=torch.uint8, device=dev)
    tiers = kvq.TIER_A | (kvq.TIER_B if w.tier_b else 0)
    mp = kvq.meter_params(tiers, w.n_layers, Hq, w.n_steps, w.delta_req, w.tau)
    kvq.decode_attn(cache, q, torch.from_numpy(bt).to(dev), torch.from_numpy(lens.astype(np.int32)).to(dev), out, ws,
                    prefix=prefix, prefix_len=w.prefix_len, sm_scale=SM_SCALE, meter=mp, meter_state=ms, err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    out_h, ms_h = out.cpu().numpy().astype(np.float64), ms.cpu().numpy().astype(np.float64)
    q_h = q.float().cpu().numpy().astype(np.float64)
    planes = _host_planes(cache)
    if prefix is not None:   # the shared prefix's stored rows, every kv head
        pplanes = _host_planes(prefix)
        npp = (w.prefix_len + 15) // 16
        pslots = np.arange(w.prefix_len)
        for h in range(Hkv):
            prow = oracle_cache_rows(pre[0][:, h:h + 1], pre[1][:, h:h + 1], pslots, w.prefix_k_fmt, w.prefix_v_fmt,
                                     pre[2], layer, heads=[h])
            _check_stored(pplanes, npp, Hkv, h, pslots, w.prefix_k_fmt, w.prefix_v_fmt, prow)
    for s, h in units:
        k32, v32, slots = keep[s]
        k1, v1 = k32[:, h:h + 1], v32[:, h:h + 1]
        rows = oracle_cache_rows(k1, v1, slots, w.k_fmt, w.v_fmt, seed, layer, heads=[h])
        # append bit-exactness on the sampled unit: codes, scales, witness
        _check_stored(planes, num_pages, Hkv, h, slots, w.k_fmt, w.v_fmt, rows)
        kk, kh, vh, ww = k1[:, 0], rows["kh"][:, 0], rows["vh"][:, 0], fp16_value(rows["w16"][:, 0])
        sk = fp16_value(rows["ksb"][:, 0]) if rows["ksb"] is not None else None
        if pre is not None:
            prow = oracle_cache_rows(pre[0][:, h:h + 1], pre[1][:, h:h + 1], np.arange(w.prefix_len), w.prefix_k_fmt,
                                     w.prefix_v_fmt, pre[2], layer, heads=[h])
            kk = np.concatenate([pre[0][:, h], kk])
            kh = np.concatenate([prow["kh"][:, 0], kh])
            vh = np.concatenate([prow["vh"][:, 0], vh])
            ww = np.concatenate([fp16_value(prow["w16"][:, 0]), ww])
        tb = dict(delta_req=w.delta_req, n_layers=w.n_layers, n_q_heads=w.n_q_heads, n_steps=w.n_steps) \
            if w.tier_b else None
        r = OA.decode_head(q_h[s, h * G:(h + 1) * G], kk, kh, vh, ww, SM_SCALE, s_k=sk, tier_b=tb)
        got = out_h[s, h * G:(h + 1) * G]
        rel = np.linalg.norm(got - r.out, axis=-1) / np.linalg.norm(r.out, axis=-1)
        assert rel.max() <= 2e-3, (s, h, rel.max())
        la = ms_h[s, h * G:(h + 1) * G, 0]
        assert np.max(np.abs(la - r.log_am1_a)) <= 1e-4, (s, h, la, r.log_am1_a)
        assert np.all(OA.meter_from_log_am1(la) >= r.tv)
        assert np.allclose(ms_h[s, h * G:(h + 1) * G, 3], kk.shape[0])
        if w.tier_b:
            lb = ms_h[s, h * G:(h + 1) * G, 1]
            assert np.max(np.abs(lb - r.log_am1_b)) <= 1e-4, (s, h, lb, r.log_am1_b)
