"""Parity harness: one seeded decode case through the C ABI (GPU) and through the oracle (CPU).

The inputs come from ``workloads`` (seeded, shared by both sides); the oracle
never sees a value the CUDA path produced, and the CUDA path never calls the
oracle.  A case is one layer of a (possibly reduced) workload: every sequence's
suffix tokens (and the shared prefix, if any) are appended with kvq_append,
then kvq_decode_attn and kvq_meter run once.
"""
from __future__ import annotations

import math

import numpy as np

import workloads as W
from oracle import attention as OA
from oracle.encoders import fp16_value
from oracle.philox import dither
from oracle.quant import (bypass_channels, dequantize, dequantize_int8_bypass, dequantize_int8_groups, quantize,
                          quantize_int8_bypass, quantize_int8_groups, value_witness_bits, witness_bits)

SM_SCALE = float(np.float32(1.0 / math.sqrt(128)))
PREFIX_SEED_UNIT = 777_777


def cache_seed(w, layer: int) -> int:
    return (0x5EED_0000_0000 + w.wid * 1_000_003 + layer) & 0xFFFFFFFFFFFFFFFF


def make_inputs(w, layer: int = 0):
    """Seeded binary32 inputs of one layer, plus the paging structure."""
    lens = W.seq_lengths(w)
    B, Hkv = w.batch, w.n_kv_heads
    seqs = []
    for s in range(B):
        k, v, q = W.gen_unit_cpu(w, s, layer, int(lens[s]), first_pos=w.prefix_len)
        seqs.append((k, v, q))
    pages = (lens + W.PAGE - 1) // W.PAGE
    max_pages = max(1, int(pages.max(initial=1)))
    if w.random_pages:
        bt = W.permuted_block_table(lens, W.unit_seed(w, 424_242 + layer), max_pages)
    else:
        bt = W.identity_block_table(lens, max_pages)
    num_pages = int(pages.sum())
    pre = None
    if w.prefix_len:
        pk, pv, _ = W.gen_unit_cpu(w, 0, layer, w.prefix_len, first_pos=0, seed_unit=PREFIX_SEED_UNIT + layer)
        pre = (pk, pv)
    q = np.stack([sq[2] for sq in seqs]) if B else np.zeros((0, w.n_q_heads, 128), np.float32)
    pairs = W.bypass_pair_table(w, layer) if w.bypass_pairs else None
    return dict(lens=lens, seqs=seqs, bt=bt, num_pages=max(num_pages, 1), prefix=pre, q=q, layer=layer,
                seed=cache_seed(w, layer), prefix_seed=cache_seed(w, 10_000 + layer), pairs=pairs)


def _oracle_quant_rows(x32, fmt, xi):
    if fmt == "int8g32":   # one scale per token per 32-channel group: sb [..., 4]
        codes, sb, valid = quantize_int8_groups(x32, xi, group=32)
        return codes, sb, dequantize_int8_groups(codes, sb, xi), valid
    codes, sb, valid = quantize(x32, fmt, xi if fmt == "int8" else None)
    xh = dequantize(codes, sb, fmt, xi if fmt == "int8" else None)
    return codes, sb, xh, valid


def oracle_cache_rows(k32, v32, slots, k_fmt, v_fmt, seed, layer, heads=None, pairs=None):
    """Oracle quantization of tokens [n, Hkv, 128] written at ``slots`` [n].

    ``heads``: kv-head index of each column of the inputs (defaults to 0..Hkv-1); it keys the dither.
    ``pairs``: [Hkv, m] fixed-channel bypass of INT8 keys (per column of the inputs), or None."""
    n, Hkv, _ = k32.shape
    heads = (np.arange(Hkv) if heads is None else np.asarray(heads))[None, :, None]
    xi = dither(seed, layer, heads, np.asarray(slots)[:, None, None], np.arange(128)[None, None, :])
    kob = None
    if pairs is not None and np.asarray(pairs).shape[1] > 0:
        assert k_fmt == "int8"
        m = np.asarray(pairs).shape[1]
        kc = np.zeros((n, Hkv, 128), np.int8)
        ksb = np.zeros((n, Hkv), np.uint16)
        kh = np.zeros((n, Hkv, 128))
        kob = np.zeros((n, Hkv, 2 * m), np.uint16)
        kval = np.ones((n, Hkv), bool)
        for h in range(Hkv):
            c_, s_, o_, v_ = quantize_int8_bypass(k32[:, h], xi[:, h], pairs[h])
            kc[:, h], ksb[:, h], kob[:, h], kval[:, h] = c_, s_, o_, v_
            kh[:, h] = dequantize_int8_bypass(c_, s_, o_, xi[:, h], pairs[h])
    else:
        kc, ksb, kh, kval = _oracle_quant_rows(k32, k_fmt, xi)
    vc, vsb, vh, vval = _oracle_quant_rows(v32, v_fmt, xi)
    w16 = witness_bits(kh, k32)
    vw16 = value_witness_bits(vh, v32)
    return dict(kc=kc, ksb=ksb, kh=kh, vc=vc, vsb=vsb, vh=vh, w16=w16, vw16=vw16, kob=kob, valid=kval & vval)


def reference_case(w, layer: int = 0, inputs=None, tier_b: bool | None = None):
    """Oracle results of the case: per (seq, q head) out, lse, TV, ln(A-1), meter, Tier B."""
    inp = inputs or make_inputs(w, layer)
    tier_b = w.tier_b if tier_b is None else tier_b
    B, Hkv, G = w.batch, w.n_kv_heads, w.group
    pre_rows = None
    if inp["prefix"] is not None:
        pk, pv = inp["prefix"]
        pre_rows = oracle_cache_rows(pk, pv, np.arange(w.prefix_len), w.prefix_k_fmt, w.prefix_v_fmt,
                                     inp["prefix_seed"], layer)
    res = {k: np.zeros((B, w.n_q_heads) + sh) for k, sh in
           (("out", (128,)), ("lse", ()), ("tv", ()), ("log_am1", ()), ("meter", ()), ("raw", ()),
            ("log_am1_b", ()), ("cert_b", ()), ("value_r", ()), ("value_vmax", ()), ("out_bound", ()),
            ("out_err", ()), ("c_max", ()), ("om", ()), ("meter_2s", ()), ("meter_tanh", ()))}
    rows_all = []
    for s in range(B):
        k32, v32, q = inp["seqs"][s]
        n = k32.shape[0]
        slots = W.slot_mapping(inp["bt"], s, np.arange(n)) if n else np.zeros(0, np.int32)
        rows = oracle_cache_rows(k32, v32, slots, w.k_fmt, w.v_fmt, inp["seed"], layer, pairs=inp.get("pairs"))
        rows_all.append((slots, rows))
        for g in range(Hkv):
            kk, kh, vh, ww = k32[:, g], rows["kh"][:, g], rows["vh"][:, g], fp16_value(rows["w16"][:, g])
            vv, vw = v32[:, g], fp16_value(rows["vw16"][:, g])
            sk = fp16_value(rows["ksb"][:, g]) if rows["ksb"] is not None else None
            if pre_rows is not None:
                pk, pv = inp["prefix"]
                kk = np.concatenate([pk[:, g], kk])
                kh = np.concatenate([pre_rows["kh"][:, g], kh])
                vh = np.concatenate([pre_rows["vh"][:, g], vh])
                ww = np.concatenate([fp16_value(pre_rows["w16"][:, g]), ww])
                vv = np.concatenate([pv[:, g], vv])
                vw = np.concatenate([fp16_value(pre_rows["vw16"][:, g]), vw])
            qs = q[g * G:(g + 1) * G].astype(np.float64)
            S = kh.shape[0]
            if S == 0:
                res["log_am1"][s, g * G:(g + 1) * G] = -np.inf
                continue
            tb = dict(delta_req=w.delta_req, n_layers=w.n_layers, n_q_heads=w.n_q_heads,
                      n_steps=w.n_steps) if tier_b else None
            byp = None
            if rows["kob"] is not None:
                byp = dict(channels=bypass_channels(inp["pairs"][g]), values=fp16_value(rows["kob"][:, g]))
            r = OA.decode_head(qs, kk, kh, vh, ww, SM_SCALE, s_k=sk, tier_b=tb, vw=vw, v_exact=vv, bypass=byp)
            sl = slice(g * G, (g + 1) * G)
            res["out"][s, sl] = r.out
            res["lse"][s, sl] = r.lse
            res["tv"][s, sl] = r.tv
            res["log_am1"][s, sl] = r.log_am1_a
            res["meter"][s, sl] = r.meter_a
            res["raw"][s, sl] = r.raw_a
            res["log_am1_b"][s, sl] = r.log_am1_b
            res["cert_b"][s, sl] = r.cert_b
            res["value_r"][s, sl] = r.value_r
            res["value_vmax"][s, sl] = r.value_vmax
            res["out_bound"][s, sl] = r.out_bound_a
            res["out_err"][s, sl] = r.out_err
            res["c_max"][s, sl] = r.c_max
            res["om"][s, sl] = r.one_minus_a_minus
            res["meter_2s"][s, sl] = r.meter_two_sided
            res["meter_tanh"][s, sl] = r.meter_tanh
    res["rows"] = rows_all
    res["prefix_rows"] = pre_rows
    return res


def run_case_gpu(w, layer: int = 0, inputs=None, meter: bool = True, tier_b: bool | None = None,
                 q_dtype=None, device="cuda", value: bool = False, shapes: bool = False):
    """Append + decode (+ meter) of the case through the C ABI; returns host arrays and the caches."""
    import torch

    import quantized_kv_cache_kvq_gb300 as kvq

    inp = inputs or make_inputs(w, layer)
    tier_b = w.tier_b if tier_b is None else tier_b
    B, Hkv, Hq = w.batch, w.n_kv_heads, w.n_q_heads
    dev = torch.device(device)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    pairs = inp.get("pairs")
    cache = kvq.PagedCache(w.k_fmt, w.v_fmt, Hkv, inp["num_pages"], layer=layer, seed=inp["seed"], device=dev,
                           value_witness=value,
                           outlier_pairs=torch.from_numpy(pairs).to(dev) if pairs is not None else None)
    for s in range(B):
        k32, v32, _ = inp["seqs"][s]
        n = k32.shape[0]
        if n == 0:
            continue
        slots = W.slot_mapping(inp["bt"], s, np.arange(n))
        kvq.append(cache, torch.from_numpy(k32).to(dev), torch.from_numpy(v32).to(dev),
                   torch.from_numpy(slots).to(dev), err)
    prefix = None
    if inp["prefix"] is not None:
        pk, pv = inp["prefix"]
        npp = (w.prefix_len + W.PAGE - 1) // W.PAGE
        prefix = kvq.PagedCache(w.prefix_k_fmt, w.prefix_v_fmt, Hkv, npp, layer=layer, seed=inp["prefix_seed"],
                                device=dev, value_witness=value)
        kvq.append(prefix, torch.from_numpy(pk).to(dev), torch.from_numpy(pv).to(dev),
                   torch.arange(w.prefix_len, dtype=torch.int32, device=dev), err)
    qd = q_dtype or (torch.bfloat16 if w.q_dtype == "bf16" else torch.float32)
    q = torch.from_numpy(inp["q"]).to(dev).to(qd).contiguous()
    bt = torch.from_numpy(inp["bt"]).to(dev)
    lens = torch.from_numpy(inp["lens"].astype(np.int32)).to(dev)
    out = torch.empty((B, Hq, 128), dtype=torch.float32, device=dev)
    ms = torch.empty((B, Hq, 8), dtype=torch.float32, device=dev)
    ws = torch.empty(kvq.decode_workspace_size(B, Hkv, Hq), dtype=torch.uint8, device=dev)
    mp = None
    if meter:
        mp = kvq.meter_params(kvq.TIER_A | (kvq.TIER_B if tier_b else 0) | (kvq.TIER_V if value else 0)
                              | (kvq.TIER_S if shapes else 0), w.n_layers, w.n_q_heads, w.n_steps, w.delta_req, w.tau)
    kvq.decode_attn(cache, q, bt, lens, out, ws, prefix=prefix, prefix_len=w.prefix_len, sm_scale=SM_SCALE,
                    meter=mp, meter_state=ms if meter else None, err=err)
    res = dict(out=out.cpu().numpy().astype(np.float64), err=int(err.item()), cache=cache, prefix=prefix,
               inputs=inp)
    if meter:
        msn = ms.cpu().numpy().astype(np.float64)
        res["state"] = msn
        res["log_am1"] = msn[..., 0]
        res["log_am1_b"] = msn[..., 1]
        res["lse"] = msn[..., 2]
        res["meter"] = OA.meter_from_log_am1(msn[..., 0])
        res["value_r"] = msn[..., 4]
        res["value_vmax"] = msn[..., 5]
        res["c_max"] = msn[..., 6]
        res["om"] = msn[..., 7]
        res["mp"] = mp
        res["ms_dev"] = ms
    return res
