"""kvq_decode_attn_append: the decode step's append and attention in one call (GPU).

The append of each sequence's newest token runs as its own grid, which the decode overlaps and waits
for only before loading the pages that hold those tokens.  The fused call must leave the cache
byte-identical to kvq_append of the same tokens (WitCert Sec. 6.2.1: the write side and the read
side share one dither stream and one stored form) in every plane, the value witness included, and
its outputs and meter state (value side on) must equal those of kvq_append followed by
kvq_decode_attn bit for bit.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import workloads as W  # noqa: E402
from tests.parity import SM_SCALE, make_inputs, reference_case  # noqa: E402

CASES = {
    "cartridge": lambda: W.reduced(W.WORKLOADS["qwen3_8b_cartridge"], batch=3, seq_len=77),
    "int8": lambda: W.reduced(W.WORKLOADS["int8_7b_certified"], batch=3, seq_len=150),
    "int8g32": lambda: W.reduced(W.WORKLOADS["int8_7b_certified"], batch=3, seq_len=150, k_fmt="int8g32",
                                 v_fmt="int8g32"),
    "fp8raw": lambda: W.reduced(W.WORKLOADS["fp8_raw_stress"], batch=2, seq_len=100),
    "ragged": lambda: W.reduced(W.WORKLOADS["ragged_paged"], batch=5, ragged=(1, 300)),
}


@pytest.fixture(scope="module")
def kvq():
    import quantized_kv_cache_kvq_gb300 as m

    m.load()
    return m


def _inputs(name):
    w = CASES[name]()
    inp = make_inputs(w)
    if name == "ragged":  # an empty sequence and a single-token one
        lens = inp["lens"].copy()
        lens[1], lens[3] = 0, 1
        inp["seqs"] = [W.gen_unit_cpu(w, s, 0, int(n)) for s, n in enumerate(lens)]
        inp["q"] = np.stack([sq[2] for sq in inp["seqs"]])
        inp["lens"] = lens
        inp["bt"] = W.block_table_for(w, lens)
        inp["num_pages"] = max(1, int(((lens + 15) // 16).sum()))
    return w, inp


def _run(kvq, w, inp, fused):
    dev = torch.device("cuda")
    B, Hkv, Hq = w.batch, w.n_kv_heads, w.n_q_heads
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    cache = kvq.PagedCache(w.k_fmt, w.v_fmt, Hkv, inp["num_pages"], seed=inp["seed"], device=dev, value_witness=True)
    k_new = torch.zeros((B, Hkv, 128), device=dev)
    v_new = torch.zeros((B, Hkv, 128), device=dev)
    for s in range(B):
        k32, v32, _ = inp["seqs"][s]
        n = k32.shape[0]
        if n == 0:
            continue
        upto = n - 1 if fused else n
        if upto:
            slots = W.slot_mapping(inp["bt"], s, np.arange(upto))
            kvq.append(cache, torch.from_numpy(k32[:upto]).to(dev), torch.from_numpy(v32[:upto]).to(dev),
                       torch.from_numpy(slots).to(dev), err)
        k_new[s] = torch.from_numpy(k32[n - 1]).to(dev)
        v_new[s] = torch.from_numpy(v32[n - 1]).to(dev)
    prefix = None
    if w.prefix_len:
        pk, pv = inp["prefix"]
        prefix = kvq.PagedCache(w.prefix_k_fmt, w.prefix_v_fmt, Hkv, (w.prefix_len + 15) // 16,
                                seed=inp["prefix_seed"], device=dev, value_witness=True)
        kvq.append(prefix, torch.from_numpy(pk).to(dev), torch.from_numpy(pv).to(dev),
                   torch.arange(w.prefix_len, dtype=torch.int32, device=dev), err)
    q = torch.from_numpy(inp["q"]).to(dev).to(torch.bfloat16 if w.q_dtype == "bf16" else torch.float32).contiguous()
    bt = torch.from_numpy(inp["bt"]).to(dev)
    lens = torch.from_numpy(inp["lens"].astype(np.int32)).to(dev)
    out = torch.full((B, Hq, 128), float("nan"), device=dev)
    ms = torch.full((B, Hq, 8), float("nan"), device=dev)
    ws = torch.empty(kvq.decode_workspace_size(B, Hkv, Hq), dtype=torch.uint8, device=dev)
    mp = kvq.meter_params(kvq.TIER_A | kvq.TIER_V | (kvq.TIER_B if w.tier_b else 0), w.n_layers, Hq, w.n_steps,
                          w.delta_req, w.tau)
    kw = dict(prefix=prefix, prefix_len=w.prefix_len, sm_scale=SM_SCALE, meter=mp, meter_state=ms, err=err)
    if fused:
        kvq.decode_attn_append(cache, k_new, v_new, q, bt, lens, out, ws, **kw)
    else:
        kvq.decode_attn(cache, q, bt, lens, out, ws, **kw)
    torch.cuda.synchronize()
    planes = [t.cpu().numpy() for t in (cache.k, cache.v, cache.k_scale, cache.v_scale, cache.witness, cache.v_witness)
              if t is not None]
    return dict(err=int(err.item()), planes=planes, out=out.cpu().numpy(), ms=ms.cpu().numpy())


@pytest.mark.parametrize("name", list(CASES))
def test_fused_append_equals_append_then_decode(kvq, name):
    w, inp = _inputs(name)
    a = _run(kvq, w, inp, fused=True)
    b = _run(kvq, w, inp, fused=False)
    assert a["err"] == 0 and b["err"] == 0
    for pa, pb in zip(a["planes"], b["planes"]):
        assert np.array_equal(pa, pb)
    assert np.array_equal(a["out"], b["out"], equal_nan=True)
    assert np.array_equal(a["ms"], b["ms"], equal_nan=True)
    if name == "int8":  # and the fused call against the oracle
        ref = reference_case(w, inputs=inp)
        rel = np.linalg.norm(a["out"] - ref["out"], axis=-1) / np.linalg.norm(ref["out"], axis=-1)
        assert rel.max() <= 2e-3


def test_fused_append_reports_nonfinite(kvq):
    w, inp = _inputs("cartridge")
    k32, v32, _ = inp["seqs"][1]
    k32 = k32.copy()
    k32[-1, 2, 5] = np.inf
    inp["seqs"][1] = (k32, v32, inp["seqs"][1][2])
    a = _run(kvq, w, inp, fused=True)
    assert a["err"] == 6  # KVQ_ERR_NONFINITE_INPUT
