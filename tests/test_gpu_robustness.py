"""Graph capture, split-count invariance, determinism and the bounded-wait failure path (GPU).

* WitCert §6.2.1 acceptance: replaying a captured decode step is bit-identical to eager execution and
  interleaved replays agree exactly (the dither is keyed by cache coordinates, not by scheduling).
* WitCert §6.2.2: the split-KV merge gives the same result for any split; here the same sequences are
  decoded inside batches of different sizes (different piece boundaries) and must agree to rounding.
* Failure detection without a GPU fault: a wait that nothing completes reports KVQ_ERR_TIMEOUT through
  the error word after its wall-clock limit, and the next launch works.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import workloads as W  # noqa: E402
from tests.parity import SM_SCALE, make_inputs  # noqa: E402


@pytest.fixture(scope="module")
def kvq():
    import quantized_kv_cache_kvq_gb300 as m

    m.load()
    return m


def _cache_for(kvq, w, inp, dev):
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    cache = kvq.PagedCache(w.k_fmt, w.v_fmt, w.n_kv_heads, inp["num_pages"], seed=inp["seed"], device=dev)
    for s in range(len(inp["lens"])):
        k32, v32, _ = inp["seqs"][s]
        if k32.shape[0] == 0:
            continue
        slots = W.slot_mapping(inp["bt"], s, np.arange(k32.shape[0]))
        kvq.append(cache, torch.from_numpy(k32).to(dev), torch.from_numpy(v32).to(dev),
                   torch.from_numpy(slots).to(dev), err)
    return cache, err


# the INT8 and cartridge layouts run 12 warps per CTA with warp-uniform copy addresses; the raw FP8 layout runs 16
# warps with the predicated copy issue
GRAPH_CASES = {
    "int8": lambda: W.reduced(W.WORKLOADS["int8_7b_certified"], batch=2, seq_len=300, prefix_len=0),
    "cartridge": lambda: W.reduced(W.WORKLOADS["qwen3_8b_cartridge"], batch=2, seq_len=200),
    "fp8raw": lambda: W.reduced(W.WORKLOADS["fp8_raw_stress"], batch=2, seq_len=700),
}


@pytest.mark.parametrize("name", list(GRAPH_CASES))
def test_graph_replay_bit_identical_to_eager(kvq, name):
    w = GRAPH_CASES[name]()
    dev = torch.device("cuda")
    inp = make_inputs(w)
    cache, err = _cache_for(kvq, w, inp, dev)
    prefix = None
    if w.prefix_len:
        pk, pv = inp["prefix"]
        prefix = kvq.PagedCache(w.prefix_k_fmt, w.prefix_v_fmt, w.n_kv_heads, (w.prefix_len + 15) // 16,
                                seed=inp["prefix_seed"], device=dev)
        kvq.append(prefix, torch.from_numpy(pk).to(dev), torch.from_numpy(pv).to(dev),
                   torch.arange(w.prefix_len, dtype=torch.int32, device=dev), err)
    B, Hq = w.batch, w.n_q_heads
    q = torch.from_numpy(inp["q"]).to(dev).to(torch.bfloat16).contiguous()
    bt = torch.from_numpy(inp["bt"]).to(dev)
    lens = torch.from_numpy(inp["lens"].astype(np.int32)).to(dev)
    ws = torch.empty(kvq.decode_workspace_size(B, w.n_kv_heads, Hq), dtype=torch.uint8, device=dev)
    tiers = kvq.TIER_A | (kvq.TIER_B if w.tier_b else 0)
    mp = kvq.meter_params(tiers, w.n_layers, Hq, w.n_steps, w.delta_req, w.tau)
    out = torch.empty((B, Hq, 128), device=dev)
    ms = torch.empty((B, Hq, 8), device=dev)
    meter_a = torch.empty((1, B, Hq), device=dev)
    raw_a = torch.empty((1, B, Hq), device=dev)
    counts = torch.zeros(4, dtype=torch.int32, device=dev)
    # the new token of each sequence is re-appended every step (same slot, same values)
    k_new = torch.randn((B, w.n_kv_heads, 128), device=dev)
    v_new = torch.randn((B, w.n_kv_heads, 128), device=dev)
    last = np.array([W.slot_mapping(inp["bt"], s, [inp["lens"][s] - 1])[0] for s in range(B)], dtype=np.int32)
    slots = torch.from_numpy(last).to(dev)

    def step():
        kvq.append(cache, k_new, v_new, slots, err)
        kvq.decode_attn(cache, q, bt, lens, out, ws, prefix=prefix, prefix_len=w.prefix_len, sm_scale=SM_SCALE,
                        meter=mp, meter_state=ms, err=err)
        kvq.meter(ms.view(1, B, Hq, 8), 1, B, Hq, mp, meter_a, raw_a, counts)

    step()
    torch.cuda.synchronize()
    eager = [t.clone() for t in (out, ms, meter_a, raw_a, counts)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(5):
        for t in (out, ms, meter_a, raw_a):
            t.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        for a, b in zip((out, ms, meter_a, raw_a, counts), eager):
            assert torch.equal(a, b) or torch.equal(torch.nan_to_num(a), torch.nan_to_num(b))
        step()  # interleave an eager step
        torch.cuda.synchronize()
        assert torch.equal(out, eager[0])
    assert err.item() == 0


def test_split_count_invariance(kvq):
    """The same three sequences decoded alone and inside a 9-sequence batch: different piece splits."""
    dev = torch.device("cuda")
    w = W.reduced(W.WORKLOADS["ragged_paged"], batch=9, ragged=(300, 3000), random_pages=False)
    inp = make_inputs(w)
    cache, err = _cache_for(kvq, w, inp, dev)
    Hq, Hkv = w.n_q_heads, w.n_kv_heads
    mp = kvq.meter_params(kvq.TIER_A, 1, Hq, 256, 1e-2, 0.2)
    q_all = torch.from_numpy(inp["q"]).to(dev).to(torch.bfloat16).contiguous()

    def run(idx):
        B = len(idx)
        bt = torch.from_numpy(inp["bt"][idx]).to(dev)
        lens = torch.from_numpy(inp["lens"][idx].astype(np.int32)).to(dev)
        out = torch.empty((B, Hq, 128), device=dev)
        ms = torch.empty((B, Hq, 8), device=dev)
        ws = torch.empty(kvq.decode_workspace_size(B, Hkv, Hq), dtype=torch.uint8, device=dev)
        kvq.decode_attn(cache, q_all[idx].contiguous(), bt, lens, out, ws, sm_scale=SM_SCALE, meter=mp,
                        meter_state=ms, err=err)
        torch.cuda.synchronize()
        return out.cpu().numpy().astype(np.float64), ms.cpu().numpy().astype(np.float64)

    full_o, full_m = run(list(range(9)))
    for sub in ([2], [7], [0, 4, 8]):
        o, m = run(sub)
        ref_o, ref_m = full_o[sub], full_m[sub]
        rel = np.linalg.norm(o - ref_o, axis=-1) / np.linalg.norm(ref_o, axis=-1)
        # pieces round their softmax weights to fp16 against their own running max, so a different split
        # moves the output by float16 rounding noise only; a merge error would be O(1)
        assert rel.max() <= 2e-4, rel.max()
        assert np.max(np.abs(m[..., 0] - ref_m[..., 0])) <= 1e-4   # ln(A-1)
        assert np.max(np.abs(m[..., 2] - ref_m[..., 2])) <= 1e-5   # log-sum-exp
    assert err.item() == 0


def test_bounded_wait_reports_timeout_and_context_survives(kvq):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.debug_wait_timeout(50_000_000, err)  # 50 ms limit
    torch.cuda.synchronize()
    assert err.item() == 8  # KVQ_ERR_TIMEOUT
    # the context still runs kernels
    x = torch.arange(1024, device="cuda", dtype=torch.float32)
    out = torch.empty(1024, dtype=torch.int16, device="cuda")
    kvq.debug_encode(2, x, out)
    torch.cuda.synchronize()
    assert out.view(torch.float16).float().cpu().equal(x.cpu())


def test_page_index_range_refused(kvq):
    """Calls whose flattened (sequence, kv head, page) space would not fit 32-bit page indices are refused
    on the host (KVQ_ERR_INVALID_ARG) before any launch; the block table is never read."""
    import ctypes

    dev = torch.device("cuda")
    B, Hkv, Hq = 2, 8, 32
    cache = kvq.PagedCache("bf16", "bf16", Hkv, 4, device=dev)
    q = torch.zeros((B, Hq, 128), device=dev)
    out = torch.empty((B, Hq, 128), device=dev)
    bt = torch.zeros((B, 4), dtype=torch.int32, device=dev)
    lens = torch.ones(B, dtype=torch.int32, device=dev)
    ws = torch.empty(kvq.decode_workspace_size(B, Hkv, Hq), dtype=torch.uint8, device=dev)
    d = cache.desc()
    max_pages = (1 << 31) // (B * Hkv) + 1  # B * Hkv * max_pages > 2^31 - 1
    rc = kvq.lib().kvq_decode_attn(ctypes.byref(d), None, 0, q.data_ptr(), 0, B, Hq, bt.data_ptr(), max_pages,
                                   lens.data_ptr(), 1.0 / 128 ** 0.5, None, out.data_ptr(), None, ws.data_ptr(),
                                   ws.numel(), None, None)
    assert rc == 1  # KVQ_ERR_INVALID_ARG
    # a normal call on the same buffers still runs
    kvq.decode_attn(cache, q, bt, lens, out, ws)
    torch.cuda.synchronize()
