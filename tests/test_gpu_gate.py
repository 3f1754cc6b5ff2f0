"""GPU parity of the gate support (WitCert Sec. 6.3.5 block-level paging; Sec. 6.1 "Gate") via the C ABI.

kvq_decode_attn_ex writes, per (sequence, query head, page), ln sum_{t in page} e^{x_t} (e^{c_t} - 1);
exp(value - lse) is the page's contribution to A - 1.  kvq_gate turns them into the shortest greedy
page-in list; kvq_zero_witness zeroes repaired slots.  Bars: contributions close to the oracle
(relative, pages above 1e-7 of the total) and summing to A - 1 within 1e-4; the plan is sorted by contribution
and is the shortest prefix of that order reaching the meter target; zeroing a page's witness removes
exactly that page's contribution from A - 1.
(Contributions: 5e-4 relative, see the comment at the check.)
"""
import math

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import workloads as W  # noqa: E402
from oracle import attention as OA  # noqa: E402
from oracle.encoders import fp16_value  # noqa: E402
from oracle.meter import page_log_contrib  # noqa: E402
from tests.parity import SM_SCALE, make_inputs, reference_case  # noqa: E402

CASES = {
    "tiny": lambda: W.reduced(W.WORKLOADS["tiny"], seq_len=300),
    "cartridge": lambda: W.reduced(W.WORKLOADS["qwen3_8b_cartridge"], batch=2, seq_len=150),
    "int8_massive": lambda: W.reduced(W.WORKLOADS["int8_7b_certified"], batch=2, seq_len=333, massive_pairs=4,
                                      massive_scale=30.0),
    "ragged": lambda: W.reduced(W.WORKLOADS["ragged_paged"], batch=3, ragged=(40, 700)),
}


@pytest.fixture(scope="module")
def kvq():
    import quantized_kv_cache_kvq_gb300 as m

    m.load()
    return m


def _run(kvq, w, inp, zero_slots=None):
    from tests.parity import run_case_gpu  # builds the caches; reuse its steps here with the _ex entry

    dev = torch.device("cuda")
    B, Hkv, Hq = w.batch, w.n_kv_heads, w.n_q_heads
    g = run_case_gpu(w, inputs=inp, meter=True)  # fills caches (and checks the plain path runs)
    cache, prefix = g["cache"], g["prefix"]
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    if zero_slots is not None:
        kvq.zero_witness(cache, torch.from_numpy(zero_slots).to(dev), err)
    q = torch.from_numpy(inp["q"]).to(dev).to(torch.bfloat16 if w.q_dtype == "bf16" else torch.float32).contiguous()
    bt = torch.from_numpy(inp["bt"]).to(dev)
    lens = torch.from_numpy(inp["lens"].astype(np.int32)).to(dev)
    stride = (w.prefix_len + 15) // 16 + inp["bt"].shape[1]
    contrib = torch.full((B, Hq, stride), float("nan"), device=dev)
    out = torch.empty((B, Hq, 128), device=dev)
    ms = torch.empty((B, Hq, 8), device=dev)
    ws = torch.empty(kvq.decode_workspace_size(B, Hkv, Hq), dtype=torch.uint8, device=dev)
    mp = kvq.meter_params(kvq.TIER_A | (kvq.TIER_B if w.tier_b else 0), w.n_layers, Hq, w.n_steps, w.delta_req, w.tau)
    kvq.decode_attn_ex(cache, q, bt, lens, out, ws, prefix=prefix, prefix_len=w.prefix_len, sm_scale=SM_SCALE,
                       meter=mp, meter_state=ms, page_log_contrib=contrib, err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    return dict(contrib=contrib, ms=ms, lens=lens, cache=cache, out=out.cpu().numpy())


def _oracle_contrib(w, inp, ref, s, h):
    """Per-page log contributions of (sequence s, query head h): prefix pages, then live pages."""
    g = h // w.group
    q = inp["q"][s, h].astype(np.float64)
    parts = []
    rows = ref["rows"][s][1]
    if ref["prefix_rows"] is not None:
        pr = ref["prefix_rows"]
        x = SM_SCALE * (pr["kh"][:, g] @ q)
        c = OA.tier_a_radius(q, fp16_value(pr["w16"][:, g]), SM_SCALE)
        parts.append(page_log_contrib(x, c))
    x = SM_SCALE * (rows["kh"][:, g] @ q)
    c = OA.tier_a_radius(q, fp16_value(rows["w16"][:, g]), SM_SCALE)
    parts.append(page_log_contrib(x, c))
    return np.concatenate(parts)


@pytest.mark.parametrize("name", list(CASES))
def test_page_contributions_and_gate(kvq, name):
    w = CASES[name]()
    inp = make_inputs(w)
    ref = reference_case(w, inputs=inp)
    r = _run(kvq, w, inp)
    lc = r["contrib"].cpu().numpy().astype(np.float64)
    ms = r["ms"].cpu().numpy().astype(np.float64)
    for s in range(w.batch):
        P = (w.prefix_len + 15) // 16 + (int(inp["lens"][s]) + 15) // 16
        for h in range(w.n_q_heads):
            lse = ms[s, h, 2]
            got = np.exp(lc[s, h, :P] - lse)
            exp_ = np.exp(_oracle_contrib(w, inp, ref, s, h) - ref["lse"][s, h])
            total = max(exp_.sum(), 1e-300)
            big = exp_ > 1e-7 * total
            # a page's contribution is exp of a few logits, so it carries their absolute fp32 error (no
            # averaging as in ln(A - 1)): up to ~1e-4 when the INT8 scale is large (massive pairs, no bypass:
            # s ~ 0.7, fp32 sums of 128 products ~300), hence 5e-4 relative
            assert np.all(np.abs(got[big] - exp_[big]) <= 5e-4 * exp_[big])
            assert np.all(np.abs(got[~big] - exp_[~big]) <= 1e-7 * total)
            assert got.sum() == pytest.approx(math.exp(ms[s, h, 0]), rel=1e-4)
    # the plan
    tau = 1e-4 if name in ("cartridge", "tiny", "ragged") else 0.2
    B, Hq = w.batch, w.n_q_heads
    n_in = torch.empty((B, Hq), dtype=torch.int32, device="cuda")
    lst = torch.empty((B, Hq, 64), dtype=torch.int32, device="cuda")
    kvq.gate(r["contrib"], r["ms"], r["lens"], w.prefix_len, tau, n_in, lst)
    n_in, lst = n_in.cpu().numpy(), lst.cpu().numpy()
    target = math.sqrt(1 + 2 * tau) - 1
    any_work = False
    for s in range(B):
        P = (w.prefix_len + 15) // 16 + (int(inp["lens"][s]) + 15) // 16
        for h in range(Hq):
            c = np.exp(lc[s, h, :P] - ms[s, h, 2])
            am1 = math.exp(ms[s, h, 0])
            k = int(n_in[s, h])
            chosen = lst[s, h, :min(k, 64)]
            assert np.all(lst[s, h, min(k, 64):] == -1)
            if k <= 64:
                assert am1 - c[chosen].sum() <= target * (1 + 1e-5) + 1e-12            # reaches the target
                if k:
                    assert am1 - c[chosen[:-1]].sum() > target * (1 - 1e-5) - 1e-12   # and one fewer does not
                    assert np.all(np.diff(c[chosen]) <= 1e-6 * c[chosen[0]])           # in decreasing order
            any_work |= k > 0
    assert any_work


def test_zero_witness_removes_the_page_contribution(kvq):
    w = CASES["int8_massive"]()
    inp = make_inputs(w)
    before = _run(kvq, w, inp)
    page = 3  # live page 3 of sequence 0 (no prefix): zero its 16 slots for every kv head
    slots = W.slot_mapping(inp["bt"], 0, np.arange(16 * page, 16 * page + 16)).astype(np.int32)
    after = _run(kvq, w, inp, zero_slots=slots)
    b_lc, a_lc = before["contrib"].cpu().numpy(), after["contrib"].cpu().numpy()
    b_ms, a_ms = before["ms"].cpu().numpy().astype(np.float64), after["ms"].cpu().numpy().astype(np.float64)
    assert np.all(np.isneginf(a_lc[0, :, page]))
    assert np.array_equal(before["out"], after["out"])    # keys unchanged: same attention
    for h in range(w.n_q_heads):
        drop = math.exp(b_lc[0, h, page] - b_ms[0, h, 2])
        assert math.exp(a_ms[0, h, 0]) == pytest.approx(math.exp(b_ms[0, h, 0]) - drop, rel=1e-4)


def test_gate_plan_lengths_short_and_long(kvq):
    # kvq_gate alone on synthetic contributions, with A - 1 placed so that the shortest greedy prefix has a
    # chosen length per cell: 0 (already within tau), short plans, plans past the first 16 pages, and none
    # reaching the target (all pages).  Some contributions are exact duplicates (equal inputs), which must
    # come in page order.  Expected plans: the oracle's greedy page-in on the float64 contributions.
    from oracle.meter import greedy_page_in

    rng = np.random.default_rng(17)
    B, Hq, P = 2, 8, 300
    keys = rng.uniform(1.0, 3.0, size=(B, Hq, P))
    keys[:, :, 40:60] = keys[:, :, 20:40]               # duplicates: pages 40..59 equal pages 20..39
    lc = np.log(keys).astype(np.float32)
    k64 = np.exp(lc.astype(np.float64))                  # the contributions the kernel sees (lse = 0)
    tau = 1e-3
    target = math.sqrt(1 + 2 * tau) - 1                  # far below every contribution: no boundary is close
    want = [0, 1, 2, 3, 15, 16, 17, 40, 299, 300, 5, 16, 0, 33, 7, 300]
    am1 = np.empty((B, Hq))
    for cell, k in enumerate(want):
        s, h = divmod(cell, Hq)
        srt = np.sort(k64[s, h])[::-1]
        am1[s, h] = (srt[:k].sum() + 0.5 * target) if k < P else srt.sum() + 2.0
    state = np.zeros((B, Hq, 8), dtype=np.float32)
    state[..., 0] = np.log(am1)
    lens = torch.full((B,), P * 16, dtype=torch.int32, device="cuda")
    n_in = torch.empty((B, Hq), dtype=torch.int32, device="cuda")
    lst = torch.empty((B, Hq, 64), dtype=torch.int32, device="cuda")
    kvq.gate(torch.from_numpy(lc).cuda(), torch.from_numpy(state).cuda(), lens, 0, tau, n_in, lst)
    n_in, lst = n_in.cpu().numpy(), lst.cpu().numpy()
    for cell, k in enumerate(want):
        s, h = divmod(cell, Hq)
        # A - 1 as the kernel reads it (binary32 state)
        ref_k, ref_list = greedy_page_in(k64[s, h], float(np.exp(np.float64(state[s, h, 0]))), tau, max_pages=64)
        assert ref_k == k
        assert int(n_in[s, h]) == k, (cell, int(n_in[s, h]), k)
        m = min(k, 64)
        assert np.array_equal(lst[s, h, :m], ref_list[:m]), cell
        assert np.all(lst[s, h, m:] == -1)


def test_gate_plan_with_non_finite_contributions(kvq):
    # a NaN contribution (from non-finite inputs, which the decode reports) counts as none; -inf is an
    # empty page.  Cells: all NaN (no plan reaches the target: every page), half NaN, NaN next to -inf.
    from oracle.meter import greedy_page_in

    rng = np.random.default_rng(23)
    B, Hq, P = 1, 4, 40
    keys = rng.uniform(1.0, 3.0, size=(B, Hq, P))
    lc = np.log(keys).astype(np.float32)
    lc[0, 0, :] = np.nan
    lc[0, 1, ::2] = np.nan
    lc[0, 2, :5] = np.nan
    lc[0, 2, 5:10] = -np.inf
    k64 = np.exp(lc.astype(np.float64))
    k64[~np.isfinite(k64)] = 0.0   # NaN -> none, exp(-inf) = 0 already
    tau = 1e-3
    target = math.sqrt(1 + 2 * tau) - 1
    want = [P, 3, 4, 0]
    am1 = np.empty((B, Hq))
    for h, k in enumerate(want):
        srt = np.sort(k64[0, h])[::-1]
        am1[0, h] = (srt[:k].sum() + 0.5 * target) if h else 5.0
    state = np.zeros((B, Hq, 8), dtype=np.float32)
    state[..., 0] = np.log(am1)
    lens = torch.full((B,), P * 16, dtype=torch.int32, device="cuda")
    n_in = torch.empty((B, Hq), dtype=torch.int32, device="cuda")
    lst = torch.empty((B, Hq, 64), dtype=torch.int32, device="cuda")
    kvq.gate(torch.from_numpy(lc).cuda(), torch.from_numpy(state).cuda(), lens, 0, tau, n_in, lst)
    torch.cuda.synchronize()
    n_in, lst = n_in.cpu().numpy(), lst.cpu().numpy()
    for h, k in enumerate(want):
        ref_k, ref_list = greedy_page_in(k64[0, h], float(np.exp(np.float64(state[0, h, 0]))), tau, max_pages=64)
        assert ref_k == k and int(n_in[0, h]) == k, (h, int(n_in[0, h]), k)
        if h:  # with distinct finite keys the order is unique (the all-NaN cell ties every page)
            assert np.array_equal(lst[0, h, :k], ref_list[:k])
        assert np.all(lst[0, h, min(k, 64):] == -1)
