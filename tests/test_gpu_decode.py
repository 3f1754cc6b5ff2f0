"""GPU parity of kvq_decode_attn (+ fused meter) against the oracle on reduced workloads.

Bar (spec tolerances): output within 2e-3 relative per (sequence, head)
(max over cells of ||o_gpu - o_ref|| / ||o_ref||); ln(A - 1) within 1e-4
absolute (= 1e-4 relative on A - 1) for Tier A and Tier B; the meter never
below the oracle's exact TV.  Sizes span several pages per warp, partial last
pages, a shared prefix whose end is not page aligned, ragged lengths with a
random page permutation, and GQA groups of 4 and 7.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import workloads as W  # noqa: E402
from tests.parity import make_inputs, reference_case, run_case_gpu  # noqa: E402

CASES = {
    "tiny": W.WORKLOADS["tiny"],
    "cartridge": W.reduced(W.WORKLOADS["qwen3_8b_cartridge"], batch=3, seq_len=333),
    "int8": W.reduced(W.WORKLOADS["int8_7b_certified"], batch=3, seq_len=517),
    "fp8raw": W.reduced(W.WORKLOADS["fp8_raw_stress"], batch=2, seq_len=901),
    "ragged": W.reduced(W.WORKLOADS["ragged_paged"], batch=7, ragged=(17, 2500)),
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


@pytest.mark.parametrize("name", list(CASES))
def test_decode_parity(kvq, name):
    w = CASES[name]
    inp = make_inputs(w, layer=1)
    gpu = run_case_gpu(w, layer=1, inputs=inp)
    ref = reference_case(w, layer=1, inputs=inp)
    _check(w, gpu, ref)


def test_meter_off_output_bit_identical(kvq):
    w = CASES["cartridge"]
    inp = make_inputs(w, layer=0)
    on = run_case_gpu(w, inputs=inp, meter=True)
    off = run_case_gpu(w, inputs=inp, meter=False)
    assert np.array_equal(on["out"], off["out"])


def test_fp32_query_path(kvq):
    w = W.reduced(W.WORKLOADS["tiny"], seq_len=300, q_dtype="f32")
    inp = make_inputs(w)
    gpu = run_case_gpu(w, inputs=inp)
    _check(w, gpu, reference_case(w, inputs=inp))
    w8 = W.reduced(CASES["fp8raw"], q_dtype="f32")
    inp = make_inputs(w8)
    gpu = run_case_gpu(w8, inputs=inp)
    _check(w8, gpu, reference_case(w8, inputs=inp))
    # dithered INT8 with Tier B: the key products add the query's low part, the dither products and their
    # 9/2 sum_c q_c start value use the high part
    wi = W.reduced(CASES["int8"], q_dtype="f32")
    inp = make_inputs(wi)
    gpu = run_case_gpu(wi, inputs=inp)
    _check(wi, gpu, reference_case(wi, inputs=inp))
    # shared K16/V8 prefix + BF16 suffix: both segments' page bodies with the low-part products
    wc = W.reduced(CASES["cartridge"], q_dtype="f32")
    inp = make_inputs(wc)
    gpu = run_case_gpu(wc, inputs=inp)
    _check(wc, gpu, reference_case(wc, inputs=inp))


def test_empty_and_single_token_sequences(kvq):
    w = W.reduced(W.WORKLOADS["ragged_paged"], batch=4, ragged=(1, 40))
    inp = make_inputs(w)
    lens = np.array([0, 1, 17, 0], dtype=np.int64)
    inp["seqs"] = [W.gen_unit_cpu(w, s, 0, int(n)) for s, n in enumerate(lens)]
    inp["q"] = np.stack([sq[2] for sq in inp["seqs"]])
    inp["lens"] = lens
    inp["bt"] = W.identity_block_table(lens, 2)
    inp["num_pages"] = int(((lens + 15) // 16).sum())
    gpu = run_case_gpu(w, inputs=inp)
    ref = reference_case(w, inputs=inp)
    assert gpu["err"] == 0
    assert np.all(gpu["out"][[0, 3]] == 0.0)
    assert np.all(np.isneginf(gpu["log_am1"][[0, 3]]))
    sel = [1, 2]
    rel = np.linalg.norm(gpu["out"][sel] - ref["out"][sel], axis=-1) / np.linalg.norm(ref["out"][sel], axis=-1)
    assert rel.max() <= 2e-3


# one 12-warp layout with branch-issued copies (tiny), one with warp-uniform descriptors (INT8), and the 16-warp
# raw FP8 layout, whose copy issue predicates the invalid page instead of branching around it
BAD_BT_CASES = {
    "tiny": lambda: W.reduced(W.WORKLOADS["tiny"], seq_len=64),
    "int8": lambda: W.reduced(W.WORKLOADS["int8_7b_certified"], batch=2, seq_len=96),
    "fp8raw": lambda: W.reduced(W.WORKLOADS["fp8_raw_stress"], batch=2, seq_len=96),
}


@pytest.mark.parametrize("name", list(BAD_BT_CASES))
def test_bad_block_table_reported(kvq, name):
    w = BAD_BT_CASES[name]()
    inp = make_inputs(w)
    inp["bt"] = inp["bt"].copy()
    inp["bt"][0, 2] = 10_000  # beyond the cache
    gpu = run_case_gpu(w, inputs=inp)
    assert gpu["err"] == 5  # KVQ_ERR_DEVICE_BOUNDS
    if w.batch > 1:
        # the other sequences are untouched by the skipped page
        ref = reference_case(w, inputs=inp)
        rel = np.linalg.norm(gpu["out"][1:] - ref["out"][1:], axis=-1) / np.linalg.norm(ref["out"][1:], axis=-1)
        assert rel.max() <= 2e-3


def test_workspace_too_small(kvq):
    import quantized_kv_cache_kvq_gb300 as m

    cache = m.PagedCache("bf16", "e4m3s", 8, 4)
    q = torch.zeros((1, 32, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((1, 32, 128), device="cuda")
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(m.KvqError) as e:
        m.decode_attn(cache, q, torch.zeros((1, 4), dtype=torch.int32, device="cuda"),
                      torch.tensor([60], dtype=torch.int32, device="cuda"), out, ws)
    assert e.value.status == 3
