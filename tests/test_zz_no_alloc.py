"""kvq_decode_attn_noalloc: the decode entry point for callers that cannot allocate device scratch.

Some callers cannot call cudaMalloc for the decode workspace: a plugin or
embedding host that owns every device allocation and passes the library only
inputs and outputs, or a serving loop that forbids allocation on the request
path.  For them the library keeps its scratch in a file-scope device array.
This test calls that entry point through the C ABI twice in a row and checks
both results against the workspace-taking kvq_decode_attn on the same inputs
(same kernels, so the outputs match exactly, which is inside the 2e-3 / 1e-4
parity tolerances), and that an oversized request is refused.  It is collected
last and needs no state from other tests.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import workloads as W  # noqa: E402
from tests.parity import SM_SCALE, make_inputs  # noqa: E402


def _setup(kvq, w):
    inp = make_inputs(w, layer=0)
    dev = torch.device("cuda")
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    cache = kvq.PagedCache(w.k_fmt, w.v_fmt, w.n_kv_heads, inp["num_pages"], seed=inp["seed"], device=dev)
    for s in range(w.batch):
        k32, v32, _ = inp["seqs"][s]
        slots = W.slot_mapping(inp["bt"], s, np.arange(k32.shape[0]))
        kvq.append(cache, torch.from_numpy(k32).to(dev), torch.from_numpy(v32).to(dev),
                   torch.from_numpy(slots).to(dev), err)
    prefix = None
    if w.prefix_len:
        pk, pv = inp["prefix"]
        prefix = kvq.PagedCache(w.prefix_k_fmt, w.prefix_v_fmt, w.n_kv_heads, (w.prefix_len + 15) // 16,
                                seed=inp["prefix_seed"], device=dev)
        kvq.append(prefix, torch.from_numpy(pk).to(dev), torch.from_numpy(pv).to(dev),
                   torch.arange(w.prefix_len, dtype=torch.int32, device=dev), err)
    q = torch.from_numpy(inp["q"]).to(dev).to(torch.bfloat16 if w.q_dtype == "bf16" else torch.float32)
    return dict(cache=cache, prefix=prefix, q=q.contiguous(), bt=torch.from_numpy(inp["bt"]).to(dev),
                lens=torch.from_numpy(inp["lens"].astype(np.int32)).to(dev), err=err)


def test_noalloc_matches_workspace_entry_point_twice():
    import quantized_kv_cache_kvq_gb300 as kvq

    assert torch.cuda.is_available()
    kvq.load()
    w = W.reduced(W.WORKLOADS["qwen3_8b_cartridge"], batch=3, seq_len=333)
    c = _setup(kvq, w)
    B, Hq = w.batch, w.n_q_heads
    mp = kvq.meter_params(kvq.TIER_A, w.n_layers, Hq, w.n_steps, w.delta_req, w.tau)
    out_ref = torch.empty((B, Hq, 128), device="cuda")
    ms_ref = torch.empty((B, Hq, 8), device="cuda")
    ws = torch.empty(kvq.decode_workspace_size(B, w.n_kv_heads, Hq), dtype=torch.uint8, device="cuda")
    kvq.decode_attn(c["cache"], c["q"], c["bt"], c["lens"], out_ref, ws, prefix=c["prefix"], prefix_len=w.prefix_len,
                    sm_scale=SM_SCALE, meter=mp, meter_state=ms_ref, err=c["err"])
    for _ in range(2):
        out = torch.full((B, Hq, 128), float("nan"), device="cuda")
        ms = torch.full((B, Hq, 8), float("nan"), device="cuda")
        kvq.decode_attn_noalloc(c["cache"], c["q"], c["bt"], c["lens"], out, prefix=c["prefix"],
                                prefix_len=w.prefix_len, sm_scale=SM_SCALE, meter=mp, meter_state=ms, err=c["err"])
        torch.cuda.synchronize()
        assert c["err"].item() == 0
        o, r = out.cpu().numpy().astype(np.float64), out_ref.cpu().numpy().astype(np.float64)
        rel = np.linalg.norm(o - r, axis=-1) / np.linalg.norm(r, axis=-1)
        assert rel.max() <= 2e-3
        assert np.max(np.abs(ms.cpu().numpy()[..., 0] - ms_ref.cpu().numpy()[..., 0])) <= 1e-4
        assert np.array_equal(out.cpu().numpy(), out_ref.cpu().numpy())


def test_noalloc_rejects_oversized_request():
    import quantized_kv_cache_kvq_gb300 as kvq

    kvq.load()
    # a batch whose workspace exceeds the 16 MiB static scratch is refused before any launch
    B, Hkv, Hq = 1000, 8, 64
    assert kvq.decode_workspace_size(B, Hkv, Hq) > (16 << 20)
    cache = kvq.PagedCache("bf16", "e4m3s", Hkv, 1)
    q = torch.zeros((B, Hq, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((B, Hq, 128), device="cuda")
    with pytest.raises(kvq.KvqError) as e:
        kvq.decode_attn_noalloc(cache, q, torch.zeros((B, 1), dtype=torch.int32, device="cuda"),
                                torch.zeros(B, dtype=torch.int32, device="cuda"), out)
    assert e.value.status == 3  # KVQ_ERR_WORKSPACE_TOO_SMALL
