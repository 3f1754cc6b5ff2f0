"""The bench's algorithmic byte counts, checked against the oracle's byte account (CPU).

Every GB/s figure of bench.py divides these bytes by a time, so they are pinned here against:
* the oracle's per-(token, kv head) account (codes, fp16 scales, the 32-byte witness), for every
  layout pair, and its per-step account (live tokens once per layer and kv head, the shared prefix
  once per layer) on every workload;
* the page's payload table ("Compress the shared cartridge", 144 / 108 / 72 KiB per token for
  36 layers x 8 kv heads x d = 128), through the bench's own code-byte table;
* the optional planes: the 4-byte value witness and the fp16 key outlier tile (8 columns for up to
  4 bypassed pairs, 16 for up to 8).
"""
import json
import os

import pytest

import bench
import workloads as W
from oracle import bytes as OB

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "byte_table.json")
FMTS = ("bf16", "e4m3", "e4m3s", "int8")


@pytest.mark.parametrize("k_fmt", FMTS)
@pytest.mark.parametrize("v_fmt", FMTS)
def test_token_head_bytes_match_the_oracle(k_fmt, v_fmt):
    assert bench.token_head_bytes(k_fmt, v_fmt) == OB.kv_bytes_per_token_head(k_fmt, v_fmt, meter=True)
    assert bench.token_head_bytes(k_fmt, v_fmt, meter=False) == OB.kv_bytes_per_token_head(k_fmt, v_fmt, meter=False)
    base = bench.token_head_bytes(k_fmt, v_fmt)
    assert bench.token_head_bytes(k_fmt, v_fmt, value_side=True) == base + 4        # (rho^v, ||v||) fp16
    for m, extra in ((1, 16), (4, 16), (5, 32), (8, 32)):                            # 8 or 16 fp16 columns
        assert bench.token_head_bytes(k_fmt, v_fmt, bypass=m) == base + extra


def test_bytes_per_token_head_of_each_layout():
    # K16/V8 418 B, BF16/BF16 544 B, INT8-dither 292 B, K8/V8 raw 288 B (witness and scales included)
    assert bench.token_head_bytes("bf16", "e4m3s") == 418
    assert bench.token_head_bytes("bf16", "bf16") == 544
    assert bench.token_head_bytes("int8", "int8") == 292
    assert bench.token_head_bytes("e4m3", "e4m3") == 288


def test_group_scaled_int8_bytes():
    # one fp16 scale per token per 32-channel group: 136 B per side (WitCert 6.2.3), plus the 32-byte witness
    assert bench.token_head_bytes("int8g32", "int8g32", meter=False) == 2 * OB.int8_side_bytes("token", group=32) == 272
    assert bench.token_head_bytes("int8g32", "int8g32") == OB.kv_bytes_per_token_head("int8g32", "int8g32") == 304
    w = W.reduced(W.WORKLOADS["int8_7b_certified"], k_fmt="int8g32", v_fmt="int8g32")
    lens = W.seq_lengths(w)
    assert bench.step_bytes(w, lens) == OB.decode_step_bytes(w.batch, w.n_layers, w.n_kv_heads, lens, "int8g32",
                                                             "int8g32")


def test_payload_table_of_the_page():
    g = json.load(open(GOLDEN))
    L, H, d = g["model"]["n_layers"], g["model"]["n_kv_heads"], g["model"]["head_dim"]
    for row in g["rows"]:
        payload = L * H * d * (bench.CODE_BYTES[row["k"]] + bench.CODE_BYTES[row["v"]])
        assert payload == row["kib_per_token"] * 1024, row["layout"]
        assert payload == OB.payload_bytes_per_token(row["k"], row["v"], L, H, d)


@pytest.mark.parametrize("name", sorted(W.WORKLOADS))
def test_step_bytes_match_the_oracle(name):
    w = W.WORKLOADS[name]
    lens = W.seq_lengths(w)
    want = OB.decode_step_bytes(w.batch, w.n_layers, w.n_kv_heads, lens, w.k_fmt, w.v_fmt, w.prefix_len,
                                w.prefix_k_fmt, w.prefix_v_fmt)
    assert bench.step_bytes(w, lens) == want


def test_cartridge_step_is_30_gb():
    w = W.WORKLOADS["qwen3_8b_cartridge"]
    b = bench.step_bytes(w, W.seq_lengths(w))
    # 36 x (16 x 11,996 x 8 x 544 + 632 x 8 x 418) bytes
    assert b == 36 * (16 * 11996 * 8 * 544 + 632 * 8 * 418)
    assert round(b / 1e9, 2) == 30.15
