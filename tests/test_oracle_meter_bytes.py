"""Pins of the oracle's meter finalisation, ranking and byte account (CPU)."""
import json
import math
import os

import numpy as np
import pytest

from oracle import bytes as B
from oracle import meter as M

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_finalize_closed_forms():
    # A = 1.1: meter = 1/2 (1.21 - 1) = 0.105
    meter, raw = M.finalize(np.array([math.log(0.1), -np.inf, 0.0, 700.0]))
    assert meter[0] == pytest.approx(0.105, rel=1e-14)
    assert raw[0] == pytest.approx(math.log(0.105), rel=1e-14)
    assert meter[1] == 0.0 and raw[1] == -np.inf
    assert meter[2] == 1.0 and raw[2] == pytest.approx(math.log(1.5), rel=1e-14)
    assert meter[3] == 1.0 and raw[3] == pytest.approx(1400 - math.log(2), rel=1e-14)


def test_coverage_counts_strictly_below_tau():
    m = np.array([0.0, 0.19999, 0.2, 0.5, np.nan, 1.0])
    assert M.coverage(m, 0.2) == 2
    assert M.coverage(m, 1.0) == 4


def test_rank_cells_matches_brute_force_with_ties():
    rng = np.random.default_rng(3)
    raw = np.round(rng.standard_normal((3, 4, 5)), 1)   # many exact ties
    raw[1, 2, 3] = np.nan
    out = M.rank_cells(raw)
    for b in range(3):
        flat = raw[b].reshape(-1)
        key = [(-(np.inf if np.isnan(v) else v), i) for i, v in enumerate(flat)]
        assert list(out[b]) == [i for _, i in sorted(key)]


def test_page2_byte_table():
    g = json.load(open(os.path.join(GOLD, "byte_table.json")))
    m = g["model"]
    for row in g["rows"]:
        per_tok = B.payload_bytes_per_token(row["k"], row["v"], m["n_layers"], m["n_kv_heads"], m["head_dim"])
        assert per_tok == row["kib_per_token"] * 1024
        assert round(per_tok * g["full_tokens"] / 2**30, 3) == row["gib_full"]
        assert round(per_tok * g["cartridge_tokens"] / 2**20, 3) == row["mib_cartridge"]
    full = B.payload_bytes_per_token("bf16", "bf16", 36, 8) * 632 / 2**20
    k16v8 = B.payload_bytes_per_token("bf16", "e4m3", 36, 8) * 632 / 2**20
    assert round(full - k16v8, 3) == g["k16v8_saving_mib_printed"]


def test_decode_bytes_per_token_head():
    # codes + scales + 32-byte witness (WitCert §4.1: 2B = 32 bytes per token per head at B = 16)
    assert B.kv_bytes_per_token_head("bf16", "e4m3s") == 256 + 128 + 2 + 32
    assert B.kv_bytes_per_token_head("bf16", "bf16") == 512 + 32
    assert B.kv_bytes_per_token_head("int8", "int8") == 256 + 4 + 32
    assert B.kv_bytes_per_token_head("e4m3", "e4m3") == 256 + 32
    assert B.kv_bytes_per_token_head("bf16", "bf16", meter=False) == 512
