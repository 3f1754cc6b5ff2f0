"""Seeded synthetic decode workloads: shapes, value distributions and paging structure.

This module holds no arithmetic of the quantized-KV method.  It only builds
inputs -- pre-RoPE Gaussian keys, values and queries, the rotary embedding that
turns them into the binary32 post-RoPE keys the cache stores, block tables and
slot mappings -- and it is the one module the float64 oracle, the tests and
the benchmark share.

Workload recipe (all five shapes; the rotary embedding is applied in float64
and rounded once to binary32, which makes that binary32 key "the exact key"):

* pre-RoPE K, V and q are N(0, 1); RoPE theta = 1e6, half-split pairing
  (pair j = coordinates (j, j + 64), angle = position * theta**(-2j/128));
* keys at positions 0..S-1 and the query at position S;
* the cartridge workload's shared prefix holds positions 0..631 with a sink at
  position 0 whose pre-RoPE key and value are scaled by 10; the live suffix
  holds positions 632.. and the query sits after it;
* the FP8 raw-cast workload scales 4 distinct, seeded pre-RoPE key channels per
  (layer, kv head) by 20 for every token;
* the ragged workload draws 128 lengths log-uniform in [1,024, 131,072] and
  places pages by a seeded random permutation of the physical pages.

Seeds: unit seed = 1000 * workload id + unit index.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import numpy as np

__all__ = [
    "Workload",
    "WORKLOADS",
    "rope_tables",
    "apply_rope",
    "unit_seed",
    "seq_lengths",
    "outlier_channels",
    "gen_unit_cpu",
    "identity_block_table",
    "permuted_block_table",
    "slot_mapping",
    "gen_tokens_gpu",
    "block_table_for",
]

HEAD_DIM = 128
PAGE = 16


@dataclass(frozen=True)
class Workload:
    wid: int
    name: str
    batch: int
    n_layers: int
    n_kv_heads: int
    n_q_heads: int
    k_fmt: str
    v_fmt: str
    seq_len: int = 0                 # live tokens per sequence (fixed lengths)
    ragged: tuple | None = None      # (lo, hi) log-uniform lengths
    prefix_len: int = 0              # shared prefix ("cartridge") tokens
    prefix_k_fmt: str | None = None
    prefix_v_fmt: str | None = None
    sink_scale: float = 1.0          # scale of the pre-RoPE K and V at absolute position 0
    n_outliers: int = 0              # outlier pre-RoPE key channels per (layer, kv head)
    outlier_scale: float = 1.0
    massive_pairs: int = 0           # RoPE pairs (channels j, j + 64) of the pre-RoPE key scaled per (layer, kv head)
    massive_scale: float = 1.0
    bypass_pairs: int = 0            # fixed-channel bypass: the cache stores the massive pairs in fp16
    q_dtype: str = "bf16"            # 'bf16' or 'f32' query as handed to the kernel
    tier_b: bool = False
    delta_req: float = 1e-2
    n_steps: int = 256               # T in delta_loc = delta_req / (L H T)
    random_pages: bool = False
    rope_theta: float = 1e6
    tau: float = 0.2
    extra: dict = field(default_factory=dict)

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads


WORKLOADS = {
    "tiny": Workload(1, "tiny", batch=1, n_layers=1, n_kv_heads=8, n_q_heads=32,
                     k_fmt="bf16", v_fmt="e4m3s", seq_len=512, q_dtype="f32"),
    "qwen3_8b_cartridge": Workload(2, "qwen3_8b_cartridge", batch=16, n_layers=36, n_kv_heads=8, n_q_heads=32,
                                   k_fmt="bf16", v_fmt="bf16", seq_len=11996, prefix_len=632,
                                   prefix_k_fmt="bf16", prefix_v_fmt="e4m3s", sink_scale=10.0),
    "int8_7b_certified": Workload(3, "int8_7b_certified", batch=64, n_layers=28, n_kv_heads=4, n_q_heads=28,
                                  k_fmt="int8", v_fmt="int8", seq_len=32768, tier_b=True, delta_req=1e-3),
    "fp8_raw_stress": Workload(4, "fp8_raw_stress", batch=32, n_layers=36, n_kv_heads=8, n_q_heads=32,
                               k_fmt="e4m3", v_fmt="e4m3", seq_len=65536, n_outliers=4, outlier_scale=20.0),
    "ragged_paged": Workload(5, "ragged_paged", batch=128, n_layers=36, n_kv_heads=8, n_q_heads=32,
                             k_fmt="bf16", v_fmt="e4m3s", ragged=(1024, 131072), random_pages=True),
}


def unit_seed(w: Workload, unit: int) -> int:
    return 1000 * w.wid + unit


def seq_lengths(w: Workload) -> np.ndarray:
    """Live (suffix) token count of every sequence."""
    if w.ragged is None:
        return np.full(w.batch, w.seq_len, dtype=np.int64)
    rng = np.random.default_rng(unit_seed(w, 999_983))
    lo, hi = w.ragged
    u = rng.random(w.batch)
    return np.floor(np.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))).astype(np.int64).clip(lo, hi)


def outlier_channels(w: Workload, layer: int, kv_head: int) -> np.ndarray:
    """The seeded set of pre-RoPE key channels scaled for (layer, kv_head)."""
    if not w.n_outliers:
        return np.zeros(0, dtype=np.int64)
    rng = np.random.default_rng(unit_seed(w, 500_000 + layer * 64 + kv_head))
    return np.sort(rng.choice(HEAD_DIM, size=w.n_outliers, replace=False))


def massive_pairs(w: Workload, layer: int, kv_head: int) -> np.ndarray:
    """The seeded set of RoPE pairs j (pre-RoPE key channels j and j + 64 scaled) of (layer, kv_head);
    the fixed-channel bypass of the cache uses the same set (a calibration that found them)."""
    if not w.massive_pairs:
        return np.zeros(0, dtype=np.int64)
    rng = np.random.default_rng(unit_seed(w, 600_000 + layer * 64 + kv_head))
    return np.sort(rng.choice(HEAD_DIM // 2, size=w.massive_pairs, replace=False))


def bypass_pair_table(w: Workload, layer: int) -> np.ndarray:
    """[Hkv, m] int32 bypassed pairs of a layer (m = w.bypass_pairs), or an empty [Hkv, 0] table."""
    m = w.bypass_pairs
    t = np.zeros((w.n_kv_heads, m), dtype=np.int32)
    for h in range(w.n_kv_heads):
        t[h] = massive_pairs(w, layer, h)[:m]
    return t


def rope_tables(positions: np.ndarray, theta: float = 1e6):
    """cos/sin [n, 64] in float64 for half-split RoPE: angle = pos * theta**(-2j/128)."""
    j = np.arange(HEAD_DIM // 2, dtype=np.float64)
    inv = theta ** (-2.0 * j / HEAD_DIM)
    ang = np.asarray(positions, dtype=np.float64)[:, None] * inv[None, :]
    return np.cos(ang), np.sin(ang)


def apply_rope(x: np.ndarray, positions: np.ndarray, theta: float = 1e6) -> np.ndarray:
    """Rotate x [n, ..., 128] (pre-RoPE) at ``positions`` [n]; float64 math, rounded once to binary32."""
    x = np.asarray(x, dtype=np.float64)
    cos, sin = rope_tables(positions, theta)
    shape = (x.shape[0],) + (1,) * (x.ndim - 2) + (HEAD_DIM // 2,)
    cos = cos.reshape(shape)
    sin = sin.reshape(shape)
    a, b = x[..., : HEAD_DIM // 2], x[..., HEAD_DIM // 2:]
    return np.concatenate([a * cos - b * sin, b * cos + a * sin], axis=-1).astype(np.float32)


def gen_unit_cpu(w: Workload, seq: int, layer: int, n_tokens: int, first_pos: int = 0, seed_unit: int | None = None):
    """Binary32 post-RoPE K, V [n_tokens, Hkv, 128] and the query [Hq, 128] of one (sequence, layer).

    ``first_pos``: absolute position of the first token (the suffix of the cartridge workload
    starts after the prefix).  The query sits at position first_pos + n_tokens.  The query is
    rounded to bfloat16 (RNE via the binary32 bit pattern) when the workload's query dtype is bf16.
    """
    unit = seed_unit if seed_unit is not None else seq * 1000 + layer
    rng = np.random.default_rng(unit_seed(w, unit))
    k = rng.standard_normal((n_tokens, w.n_kv_heads, HEAD_DIM))
    v = rng.standard_normal((n_tokens, w.n_kv_heads, HEAD_DIM))
    q = rng.standard_normal((1, w.n_q_heads, HEAD_DIM))
    pos = np.arange(first_pos, first_pos + n_tokens)
    if w.sink_scale != 1.0 and first_pos == 0 and n_tokens > 0:
        k[0] *= w.sink_scale
        v[0] *= w.sink_scale
    for h in range(w.n_kv_heads):
        ch = outlier_channels(w, layer, h)
        if ch.size:
            k[:, h, ch] *= w.outlier_scale
        pj = massive_pairs(w, layer, h)
        if pj.size:
            k[:, h, np.concatenate([pj, pj + HEAD_DIM // 2])] *= w.massive_scale
    k32 = apply_rope(k, pos, w.rope_theta)
    v32 = v.astype(np.float32)
    q32 = apply_rope(q, np.array([first_pos + n_tokens]), w.rope_theta)[0]
    if w.q_dtype == "bf16":
        q32 = round_bf16_input(q32)
    return k32, v32, q32


def round_bf16_input(x32: np.ndarray) -> np.ndarray:
    """Input conditioning only: the bfloat16 query the kernel is handed, as binary32 values.

    Uses torch's own float32 -> bfloat16 conversion (round-to-nearest-even)."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32)).to(torch.bfloat16).float().numpy()


def identity_block_table(seq_lens, max_pages: int | None = None, start_page: int = 0) -> np.ndarray:
    """Pages of each sequence laid out back to back: [B, max_pages] int32 (unused entries -1)."""
    seq_lens = np.asarray(seq_lens)
    npg = (seq_lens + PAGE - 1) // PAGE
    mp = int(max_pages if max_pages is not None else max(1, int(npg.max(initial=1))))
    bt = np.full((len(seq_lens), mp), -1, dtype=np.int32)
    p = start_page
    for i, n in enumerate(npg):
        bt[i, :n] = np.arange(p, p + n)
        p += n
    return bt


def permuted_block_table(seq_lens, seed: int, max_pages: int | None = None) -> np.ndarray:
    """Like identity_block_table, but the physical pages are a seeded random permutation."""
    bt = identity_block_table(seq_lens, max_pages)
    used = bt[bt >= 0]
    perm = np.random.default_rng(seed).permutation(used.size).astype(np.int32)
    bt[bt >= 0] = perm[used]
    return bt


def slot_mapping(block_table: np.ndarray, seq: int, positions: np.ndarray) -> np.ndarray:
    """Physical slot (page * 16 + offset) of the given in-sequence positions."""
    positions = np.asarray(positions)
    return (block_table[seq, positions // PAGE].astype(np.int64) * PAGE + positions % PAGE).astype(np.int32)


def reduced(w: Workload, **kw) -> Workload:
    """A smaller copy of a workload (parity cases that the oracle finishes in seconds)."""
    return replace(w, **kw)


def block_table_for(w: Workload, lens, layer_seed: int = 0) -> np.ndarray:
    """The block table a workload uses: identity, or a seeded permutation of the physical pages."""
    pages = (np.asarray(lens) + PAGE - 1) // PAGE
    max_pages = max(1, int(pages.max(initial=1)))
    if w.random_pages:
        return permuted_block_table(lens, unit_seed(w, 424_242 + layer_seed), max_pages)
    return identity_block_table(lens, max_pages)


def gen_tokens_gpu(w: Workload, layer: int, positions, generator, device, sink: bool = False):
    """Binary32 post-RoPE K and V [n, Hkv, 128] on the GPU for the given absolute positions.

    Same recipe as ``gen_unit_cpu`` (N(0,1) pre-RoPE, optional x10 sink at position 0, outlier key
    channels, half-split RoPE theta = 1e6 evaluated in float64 and rounded once), drawn from torch's
    seeded GPU generator.
    """
    import torch

    pos = torch.as_tensor(positions, device=device)
    n, H = int(pos.numel()), w.n_kv_heads
    k = torch.randn((n, H, HEAD_DIM), generator=generator, device=device, dtype=torch.float32)
    v = torch.randn((n, H, HEAD_DIM), generator=generator, device=device, dtype=torch.float32)
    if sink and w.sink_scale != 1.0 and n > 0:
        k[0] *= w.sink_scale
        v[0] *= w.sink_scale
    for h in range(H):
        ch = outlier_channels(w, layer, h)
        if ch.size:
            k[:, h, torch.from_numpy(ch).to(device)] *= w.outlier_scale
        pj = massive_pairs(w, layer, h)
        if pj.size:
            k[:, h, torch.from_numpy(np.concatenate([pj, pj + HEAD_DIM // 2])).to(device)] *= w.massive_scale
    j = torch.arange(HEAD_DIM // 2, device=device, dtype=torch.float64)
    inv = w.rope_theta ** (-2.0 * j / HEAD_DIM)
    ang = pos.to(torch.float64)[:, None] * inv[None, :]
    cos, sin = torch.cos(ang)[:, None, :], torch.sin(ang)[:, None, :]
    a, b = k[..., : HEAD_DIM // 2].double(), k[..., HEAD_DIM // 2:].double()
    k = torch.cat([a * cos - b * sin, b * cos + a * sin], dim=-1).float().contiguous()
    return k, v
