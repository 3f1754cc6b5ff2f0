"""Rotary position embedding applied on append, in binary32 (oracle; test infrastructure).

The cache stores post-RoPE keys ("Compress the shared cartridge" keeps the keys post-RoPE; WitCert
§4.1 builds its bands from RoPE frequency pairs).  A write path can take the pre-RoPE key and rotate
it on append (the pages list fused RoPE-on-append with the write-path work of WitCert §6.2.3); the
rotated binary32 key is then "the exact key" the witness is measured against.

Readings (the pages fix neither the table nor the arithmetic):
* half-split pairing (NeoX / Qwen rotate_half): pair j = channels (j, j + 64), j = 0..63, angle
  pos * theta**(-2 j / 128);
* the caller supplies a binary32 table [max_position][128]: cos of the 64 angles, then their sin
  (the cos/sin cache layout of serving engines); ``cos_sin_table`` builds it in float64 and rounds
  each entry once;
* each rotated channel is two rounded binary32 products and one rounded binary32 sum, with no fused
  multiply-add:  x' = fl(fl(x c) - fl(y s)),  y' = fl(fl(y c) + fl(x s)),  (x, y) = channels (j, j + 64).
  Every step is a float64 operation on binary32 operands rounded once to binary32, which equals the
  correctly rounded binary32 operation (a product of two 24-bit significands is exact in float64, and
  a sum of two binary32 numbers rounds the same either way).

Parity status: pinned by CPU tests (identity at position 0, the float64 rotation with the same table
within 1 ulp per step, pair norms, the table's cos^2 + sin^2, agreement with an independently written
float64 RoPE).
"""
from __future__ import annotations

import numpy as np

from .encoders import f32

__all__ = ["cos_sin_table", "rope_fp32"]

HEAD_DIM = 128
HALF = HEAD_DIM // 2


def cos_sin_table(max_position: int, theta: float = 1e6) -> np.ndarray:
    """[max_position][128] binary32: cos(pos * theta^(-2j/128)) for j = 0..63, then the sines."""
    j = np.arange(HALF, dtype=np.float64)
    inv_freq = theta ** (-2.0 * j / HEAD_DIM)
    ang = np.arange(max_position, dtype=np.float64)[:, None] * inv_freq[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


def rope_fp32(k32: np.ndarray, positions: np.ndarray, table: np.ndarray) -> np.ndarray:
    """Rotate binary32 keys k32 [n, 128] or [n, heads, 128] at ``positions`` [n] with the binary32 ``table``."""
    k = np.asarray(k32, dtype=np.float32).astype(np.float64)
    rows = np.asarray(table, dtype=np.float32)[np.asarray(positions)].astype(np.float64)   # [n, 128]
    if k.ndim == 3:
        rows = rows[:, None, :]
    c, s = rows[..., :HALF], rows[..., HALF:]
    x, y = k[..., :HALF], k[..., HALF:]
    xc, ys = f32(x * c).astype(np.float64), f32(y * s).astype(np.float64)
    yc, xs = f32(y * c).astype(np.float64), f32(x * s).astype(np.float64)
    return np.concatenate([f32(xc - ys), f32(yc + xs)], axis=-1).astype(np.float32)
