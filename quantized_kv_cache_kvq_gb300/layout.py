"""Tile layouts of the paged planes (the byte-offset formulas documented in include/kvq.h).

Used to read a cache back into logical [page, kv head, token, channel] order
(tests, inspection); the kernels use the same formulas in kvq_common.cuh.
"""
from __future__ import annotations

import numpy as np

__all__ = ["int8_codes", "k_offsets", "v_offsets", "w_offsets", "s_offsets", "gs_offsets", "vw_offsets", "ko_offsets", "unpack_k",
           "unpack_v", "unpack_w", "unpack_s", "unpack_gs", "unpack_vw", "unpack_ko"]


def k_offsets(fmt: str) -> np.ndarray:
    """[16 tokens, 128 channels] byte offsets in a K tile."""
    t = np.arange(16)[:, None]
    c = np.arange(128)[None, :]
    if fmt == "bf16":
        return 16 * ((((t >> 3) * 4 + (c >> 5)) * 32) + (t & 7) * 4 + ((c >> 3) & 3)) + 2 * (c & 7)
    if fmt == "int8g32":   # 32-channel scale groups: every tensor-core k-step inside one group
        return (16 * ((((t >> 3) * 2 + (c >> 6)) * 32) + (t & 7) * 4 + ((c >> 3) & 3))
                + 4 * (2 * ((c >> 5) & 1) + ((c >> 2) & 1)) + (c & 3))
    return 16 * ((((t >> 3) * 2 + (c >> 6)) * 32) + (t & 7) * 4 + ((c >> 4) & 3)) + (c & 15)


def v_offsets(fmt: str) -> np.ndarray:
    t = np.arange(16)[:, None]
    c = np.arange(128)[None, :]
    if fmt == "bf16":
        return 16 * (32 * (c >> 4) + 4 * (c & 7) + ((t & 7) >> 1)) + 4 * (2 * (t >> 3) + ((c >> 3) & 1)) + 2 * (t & 1)
    return (16 * (32 * (c >> 5) + 4 * (c & 7) + ((t & 7) >> 1)) + 8 * ((c >> 4) & 1)
            + 2 * (2 * (t >> 3) + ((c >> 3) & 1)) + (t & 1))


def w_offsets() -> np.ndarray:
    t = np.arange(16)[:, None]
    b = np.arange(16)[None, :]
    return 16 * (4 * (t & 7) + (b >> 2)) + 8 * (t >> 3) + 2 * (b & 3)


def s_offsets() -> np.ndarray:
    t = np.arange(16)
    return 2 * (2 * (t & 7) + (t >> 3))


def gs_offsets() -> np.ndarray:
    """[16 tokens, 4 groups] byte offsets in a group-scale tile (group g = channels 32g..32g+31)."""
    t = np.arange(16)[:, None]
    g = np.arange(4)[None, :]
    return 16 * (t & 7) + 4 * g + 2 * (t >> 3)


def vw_offsets() -> np.ndarray:
    """[16 tokens, 2] byte offsets in a value-witness tile: k = 0 rho^v, k = 1 ||v||."""
    t = np.arange(16)[:, None]
    k = np.arange(2)[None, :]
    return 8 * (t & 7) + 4 * k + 2 * (t >> 3)


def ko_offsets(m: int) -> np.ndarray:
    """[16 tokens, 2m] byte offsets in a key outlier tile (8 columns for m <= 4, 16 for m <= 8)."""
    t = np.arange(16)[:, None]
    col = np.arange(2 * m)[None, :]
    if m <= 4:
        return 8 * (4 * (t & 7) + (col >> 1)) + 4 * (t >> 3) + 2 * (col & 1)
    return 16 * (4 * (t & 7) + ((col & 7) >> 1)) + 8 * (col >> 3) + 4 * (t >> 3) + 2 * (col & 1)


def _gather16(tiles: np.ndarray, offs: np.ndarray) -> np.ndarray:
    u16 = np.ascontiguousarray(tiles).view(np.uint16)
    return u16[..., offs // 2]


def int8_codes(stored: np.ndarray) -> np.ndarray:
    """INT8 codes of offset-binary stored bytes (byte = code + 128)."""
    return (np.asarray(stored, dtype=np.uint8) ^ np.uint8(0x80)).view(np.int8)


def unpack_k(tiles: np.ndarray, fmt: str, num_kv_heads: int) -> np.ndarray:
    """K plane bytes [pages*heads, tile] -> codes [pages, heads, 16, 128] (uint16 bf16 bits / uint8 e4m3 bits /
    int8 codes)."""
    tiles = tiles.reshape(-1, num_kv_heads, tiles.shape[-1])
    offs = k_offsets(fmt)
    if fmt == "bf16":
        return _gather16(tiles, offs)
    return int8_codes(tiles[..., offs]) if fmt.startswith("int8") else tiles[..., offs]


def unpack_v(tiles: np.ndarray, fmt: str, num_kv_heads: int) -> np.ndarray:
    tiles = tiles.reshape(-1, num_kv_heads, tiles.shape[-1])
    offs = v_offsets(fmt)
    if fmt == "bf16":
        return _gather16(tiles, offs)
    return int8_codes(tiles[..., offs]) if fmt.startswith("int8") else tiles[..., offs]


def unpack_w(tiles: np.ndarray, num_kv_heads: int) -> np.ndarray:
    """witness plane -> fp16 bits [pages, heads, 16 tokens, 16 bands]."""
    tiles = tiles.reshape(-1, num_kv_heads, tiles.shape[-1])
    return _gather16(tiles, w_offsets())


def unpack_s(tiles: np.ndarray, num_kv_heads: int) -> np.ndarray:
    """scale plane (head-major tiles: head * num_pages + page) -> fp16 bits [pages, heads, 16 tokens]."""
    tiles = tiles.reshape(num_kv_heads, -1, tiles.shape[-1]).transpose(1, 0, 2)
    return _gather16(tiles, s_offsets())


def unpack_gs(tiles: np.ndarray, num_kv_heads: int) -> np.ndarray:
    """group-scale plane (head-major tiles) -> fp16 bits [pages, heads, 16 tokens, 4 groups]."""
    tiles = tiles.reshape(num_kv_heads, -1, tiles.shape[-1]).transpose(1, 0, 2)
    return _gather16(tiles, gs_offsets())


def unpack_vw(tiles: np.ndarray, num_kv_heads: int) -> np.ndarray:
    """value-witness plane (head-major tiles) -> fp16 bits [pages, heads, 16 tokens, 2]."""
    tiles = tiles.reshape(num_kv_heads, -1, tiles.shape[-1]).transpose(1, 0, 2)
    return _gather16(tiles, vw_offsets())


def unpack_ko(tiles: np.ndarray, num_kv_heads: int, m: int) -> np.ndarray:
    """key outlier plane (head-major tiles) -> fp16 bits [pages, heads, 16 tokens, 2m] in column order."""
    tiles = tiles.reshape(num_kv_heads, -1, tiles.shape[-1]).transpose(1, 0, 2)
    return _gather16(tiles, ko_offsets(m))
