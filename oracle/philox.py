"""Philox4x32-10 and the subtractive-dither stream (oracle; test infrastructure).

Source passages
---------------
* WitCert §6.2.1: the dither of the quantizer is drawn by Philox4x32-10 [Salmon
  et al., SC'11] from a counter built from the cache coordinates, so that the
  read side regenerates exactly the dither the write side used.
* WitCert §6.2.3 (storage side): the counter tuple is (layer, kv_head, slot,
  channel) -- the physical slot rather than the sequence position, because a
  written slot never changes under paging or prefix sharing.
* WitCert §4.2: the dither is uniform on [-1/2, 1/2).

Generator (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as
1, 2, 3", SC'11, the Philox-4x32 family): a 128-bit counter (x0, x1, x2, x3)
and a 64-bit key (k0, k1).  One round multiplies x0 and x2 by the two Philox
multipliers into 64-bit products and forms the new counter from the product
halves, the untouched words and the key:

    (hi0, lo0) = M0 * x0 ;  (hi1, lo1) = M1 * x2
    x' = (hi1 ^ x1 ^ k0,  lo1,  hi0 ^ x3 ^ k1,  lo0)

After every round the key is bumped by the two Weyl constants.  Ten rounds
give Philox4x32-10.  The constants are the published ones: M0 = 0xD2511F53,
M1 = 0xCD9E8D57, W0 = 0x9E3779B9 (golden ratio), W1 = 0xBB67AE85 (sqrt(3)-1).

Dither contract (this library's reading; the pages fix only the tuple, the
generator and the distribution):

    key     = (seed mod 2**32, seed >> 32)
    counter = (slot, layer, kv_head, channel >> 4)
    word    = output word w = ((channel >> 2) & 3) of that call
    field   = byte (channel & 3) of w, i.e. bits 8 (channel & 3) .. 8 (channel & 3) + 7
    xi      = field * 2**-8 - 1/2

so each call serves sixteen consecutive channels (the four bytes of each output
word; the pages reuse every output word of a call, here each word carries four
dithers), xi is uniform on the 256-point grid {-1/2, -1/2 + 2**-8, ..., 1/2 -
2**-8} of [-1/2, 1/2), every value is exact in fp16 (hence in binary32), and the
key and value planes of a token share the same xi.  The grid is what makes the
read side exact: xi + 9/2 = 4 + field * 2**-8 is the fp16 number whose low
mantissa byte is the field (bit pattern 0x4400 | field), so a byte permutation
of w gives it, -xi = 9/2 - (that number), and the decode's fp16 tensor-core
operands carry the write side's xi itself, not a rounding of it.  What the grid
costs is stated by ``subtractive_error_bias_bound``: for any input, the dithered
rounding error rint(y + xi) - (y + xi) takes 256 equally spaced values spanning
one unit, so its mean lies within 2**-9 of 0 (a continuous uniform xi gives
exactly 0), and its centred part is sub-Gaussian with variance proxy at most
1/12 (the moment generating function of an N-point centred grid, sinh(l/2) / (N
sinh(l/(2N))), never exceeds the continuous one, sinh(l/2) / (l/2)).

Parity status: pinned.  ``philox4x32_10`` agrees word for word with the CUDA
toolkit's own Philox4x32-10 generator (cuRAND device API, four seeds, seven
subsequences; tests/test_gpu_philox_pin.py).  On CPU it is further pinned by
properties (bijectivity through an independently written inverse, uniformity
and independence statistics, avalanche).
"""
from __future__ import annotations

import numpy as np

__all__ = ["PHILOX_M0", "PHILOX_M1", "PHILOX_W0", "PHILOX_W1", "DITHER_BITS", "philox4x32_10", "dither",
           "dither_fields", "subtractive_error_bias_bound"]

PHILOX_M0 = 0xD2511F53
PHILOX_M1 = 0xCD9E8D57
PHILOX_W0 = 0x9E3779B9
PHILOX_W1 = 0xBB67AE85
_MASK = np.uint64(0xFFFFFFFF)
DITHER_BITS = 8  # xi lies on a 2**DITHER_BITS-point grid


def _mulhilo(m: int, x: np.ndarray):
    p = np.uint64(m) * x.astype(np.uint64)  # < 2**64, exact in uint64
    return (p >> np.uint64(32)) & _MASK, p & _MASK


def philox4x32_10(ctr, key, rounds: int = 10):
    """Vectorised Philox4x32 with ``rounds`` rounds.

    ``ctr``: four arrays (broadcastable) of uint32 counter words; ``key``: two
    uint32 key words (scalars or arrays).  Returns four uint64 arrays holding the
    32-bit output words.
    """
    x0, x1, x2, x3 = (np.asarray(c, dtype=np.uint64) & _MASK for c in ctr)
    x0, x1, x2, x3 = np.broadcast_arrays(x0, x1, x2, x3)
    k0 = np.asarray(key[0], dtype=np.uint64) & _MASK
    k1 = np.asarray(key[1], dtype=np.uint64) & _MASK
    for r in range(rounds):
        if r:
            k0 = (k0 + np.uint64(PHILOX_W0)) & _MASK
            k1 = (k1 + np.uint64(PHILOX_W1)) & _MASK
        hi0, lo0 = _mulhilo(PHILOX_M0, x0)
        hi1, lo1 = _mulhilo(PHILOX_M1, x2)
        x0, x1, x2, x3 = hi1 ^ x1 ^ k0, lo1, hi0 ^ x3 ^ k1, lo0
    return x0, x1, x2, x3


def dither_words(seed: int, layer: int, kv_head, slot, channel):
    """The 32-bit Philox word that carries the dither of (layer, kv_head, slot, channel)."""
    seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    key = (seed & 0xFFFFFFFF, seed >> 32)
    slot = np.asarray(slot, dtype=np.uint64)
    channel = np.asarray(channel, dtype=np.int64)
    kv_head = np.asarray(kv_head, dtype=np.uint64)
    slot, kv_head, channel = np.broadcast_arrays(slot, kv_head, channel)
    words = philox4x32_10((slot, np.uint64(layer), kv_head, (channel >> 4).astype(np.uint64)), key)
    out = np.choose((channel >> 2) & 3, words)
    return out.astype(np.uint64)


def dither_fields(seed: int, layer: int, kv_head, slot, channel) -> np.ndarray:
    """The 8-bit field of the Philox word that is the dither of (layer, kv_head, slot, channel): byte
    (channel & 3) of the word."""
    channel = np.asarray(channel, dtype=np.int64)
    w = dither_words(seed, layer, kv_head, slot, channel)
    shift = (np.broadcast_to(channel, w.shape) & 3).astype(np.uint64) * np.uint64(8)
    return (w >> shift) & np.uint64((1 << DITHER_BITS) - 1)


def dither(seed: int, layer: int, kv_head, slot, channel) -> np.ndarray:
    """Dither values xi in [-1/2, 1/2) for broadcastable (kv_head, slot, channel) arrays (float64, exact)."""
    k = dither_fields(seed, layer, kv_head, slot, channel).astype(np.float64)
    return k * 2.0 ** -DITHER_BITS - 0.5


def subtractive_error_bias_bound() -> float:
    """Largest |E[rint(y + xi) - (y + xi)]| over inputs y when xi is uniform on the dither grid.

    For fixed y the 2**DITHER_BITS values of y + xi are equally spaced by 2**-DITHER_BITS over one
    unit, so the rounding errors are the same grid shifted into [-1/2, 1/2]; its mean is within
    half a grid step of 0.
    """
    return 2.0 ** -(DITHER_BITS + 1)
