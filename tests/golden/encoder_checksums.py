"""Writes tests/golden/encoder_checksums.json: checksums of the oracle's number encoders over EVERY binary32
bit pattern (test infrastructure; calls only oracle/).

The stored bytes of every layout are made by four encoders: bfloat16 round-to-nearest-even (BF16 keys,
"Compress the shared cartridge"), FP8 E4M3 round-to-nearest-even with saturation to +-448 (E4M3 keys and
values, same page), and binary16 round-to-nearest-even and round-up (the fp16 scales, WitCert §6.2.1; the
witness, WitCert §4.1 eq. (2)).  tests/test_gpu_encoders_exhaustive.py runs the device conversions on the
same 2^32 inputs and compares checksums chunk by chunk.

Inputs: chunk c holds the bit patterns c * 2^24 .. (c + 1) * 2^24 - 1 (256 chunks).  NaN inputs are left out
of the contract (the library flags non-finite inputs): their outputs count as 0.  Checksum of a chunk's
outputs o[j] (j = 0 .. 2^24 - 1, as unsigned integers): sum_j o[j] * m_a(j) mod 2^64 for two odd multiplier
sequences m_a(j) = (j * A_a + B_a) mod 2^64 | 1; a single differing output changes both sums.

    python tests/golden/encoder_checksums.py [--procs N]
"""
from __future__ import annotations

import argparse
import json
import multiprocessing as mp
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "encoder_checksums.json")
CHUNK_BITS = 24
N_CHUNKS = 1 << (32 - CHUNK_BITS)
KINDS = ("bf16_rne", "e4m3_rne_satfinite", "fp16_rne", "fp16_ru")
MULTIPLIERS = ((0x9E3779B97F4A7C15, 0x632BE59BD9B4E019), (0xD6E8FEB86659FD93, 0x2545F4914F6CDD1D))


def multipliers(n: int) -> list[np.ndarray]:
    j = np.arange(n, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return [(j * np.uint64(a) + np.uint64(b)) | np.uint64(1) for a, b in MULTIPLIERS]


def encode(kind: int, x32: np.ndarray) -> np.ndarray:
    from oracle.encoders import bf16_bits_rne, e4m3_bits_rne_satfinite, fp16_bits

    with np.errstate(all="ignore"):
        if kind == 0:
            out = bf16_bits_rne(x32)
        elif kind == 1:
            out = e4m3_bits_rne_satfinite(x32)
        else:
            out = fp16_bits(x32.astype(np.float64), "rne" if kind == 2 else "ru")
    return np.where(np.isnan(x32), 0, out.astype(np.uint64)).astype(np.uint64)


def chunk_checksums(c: int) -> tuple[int, list[list[str]]]:
    sys.path.insert(0, ROOT)
    bits = np.arange(c << CHUNK_BITS, (c + 1) << CHUNK_BITS, dtype=np.uint64).astype(np.uint32)
    x32 = bits.view(np.float32)
    ms = multipliers(bits.size)
    res = []
    for kind in range(len(KINDS)):
        o = encode(kind, x32)
        with np.errstate(over="ignore"):
            res.append([f"{int(np.sum(o * m, dtype=np.uint64)):016x}" for m in ms])
    return c, res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--procs", type=int, default=os.cpu_count() or 1)
    args = ap.parse_args()
    table = {k: [None] * N_CHUNKS for k in KINDS}
    with mp.get_context("spawn").Pool(args.procs) as pool:
        for c, res in pool.imap_unordered(chunk_checksums, range(N_CHUNKS)):
            for kind, name in enumerate(KINDS):
                table[name][c] = res[kind]
    doc = {"source": "oracle.encoders over all 2^32 binary32 bit patterns (tests/golden/encoder_checksums.py)",
           "chunk_bits": CHUNK_BITS, "nan_outputs": 0,
           "multipliers": [[f"{a:016x}", f"{b:016x}"] for a, b in MULTIPLIERS], "checksums": table}
    with open(OUT, "w") as f:
        json.dump(doc, f, indent=0)
        f.write("\n")


if __name__ == "__main__":
    main()
