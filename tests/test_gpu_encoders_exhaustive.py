"""The device number conversions against the oracle's encoders on EVERY binary32 input (2^32 patterns).

The stored bytes of every layout come from four conversions: bfloat16 round-to-nearest-even ("Compress
the shared cartridge": BF16 keys), FP8 E4M3 round-to-nearest-even saturating at +-448 (E4M3 keys and
values), binary16 round-to-nearest-even (the fp16 scales, WitCert §6.2.1) and binary16 round-up (the
witness, WitCert §4.1 eq. (2)).  kvq_debug_encode runs the kernels' own conversion of each kind over
all 2^32 bit patterns in 256 chunks of 2^24; per chunk two modular checksums of the outputs are
computed on the device and compared with the ones tests/golden/encoder_checksums.py wrote from the
oracle's encoders (see that script for the checksum).  NaN inputs are outside the contract (the library
flags non-finite inputs) and count as output 0 on both sides.
"""
import json
import os

import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "encoder_checksums.json")


@pytest.fixture(scope="module")
def kvq():
    import quantized_kv_cache_kvq_gb300 as m

    assert torch.cuda.is_available()
    m.load()
    return m


def _signed64(u: int) -> int:
    return u - (1 << 64) if u >= 1 << 63 else u


def test_device_encoders_over_every_binary32_input(kvq):
    with open(GOLDEN) as f:
        doc = json.load(f)
    cb = doc["chunk_bits"]
    n = 1 << cb
    kinds = ("bf16_rne", "e4m3_rne_satfinite", "fp16_rne", "fp16_ru")
    dev = torch.device("cuda")
    j = torch.arange(n, dtype=torch.int64, device=dev)
    # (j * A + B) | 1 modulo 2^64, in two's-complement int64 (wrapping arithmetic)
    ms = [(j * _signed64(int(a, 16)) + _signed64(int(b, 16))) | 1 for a, b in doc["multipliers"]]
    outs = {1: torch.empty(n, dtype=torch.uint8, device=dev)}
    for k in (0, 2, 3):
        outs[k] = torch.empty(n, dtype=torch.int16, device=dev)
    bad = []
    for c in range(1 << (32 - cb)):
        v = torch.arange(c << cb, (c + 1) << cb, dtype=torch.int64, device=dev)
        x = torch.where(v >= 1 << 31, v - (1 << 32), v).to(torch.int32).view(torch.float32)
        nan = torch.isnan(x)
        for kind, name in enumerate(kinds):
            kvq.debug_encode(kind, x, outs[kind])
            o = outs[kind].to(torch.int64) & (0xFF if kind == 1 else 0xFFFF)
            o = torch.where(nan, torch.zeros_like(o), o)
            got = [int((o * m).sum().item()) & ((1 << 64) - 1) for m in ms]
            want = [int(h, 16) for h in doc["checksums"][name][c]]
            if got != want:
                bad.append((name, c))
    assert not bad, bad[:20]
