"""Byte account per layout and per decode workload (oracle; test infrastructure).

* "Compress the shared cartridge", table "Keys carry the cartridge quantization
  loss": raw KV payload per token for Qwen3-8B (36 layers x 8 KV heads x d 128),
  without scales or metadata: BF16 K16/V16 144 KiB, K16/V8 and K8/V16 108 KiB,
  K8/V8 72 KiB; 12,628 tokens and a 632-position cartridge scale those linearly.
* WitCert §4.1: the witness costs 2B = 32 bytes per token per kv head (B = 16, fp16).
* WitCert §6.2.3: one fp16 scale per (token, kv head) per channel group.  Its Table 4
  prices the scale granularities of 8-bit K and V per token per kv head against fp16
  K+V (512 B): a 256-token block scale per channel, and per-token scales over groups
  of 16, 32 or 128 (one scalar) channels; G_c = 32 stores 136 B per side.

The decode path must read, per token and kv head: the key codes, the value
codes, their scales when the format has one, and (meter on) the witness.
"""
from __future__ import annotations

__all__ = ["CODE_BYTES", "payload_bytes_per_token", "kv_bytes_per_token_head", "decode_step_bytes",
           "int8_side_bytes", "scale_granularity_saving"]

CODE_BYTES = {"bf16": 2, "e4m3": 1, "e4m3s": 1, "int8": 1, "int8g32": 1}
HAS_SCALE = {"bf16": False, "e4m3": False, "e4m3s": True, "int8": True, "int8g32": True}
SCALE_GROUPS = {"e4m3s": 1, "int8": 1, "int8g32": 4}   # fp16 scales per (token, kv head)
WITNESS_BYTES = 32   # 16 bands x fp16
SCALE_BYTES = 2      # one fp16 scale


def payload_bytes_per_token(k_fmt: str, v_fmt: str, n_layers: int, n_kv_heads: int, head_dim: int = 128) -> int:
    """Raw K+V payload bytes per token over all layers and kv heads (no scales, no witness)."""
    return n_layers * n_kv_heads * head_dim * (CODE_BYTES[k_fmt] + CODE_BYTES[v_fmt])


def kv_bytes_per_token_head(k_fmt: str, v_fmt: str, meter: bool = True, head_dim: int = 128) -> int:
    """Bytes the decode path reads per token per kv head: codes, scales, and the witness when metered."""
    b = head_dim * (CODE_BYTES[k_fmt] + CODE_BYTES[v_fmt])
    b += SCALE_BYTES * (SCALE_GROUPS.get(k_fmt, 0) + SCALE_GROUPS.get(v_fmt, 0))
    if meter:
        b += WITNESS_BYTES
    return b


def decode_step_bytes(batch: int, n_layers: int, n_kv_heads: int, seq_lens, k_fmt: str, v_fmt: str,
                      prefix_len: int = 0, prefix_k_fmt: str | None = None, prefix_v_fmt: str | None = None,
                      meter: bool = True) -> int:
    """Algorithmic bytes of one decode step: every live token once per (layer, kv head), and a
    shared prefix once per layer (it is one buffer shared by the whole batch)."""
    per = kv_bytes_per_token_head(k_fmt, v_fmt, meter)
    live = sum(int(s) for s in seq_lens) if not isinstance(seq_lens, int) else seq_lens * batch
    total = n_layers * n_kv_heads * live * per
    if prefix_len:
        pp = kv_bytes_per_token_head(prefix_k_fmt, prefix_v_fmt, meter)
        total += n_layers * n_kv_heads * prefix_len * pp
    return total


def int8_side_bytes(granularity: str, group: int = 32, block: int = 256, head_dim: int = 128) -> float:
    """Bytes per token per kv head of one 8-bit side (K or V) with fp16 scales at a granularity:
    'token' (one scale per group of ``group`` channels of the token; group = head_dim is one scalar)
    or 'block' (one scale per channel shared by ``block`` tokens)."""
    if granularity == "token":
        assert head_dim % group == 0
        return head_dim + SCALE_BYTES * (head_dim // group)
    if granularity == "block":
        return head_dim + SCALE_BYTES * head_dim / block
    raise ValueError(granularity)


def scale_granularity_saving(k_plus_v_bytes: float, head_dim: int = 128) -> float:
    """Fraction of fp16 K+V (4 head_dim bytes per token per kv head) that a layout saves."""
    return 1.0 - k_plus_v_bytes / (2 * 2 * head_dim)
