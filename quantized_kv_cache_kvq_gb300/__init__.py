"""Python binding of libkvq (argument marshalling only).

Every step of the decode path runs in the CUDA library: this module allocates
device memory with torch, packs the C structs of ``include/kvq.h`` and calls
the C ABI with the current torch stream.  There is no CPU fallback: importing
works without a GPU (so the library can be inspected), but every compute call
needs the built ``libkvq.so`` and a CUDA device, and raises otherwise.

Entry points mirror the C names: ``append``, ``decode_attn``, ``meter``,
``decode_workspace_size``, ``debug_dither``, ``debug_encode``, plus the
``PagedCache`` helper that owns one layer's planes.
"""
from __future__ import annotations

import ctypes
import math
import os
from ctypes import POINTER, c_double, c_float, c_int32, c_int64, c_size_t, c_uint32, c_uint64, c_void_p

import torch

__all__ = [
    "FMT",
    "KvqError",
    "lib",
    "load",
    "PagedCache",
    "MeterParams",
    "append",
    "decode_attn",
    "decode_attn_noalloc",
    "decode_workspace_size",
    "append_rope",
    "meter",
    "debug_dither",
    "debug_encode",
    "tile_bytes",
    "status_string",
    "read_err",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.environ.get("KVQ_LIB") or os.path.join(_HERE, "libkvq.so")

FMT = {"bf16": 0, "e4m3": 1, "e4m3s": 2, "int8": 3, "int8g32": 4}
SCALE_TILE_BYTES = {"e4m3s": 32, "int8": 32, "int8g32": 128}  # fp16 scales of a page's 16 tokens
DTYPE = {torch.float32: 0, torch.bfloat16: 1}
TIER_A, TIER_B, TIER_V, TIER_S = 1, 2, 4, 8
METER_STATE_FLOATS = 8  # floats per (sequence, query head) cell of meter_state
HEAD_DIM, PAGE, N_BANDS = 128, 16, 16

STATUS = {
    0: "KVQ_OK",
    1: "KVQ_ERR_INVALID_ARG",
    2: "KVQ_ERR_UNSUPPORTED_LAYOUT",
    3: "KVQ_ERR_WORKSPACE_TOO_SMALL",
    4: "KVQ_ERR_CUDA",
    5: "KVQ_ERR_DEVICE_BOUNDS",
    6: "KVQ_ERR_NONFINITE_INPUT",
    7: "KVQ_ERR_RANGE",
    8: "KVQ_ERR_TIMEOUT",
}


class KvqError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {STATUS.get(status, status)}")
        self.status = status


class _Cache(ctypes.Structure):
    _fields_ = [
        ("k_fmt", c_int32),
        ("v_fmt", c_int32),
        ("num_kv_heads", c_int32),
        ("num_pages", c_int32),
        ("layer", c_int32),
        ("reserved", c_int32),
        ("dither_seed", c_uint64),
        ("k_data", c_void_p),
        ("v_data", c_void_p),
        ("k_scale", c_void_p),
        ("v_scale", c_void_p),
        ("witness", c_void_p),
        ("v_witness", c_void_p),
        ("outlier_pairs", c_void_p),
        ("n_outlier_pairs", c_int32),
        ("reserved2", c_int32),
        ("k_outlier", c_void_p),
    ]


class DecodeExtras(ctypes.Structure):
    _fields_ = [("page_log_contrib", c_void_p), ("contrib_stride", c_int32), ("reserved", c_int32)]


class MeterParams(ctypes.Structure):
    _fields_ = [
        ("tiers", c_uint32),
        ("n_layers", c_int32),
        ("n_q_heads", c_int32),
        ("n_steps", c_int32),
        ("delta_req", c_double),
        ("tau", c_float),
        ("reserved", c_int32),
    ]


_lib = None


def load(path: str = LIB_PATH):
    """Load libkvq.so (built by ``build.build()``); raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libkvq.so not built ({path}); run __graft_entry__.build()")
    L = ctypes.CDLL(path)
    L.kvq_tile_bytes.restype = c_size_t
    L.kvq_tile_bytes.argtypes = [c_int32, c_int32]
    L.kvq_append.restype = c_int32
    L.kvq_append.argtypes = [POINTER(_Cache), c_void_p, c_void_p, c_int32, c_void_p, c_int32, c_void_p, c_void_p]
    L.kvq_append_rope.restype = c_int32
    L.kvq_append_rope.argtypes = [POINTER(_Cache), c_void_p, c_void_p, c_int32, c_void_p, c_void_p, c_int32, c_void_p,
                                  c_int32, c_void_p, c_void_p]
    L.kvq_decode_workspace_size.restype = c_size_t
    L.kvq_decode_workspace_size.argtypes = [c_int32, c_int32, c_int32]
    L.kvq_decode_attn.restype = c_int32
    L.kvq_decode_attn.argtypes = [
        POINTER(_Cache), POINTER(_Cache), c_int32, c_void_p, c_int32, c_int32, c_int32, c_void_p, c_int32,
        c_void_p, c_float, POINTER(MeterParams), c_void_p, c_void_p, c_void_p, c_size_t, c_void_p, c_void_p,
    ]
    L.kvq_decode_attn_append.restype = c_int32
    L.kvq_decode_attn_append.argtypes = [
        POINTER(_Cache), c_void_p, c_void_p, c_int32, POINTER(_Cache), c_int32, c_void_p, c_int32, c_int32, c_int32,
        c_void_p, c_int32, c_void_p, c_float, POINTER(MeterParams), c_void_p, c_void_p, c_void_p, c_size_t, c_void_p,
        c_void_p,
    ]
    L.kvq_decode_attn_ex.restype = c_int32
    L.kvq_decode_attn_ex.argtypes = [
        POINTER(_Cache), c_void_p, c_void_p, c_int32, POINTER(_Cache), c_int32, c_void_p, c_int32, c_int32, c_int32,
        c_void_p, c_int32, c_void_p, c_float, POINTER(MeterParams), POINTER(DecodeExtras), c_void_p, c_void_p,
        c_void_p, c_size_t, c_void_p, c_void_p,
    ]
    L.kvq_gate.restype = c_int32
    L.kvq_gate.argtypes = [c_void_p, c_int32, c_void_p, c_int32, c_int32, c_void_p, c_int32, c_float, c_void_p,
                           c_void_p, c_int32, c_void_p]
    L.kvq_zero_witness.restype = c_int32
    L.kvq_zero_witness.argtypes = [POINTER(_Cache), c_void_p, c_int32, c_void_p, c_void_p]
    L.kvq_decode_attn_noalloc.restype = c_int32
    L.kvq_decode_attn_noalloc.argtypes = [
        POINTER(_Cache), POINTER(_Cache), c_int32, c_void_p, c_int32, c_int32, c_int32, c_void_p, c_int32,
        c_void_p, c_float, POINTER(MeterParams), c_void_p, c_void_p, c_void_p, c_void_p,
    ]
    L.kvq_meter.restype = c_int32
    L.kvq_meter.argtypes = [c_void_p, c_int32, c_int32, c_int32, POINTER(MeterParams), c_void_p, c_void_p,
                            c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]
    L.kvq_sizeof.restype = c_size_t
    L.kvq_sizeof.argtypes = [c_int32]
    L.kvq_debug_dither.restype = c_int32
    L.kvq_debug_dither.argtypes = [c_uint64, c_int32, c_int32, c_void_p, c_int32, c_void_p, c_void_p]
    L.kvq_debug_encode.restype = c_int32
    L.kvq_debug_encode.argtypes = [c_int32, c_void_p, c_int64, c_void_p, c_void_p]
    L.kvq_debug_time_decode.restype = c_int32
    L.kvq_debug_time_decode.argtypes = [c_void_p, c_void_p]
    L.kvq_debug_wait_timeout.restype = c_int32
    L.kvq_debug_wait_timeout.argtypes = [c_uint64, c_void_p, c_void_p]
    L.kvq_status_string.restype = ctypes.c_char_p
    L.kvq_status_string.argtypes = [c_int32]
    L.kvq_version.restype = c_int32
    L.kvq_version.argtypes = []
    _lib = L
    return L


def lib():
    return load()


def _check(status: int, where: str):
    if status != 0:
        raise KvqError(status, where)


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _ptr(t):
    return None if t is None else t.data_ptr()


def tile_bytes(fmt: str, plane: int) -> int:
    return int(lib().kvq_tile_bytes(FMT[fmt], plane))


def status_string(status: int) -> str:
    return lib().kvq_status_string(status).decode()


class PagedCache:
    """One layer's paged planes (device memory owned by torch tensors)."""

    def __init__(self, k_fmt: str, v_fmt: str, num_kv_heads: int, num_pages: int, layer: int = 0,
                 seed: int = 0, device="cuda", witness: bool = True, value_witness: bool = False,
                 outlier_pairs: torch.Tensor | None = None):
        self.k_fmt, self.v_fmt = k_fmt, v_fmt
        self.num_kv_heads, self.num_pages, self.layer, self.seed = num_kv_heads, num_pages, layer, seed
        n = num_pages * num_kv_heads
        kb = 4096 if k_fmt == "bf16" else 2048
        vb = 4096 if v_fmt == "bf16" else 2048
        z = dict(dtype=torch.uint8, device=device)
        self.k = torch.zeros((n, kb), **z)
        self.v = torch.zeros((n, vb), **z)
        self.k_scale = torch.zeros((n, SCALE_TILE_BYTES[k_fmt]), **z) if k_fmt in SCALE_TILE_BYTES else None
        self.v_scale = torch.zeros((n, SCALE_TILE_BYTES[v_fmt]), **z) if v_fmt in SCALE_TILE_BYTES else None
        self.witness = torch.zeros((n, 512), **z) if witness else None
        self.v_witness = torch.zeros((n, 64), **z) if value_witness else None
        # fixed-channel key outlier bypass: [num_kv_heads, m] int32 RoPE pairs (INT8-dithered keys)
        self.n_out = 0 if outlier_pairs is None else int(outlier_pairs.shape[1])
        self.outlier_pairs = None
        self.k_outlier = None
        if self.n_out:
            assert outlier_pairs.shape[0] == num_kv_heads and outlier_pairs.dtype == torch.int32
            self.outlier_pairs = outlier_pairs.to(device).contiguous()
            self.k_outlier = torch.zeros((n, 256 if self.n_out <= 4 else 512), **z)

    def desc(self) -> _Cache:
        return _Cache(FMT[self.k_fmt], FMT[self.v_fmt], self.num_kv_heads, self.num_pages, self.layer, 0,
                      self.seed & 0xFFFFFFFFFFFFFFFF, _ptr(self.k), _ptr(self.v), _ptr(self.k_scale),
                      _ptr(self.v_scale), _ptr(self.witness), _ptr(self.v_witness), _ptr(self.outlier_pairs),
                      self.n_out, 0, _ptr(self.k_outlier))

    def nbytes(self) -> int:
        return sum(t.numel() for t in (self.k, self.v, self.k_scale, self.v_scale, self.witness, self.v_witness,
                                       self.k_outlier) if t is not None)


def read_err(err: torch.Tensor) -> int:
    return int(err.item())


def append(cache: PagedCache, k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
           err: torch.Tensor | None = None, stream=None):
    """kvq_append: quantize k, v [n, Hkv, 128] (fp32 or bf16) into the slots of ``cache``."""
    assert k.is_contiguous() and v.is_contiguous() and k.dtype == v.dtype and k.shape == v.shape
    assert slot_mapping.dtype == torch.int32 and slot_mapping.is_contiguous()
    d = cache.desc()
    _check(lib().kvq_append(ctypes.byref(d), k.data_ptr(), v.data_ptr(), DTYPE[k.dtype], slot_mapping.data_ptr(),
                            int(k.shape[0]), _ptr(err), _stream(stream)), "kvq_append")


def append_rope(cache: PagedCache, k_pre: torch.Tensor, v: torch.Tensor, positions: torch.Tensor,
                cos_sin: torch.Tensor, slot_mapping: torch.Tensor, err: torch.Tensor | None = None, stream=None):
    """kvq_append_rope: rotate the pre-RoPE keys k_pre [n, Hkv, 128] at ``positions`` [n] with the fp32 table
    ``cos_sin`` [max_position, 128] (cos of the 64 pair angles, then their sin), then quantize as kvq_append."""
    assert k_pre.is_contiguous() and v.is_contiguous() and k_pre.dtype == v.dtype and k_pre.shape == v.shape
    assert slot_mapping.dtype == torch.int32 and slot_mapping.is_contiguous()
    assert positions.dtype == torch.int32 and positions.is_contiguous() and positions.numel() == k_pre.shape[0]
    assert cos_sin.dtype == torch.float32 and cos_sin.is_contiguous() and cos_sin.dim() == 2 and cos_sin.shape[1] == HEAD_DIM
    d = cache.desc()
    _check(lib().kvq_append_rope(ctypes.byref(d), k_pre.data_ptr(), v.data_ptr(), DTYPE[k_pre.dtype],
                                 positions.data_ptr(), cos_sin.data_ptr(), int(cos_sin.shape[0]),
                                 slot_mapping.data_ptr(), int(k_pre.shape[0]), _ptr(err), _stream(stream)),
           "kvq_append_rope")


def decode_workspace_size(batch: int, num_kv_heads: int, num_q_heads: int) -> int:
    return int(lib().kvq_decode_workspace_size(batch, num_kv_heads, num_q_heads))


def meter_params(tiers: int = TIER_A, n_layers: int = 1, n_q_heads: int = 1, n_steps: int = 256,
                 delta_req: float = 1e-2, tau: float = 0.2) -> MeterParams:
    return MeterParams(tiers, n_layers, n_q_heads, n_steps, delta_req, tau, 0)


def decode_attn(cache: PagedCache, q: torch.Tensor, block_table: torch.Tensor, seq_lens: torch.Tensor,
                out: torch.Tensor, workspace: torch.Tensor, *, prefix: PagedCache | None = None,
                prefix_len: int = 0, sm_scale: float | None = None, meter: MeterParams | None = None,
                meter_state: torch.Tensor | None = None, err: torch.Tensor | None = None, stream=None):
    """kvq_decode_attn for one layer: q [B, Hq, 128] -> out [B, Hq, 128] (+ meter_state [B, Hq, 8])."""
    B, Hq, D = q.shape
    assert D == HEAD_DIM and q.is_contiguous() and out.is_contiguous()
    assert block_table.dtype == torch.int32 and seq_lens.dtype == torch.int32
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(HEAD_DIM)
    d = cache.desc()
    pd = prefix.desc() if prefix is not None else None
    _check(lib().kvq_decode_attn(
        ctypes.byref(d), ctypes.byref(pd) if pd is not None else None, int(prefix_len), q.data_ptr(), DTYPE[q.dtype],
        B, Hq, block_table.data_ptr(), int(block_table.shape[1]) if block_table.dim() == 2 else 0,
        seq_lens.data_ptr(), float(sm_scale), ctypes.byref(meter) if meter is not None else None,
        out.data_ptr(), _ptr(meter_state), workspace.data_ptr(), workspace.numel() * workspace.element_size(),
        _ptr(err), _stream(stream)), "kvq_decode_attn")


def decode_attn_append(cache: PagedCache, k_new: torch.Tensor, v_new: torch.Tensor, q: torch.Tensor,
                       block_table: torch.Tensor, seq_lens: torch.Tensor, out: torch.Tensor, workspace: torch.Tensor, *,
                       prefix: PagedCache | None = None, prefix_len: int = 0, sm_scale: float | None = None,
                       meter: MeterParams | None = None, meter_state: torch.Tensor | None = None,
                       err: torch.Tensor | None = None, stream=None):
    """kvq_decode_attn_append: append each sequence's newest token (k_new, v_new [B, Hkv, 128]) and decode."""
    B, Hq, D = q.shape
    assert D == HEAD_DIM and q.is_contiguous() and out.is_contiguous()
    assert k_new.is_contiguous() and v_new.is_contiguous() and k_new.dtype == v_new.dtype and k_new.shape == v_new.shape
    assert block_table.dtype == torch.int32 and seq_lens.dtype == torch.int32
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(HEAD_DIM)
    d = cache.desc()
    pd = prefix.desc() if prefix is not None else None
    _check(lib().kvq_decode_attn_append(
        ctypes.byref(d), k_new.data_ptr(), v_new.data_ptr(), DTYPE[k_new.dtype],
        ctypes.byref(pd) if pd is not None else None, int(prefix_len), q.data_ptr(), DTYPE[q.dtype],
        B, Hq, block_table.data_ptr(), int(block_table.shape[1]) if block_table.dim() == 2 else 0,
        seq_lens.data_ptr(), float(sm_scale), ctypes.byref(meter) if meter is not None else None,
        out.data_ptr(), _ptr(meter_state), workspace.data_ptr(), workspace.numel() * workspace.element_size(),
        _ptr(err), _stream(stream)), "kvq_decode_attn_append")


def decode_attn_ex(cache: PagedCache, q: torch.Tensor, block_table: torch.Tensor, seq_lens: torch.Tensor,
                   out: torch.Tensor, workspace: torch.Tensor, *, k_new: torch.Tensor | None = None,
                   v_new: torch.Tensor | None = None, prefix: PagedCache | None = None, prefix_len: int = 0,
                   sm_scale: float | None = None, meter: MeterParams | None = None,
                   meter_state: torch.Tensor | None = None, page_log_contrib: torch.Tensor | None = None,
                   err: torch.Tensor | None = None, stream=None):
    """kvq_decode_attn_ex: decode (with the optional newest-token append) and the optional per-page
    log contributions page_log_contrib [B, Hq, stride] (fp32) for kvq_gate."""
    B, Hq, D = q.shape
    assert D == HEAD_DIM and q.is_contiguous() and out.is_contiguous()
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(HEAD_DIM)
    d = cache.desc()
    pd = prefix.desc() if prefix is not None else None
    ex = None
    if page_log_contrib is not None:
        assert page_log_contrib.dtype == torch.float32 and page_log_contrib.is_contiguous()
        ex = DecodeExtras(page_log_contrib.data_ptr(), int(page_log_contrib.shape[-1]), 0)
    _check(lib().kvq_decode_attn_ex(
        ctypes.byref(d), _ptr(k_new), _ptr(v_new), DTYPE[k_new.dtype] if k_new is not None else 0,
        ctypes.byref(pd) if pd is not None else None, int(prefix_len), q.data_ptr(), DTYPE[q.dtype], B, Hq,
        block_table.data_ptr(), int(block_table.shape[1]) if block_table.dim() == 2 else 0, seq_lens.data_ptr(),
        float(sm_scale), ctypes.byref(meter) if meter is not None else None, ctypes.byref(ex) if ex is not None else None,
        out.data_ptr(), _ptr(meter_state), workspace.data_ptr(), workspace.numel() * workspace.element_size(),
        _ptr(err), _stream(stream)), "kvq_decode_attn_ex")


def gate(page_log_contrib: torch.Tensor, meter_state: torch.Tensor, seq_lens: torch.Tensor, prefix_len: int,
         tau: float, n_page_in: torch.Tensor, page_list: torch.Tensor | None = None, stream=None):
    """kvq_gate: greedy page-in plan per (sequence, query head)."""
    B, Hq, stride = page_log_contrib.shape
    _check(lib().kvq_gate(page_log_contrib.data_ptr(), stride, meter_state.data_ptr(), B, Hq, seq_lens.data_ptr(),
                          int(prefix_len), float(tau), n_page_in.data_ptr(), _ptr(page_list),
                          int(page_list.shape[-1]) if page_list is not None else 0, _stream(stream)), "kvq_gate")


def zero_witness(cache: PagedCache, slots: torch.Tensor, err: torch.Tensor | None = None, stream=None):
    """kvq_zero_witness: zero the witness (and value witness) of repaired slots."""
    d = cache.desc()
    _check(lib().kvq_zero_witness(ctypes.byref(d), slots.data_ptr(), int(slots.numel()), _ptr(err), _stream(stream)),
           "kvq_zero_witness")


def decode_attn_noalloc(cache: PagedCache, q: torch.Tensor, block_table: torch.Tensor, seq_lens: torch.Tensor,
                        out: torch.Tensor, *, prefix: PagedCache | None = None, prefix_len: int = 0,
                        sm_scale: float | None = None, meter: MeterParams | None = None,
                        meter_state: torch.Tensor | None = None, err: torch.Tensor | None = None, stream=None):
    """kvq_decode_attn_noalloc: decode_attn with the library's own static scratch (no workspace argument).

    For callers that cannot allocate device scratch; calls share the library's scratch array, so
    calls must not overlap on the GPU."""
    B, Hq, D = q.shape
    assert D == HEAD_DIM and q.is_contiguous() and out.is_contiguous()
    assert block_table.dtype == torch.int32 and seq_lens.dtype == torch.int32
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(HEAD_DIM)
    d = cache.desc()
    pd = prefix.desc() if prefix is not None else None
    _check(lib().kvq_decode_attn_noalloc(
        ctypes.byref(d), ctypes.byref(pd) if pd is not None else None, int(prefix_len), q.data_ptr(), DTYPE[q.dtype],
        B, Hq, block_table.data_ptr(), int(block_table.shape[1]) if block_table.dim() == 2 else 0,
        seq_lens.data_ptr(), float(sm_scale), ctypes.byref(meter) if meter is not None else None,
        out.data_ptr(), _ptr(meter_state), _ptr(err), _stream(stream)), "kvq_decode_attn_noalloc")


def meter(meter_state: torch.Tensor, n_layers: int, batch: int, num_q_heads: int, params: MeterParams,
          meter_a: torch.Tensor, raw_a: torch.Tensor, counts: torch.Tensor, cert_b: torch.Tensor | None = None,
          ranking: torch.Tensor | None = None, out_bound: torch.Tensor | None = None,
          two_sided: torch.Tensor | None = None, det_tanh: torch.Tensor | None = None, stream=None):
    """kvq_meter over meter_state [L, B, Hq, 8]."""
    _check(lib().kvq_meter(meter_state.data_ptr(), n_layers, batch, num_q_heads, ctypes.byref(params),
                           meter_a.data_ptr(), raw_a.data_ptr(), _ptr(cert_b), _ptr(out_bound), _ptr(two_sided),
                           _ptr(det_tanh), counts.data_ptr(), _ptr(ranking), _stream(stream)), "kvq_meter")


def debug_dither(seed: int, layer: int, kv_head: int, slots: torch.Tensor, out: torch.Tensor, stream=None):
    _check(lib().kvq_debug_dither(seed & 0xFFFFFFFFFFFFFFFF, layer, kv_head, slots.data_ptr(), int(slots.numel()),
                                  out.data_ptr(), _stream(stream)), "kvq_debug_dither")


def debug_time_decode(start: "torch.cuda.Event | None", stop: "torch.cuda.Event | None"):
    """kvq_debug_time_decode: record these events around every decode kernel launch (None, None clears)."""
    if start is None or stop is None:
        _check(lib().kvq_debug_time_decode(None, None), "kvq_debug_time_decode")
        return
    _check(lib().kvq_debug_time_decode(start.cuda_event, stop.cuda_event), "kvq_debug_time_decode")


def debug_wait_timeout(limit_ns: int, err: torch.Tensor, stream=None):
    """kvq_debug_wait_timeout: a bounded wait that runs out; err receives KVQ_ERR_TIMEOUT."""
    _check(lib().kvq_debug_wait_timeout(int(limit_ns), err.data_ptr(), _stream(stream)), "kvq_debug_wait_timeout")


def debug_encode(kind: int, x: torch.Tensor, out: torch.Tensor, stream=None):
    _check(lib().kvq_debug_encode(kind, x.data_ptr(), int(x.numel()), out.data_ptr(), _stream(stream)),
           "kvq_debug_encode")
