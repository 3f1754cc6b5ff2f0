// append.cu -- quantize-on-append: K/V codes, fp16 scales and the band-norm witness written
// into the paged cache tiles (one warp per (token, kv head)).
//
// WitCert (arXiv 2607.28699) Sec. 4.2 "Subtractive dither": x_hat = s (round(x/s + xi) - xi),
// s = amax / (Q - 1/2), Q = 127.  Sec. 6.2.1: quantize with the stored fp16 scale.  Sec. 6.2.3:
// one scale per token per channel group (the whole 128-channel head, or 32-channel groups), dither
// keyed by the slot.  Sec. 4.1 eq. (2): the witness w_{t,b} = ||r_{t,b}|| over 16 bands of RoPE pairs, fp16.
// "Compress the shared cartridge": BF16 keys, FP8 E4M3 values (K16/V8), E4M3 keys (K8/V8).
#include "quant_row.cuh"

namespace kvq {
namespace {

// RoPE-on-append (kvq_append_rope): the caller's binary32 cos/sin table and each token's position.
struct RopeArgs {
  const int32_t* positions;
  const float* cos_sin;  // [max_pos][128]: cos of pairs 0..63, then their sin
  int max_pos;
};

// Rotate this lane's four key channels (half-split pairs: channel j with j + 64, j = 0..63; lanes 0..15
// hold channels 0..63, lanes 16..31 their partners).  Each channel is two rounded products and one
// rounded sum, no fused multiply-add: x' = x c - y s, y' = y c + x s.
__device__ __forceinline__ void rope_rotate4(float k[4], const float* row, int lane) {
  const int j0 = 4 * (lane & 15);
  const float4 cs = *reinterpret_cast<const float4*>(row + j0);
  const float4 sn = *reinterpret_cast<const float4*>(row + kHeadDim / 2 + j0);
  const float c[4] = {cs.x, cs.y, cs.z, cs.w}, s[4] = {sn.x, sn.y, sn.z, sn.w};
  float partner[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) partner[e] = __shfl_xor_sync(0xffffffffu, k[e], 16);
#pragma unroll
  for (int e = 0; e < 4; ++e)
    k[e] = lane < 16 ? __fsub_rn(__fmul_rn(k[e], c[e]), __fmul_rn(partner[e], s[e]))
                     : __fadd_rn(__fmul_rn(k[e], c[e]), __fmul_rn(partner[e], s[e]));
}

template <int KF, int VF, bool ROPE = false>
__global__ void __launch_bounds__(256, 1) append_kernel(kvq_cache c, const void* __restrict__ kin,
                                                     const void* __restrict__ vin, int in_bf16,
                                                     const int32_t* __restrict__ slots, int num_tokens,
                                                     int32_t* err, RopeArgs rope) {
  const int lane = threadIdx.x & 31;
  const long long row = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int H = c.num_kv_heads;
  if (row >= static_cast<long long>(num_tokens) * H) return;
  const int tok = static_cast<int>(row / H);
  const int head = static_cast<int>(row % H);
  const int slot = slots[tok];
  if (slot < 0) return;
  const int page = slot >> 4;
  const int t = slot & 15;
  if (page >= c.num_pages) {
    if (lane == 0) report(err, KVQ_ERR_DEVICE_BOUNDS);
    return;
  }
  float k[4], v[4];
  load_row4(kin, vin, in_bf16, static_cast<size_t>(row) * kHeadDim + lane * 4, k, v);
  if (ROPE) {  // the key arrives pre-RoPE: rotate it at the token's position (one position per warp)
    const int pos = rope.positions[tok];
    if (pos < 0 || pos >= rope.max_pos) {
      if (lane == 0) report(err, KVQ_ERR_DEVICE_BOUNDS);
      return;
    }
    rope_rotate4(k, rope.cos_sin + static_cast<size_t>(pos) * kHeadDim, lane);
  }
  const RowCodes rc = quantize_row<KF, VF>(k, v, static_cast<uint32_t>(slot), static_cast<uint32_t>(c.layer),
                                           static_cast<uint32_t>(head), c.dither_seed, c.v_witness != nullptr,
                                           c.n_outlier_pairs > 0 ? c.outlier_pairs + head * c.n_outlier_pairs : nullptr,
                                           c.n_outlier_pairs);
  const size_t tile = static_cast<size_t>(page) * H + head;
  const size_t stile = static_cast<size_t>(head) * c.num_pages + page;  // scale planes are head-major
  store_row<KF, VF>(rc, t, static_cast<uint8_t*>(c.k_data) + tile * tile_bytes_k(KF),
                    static_cast<uint8_t*>(c.v_data) + tile * tile_bytes_v(VF),
                    fmt_has_scale(KF) ? reinterpret_cast<uint8_t*>(c.k_scale) + stile * tile_bytes_s(KF) : nullptr,
                    fmt_has_scale(VF) ? reinterpret_cast<uint8_t*>(c.v_scale) + stile * tile_bytes_s(VF) : nullptr,
                    reinterpret_cast<uint8_t*>(c.witness) + tile * kTileBytesW,
                    c.v_witness ? reinterpret_cast<uint8_t*>(c.v_witness) + stile * kTileBytesVW : nullptr,
                    c.n_outlier_pairs > 0
                        ? reinterpret_cast<uint8_t*>(c.k_outlier) + stile * outlier_tile_bytes(c.n_outlier_pairs)
                        : nullptr,
                    c.n_outlier_pairs > 4);
  if (lane == 0) report_row(rc, err);
}

// The newest token of every sequence (live position seq_lens[s] - 1, its slot from the block
// table), one warp per (sequence, kv head); launched ahead of a decode that waits for it only where
// it reads those pages (programmatic dependent launch).
template <int KF, int VF>
__global__ void __launch_bounds__(256, 1) append_newest_kernel(kvq_cache c, const void* __restrict__ kin,
                                                            const void* __restrict__ vin, int in_bf16,
                                                            const int32_t* __restrict__ block_table, int max_pages,
                                                            const int32_t* __restrict__ seq_lens, int batch,
                                                            int32_t* err) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const long long row = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int H = c.num_kv_heads;
  if (row >= static_cast<long long>(batch) * H) return;
  const int seq = static_cast<int>(row / H);
  const int head = static_cast<int>(row % H);
  const int len = seq_lens[seq];
  if (len <= 0) return;
  if (len > max_pages * kPage) {
    if (lane == 0) report(err, KVQ_ERR_DEVICE_BOUNDS);
    return;
  }
  const int pos = len - 1;
  const int page = block_table[static_cast<size_t>(seq) * max_pages + pos / kPage];
  const int t = pos % kPage;
  if (page < 0 || page >= c.num_pages) {
    if (lane == 0) report(err, KVQ_ERR_DEVICE_BOUNDS);
    return;
  }
  const int slot = page * kPage + t;
  float k[4], v[4];
  load_row4(kin, vin, in_bf16, static_cast<size_t>(row) * kHeadDim + lane * 4, k, v);
  const RowCodes rc = quantize_row<KF, VF>(k, v, static_cast<uint32_t>(slot), static_cast<uint32_t>(c.layer),
                                           static_cast<uint32_t>(head), c.dither_seed, c.v_witness != nullptr,
                                           c.n_outlier_pairs > 0 ? c.outlier_pairs + head * c.n_outlier_pairs : nullptr,
                                           c.n_outlier_pairs);
  const size_t tile = static_cast<size_t>(page) * H + head;
  const size_t stile = static_cast<size_t>(head) * c.num_pages + page;
  store_row<KF, VF>(rc, t, static_cast<uint8_t*>(c.k_data) + tile * tile_bytes_k(KF),
                    static_cast<uint8_t*>(c.v_data) + tile * tile_bytes_v(VF),
                    fmt_has_scale(KF) ? reinterpret_cast<uint8_t*>(c.k_scale) + stile * tile_bytes_s(KF) : nullptr,
                    fmt_has_scale(VF) ? reinterpret_cast<uint8_t*>(c.v_scale) + stile * tile_bytes_s(VF) : nullptr,
                    reinterpret_cast<uint8_t*>(c.witness) + tile * kTileBytesW,
                    c.v_witness ? reinterpret_cast<uint8_t*>(c.v_witness) + stile * kTileBytesVW : nullptr,
                    c.n_outlier_pairs > 0
                        ? reinterpret_cast<uint8_t*>(c.k_outlier) + stile * outlier_tile_bytes(c.n_outlier_pairs)
                        : nullptr,
                    c.n_outlier_pairs > 4);
  if (lane == 0) report_row(rc, err);
}

struct NewestArgs {
  const int32_t* block_table;
  int max_pages;
  const int32_t* seq_lens;
  int batch;
};

template <int KF, int VF>
cudaError_t launch_append(const kvq_cache& c, const void* k, const void* v, int in_bf16, const int32_t* slots,
                          int n, int32_t* err, cudaStream_t s, const RopeArgs* rope) {
  const long long rows = static_cast<long long>(n) * c.num_kv_heads;
  const int threads = 256;
  const long long blocks = (rows * 32 + threads - 1) / threads;
  if (rope)
    append_kernel<KF, VF, true><<<static_cast<unsigned>(blocks), threads, 0, s>>>(c, k, v, in_bf16, slots, n, err,
                                                                                  *rope);
  else
    append_kernel<KF, VF, false><<<static_cast<unsigned>(blocks), threads, 0, s>>>(c, k, v, in_bf16, slots, n, err,
                                                                                   RopeArgs{nullptr, nullptr, 0});
  return cudaGetLastError();
}

template <int KF, int VF>
cudaError_t launch_any(const kvq_cache& c, const void* k, const void* v, int in_bf16, const int32_t* slots, int n,
                       int32_t* err, cudaStream_t s, const NewestArgs* newest, const RopeArgs* rope) {
  const int threads = 256;
  if (newest) {
    const long long rows = static_cast<long long>(newest->batch) * c.num_kv_heads;
    const long long blocks = (rows * 32 + threads - 1) / threads;
    append_newest_kernel<KF, VF><<<static_cast<unsigned>(blocks), threads, 0, s>>>(
        c, k, v, in_bf16, newest->block_table, newest->max_pages, newest->seq_lens, newest->batch, err);
    return cudaGetLastError();
  }
  return launch_append<KF, VF>(c, k, v, in_bf16, slots, n, err, s, rope);
}

template <int KF>
cudaError_t dispatch_v(int vf, const kvq_cache& c, const void* k, const void* v, int b, const int32_t* sl, int n,
                       int32_t* e, cudaStream_t s, const NewestArgs* nw = nullptr, const RopeArgs* rp = nullptr) {
  if constexpr (KF == KVQ_FMT_INT8_DITHER_G32) {  // group-scaled INT8 keys go with group-scaled INT8 values only
    return vf == KVQ_FMT_INT8_DITHER_G32 ? launch_any<KF, KVQ_FMT_INT8_DITHER_G32>(c, k, v, b, sl, n, e, s, nw, rp)
                                         : cudaErrorInvalidValue;
  } else {
    switch (vf) {
      case KVQ_FMT_BF16: return launch_any<KF, KVQ_FMT_BF16>(c, k, v, b, sl, n, e, s, nw, rp);
      case KVQ_FMT_E4M3: return launch_any<KF, KVQ_FMT_E4M3>(c, k, v, b, sl, n, e, s, nw, rp);
      case KVQ_FMT_E4M3_SCALED: return launch_any<KF, KVQ_FMT_E4M3_SCALED>(c, k, v, b, sl, n, e, s, nw, rp);
      case KVQ_FMT_INT8_DITHER: return launch_any<KF, KVQ_FMT_INT8_DITHER>(c, k, v, b, sl, n, e, s, nw, rp);
    }
    return cudaErrorInvalidValue;
  }
}

// zero the witness (and value witness) of repaired slots: one thread per (slot, kv head)
__global__ void zero_witness_kernel(kvq_cache c, const int32_t* __restrict__ slots, int n, int32_t* err) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int H = c.num_kv_heads;
  if (i >= static_cast<long long>(n) * H) return;
  const int slot = slots[i / H], head = static_cast<int>(i % H);
  if (slot < 0) return;
  const int page = slot >> 4, t = slot & 15;
  if (page >= c.num_pages) {
    report(err, KVQ_ERR_DEVICE_BOUNDS);
    return;
  }
  uint8_t* w = reinterpret_cast<uint8_t*>(c.witness) + (static_cast<size_t>(page) * H + head) * kTileBytesW;
#pragma unroll
  for (int b = 0; b < 16; ++b) *reinterpret_cast<uint16_t*>(w + w_offset(t, b)) = 0;
  if (c.v_witness) {
    uint8_t* vw = reinterpret_cast<uint8_t*>(c.v_witness) + (static_cast<size_t>(head) * c.num_pages + page) * kTileBytesVW;
    *reinterpret_cast<uint16_t*>(vw + vw_offset(t, 0)) = 0;
    *reinterpret_cast<uint16_t*>(vw + vw_offset(t, 1)) = 0;
  }
}

__global__ void debug_dither_kernel(uint64_t seed, int layer, int head, const int32_t* slots, int n, float* out) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;  // one thread per group
  if (i >= static_cast<long long>(n) * 32) return;
  const int row = static_cast<int>(i >> 5), g = static_cast<int>(i & 31);
  const float4 d = dither4(static_cast<uint32_t>(slots[row]), static_cast<uint32_t>(layer), static_cast<uint32_t>(head),
                           static_cast<uint32_t>(g), static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32));
  reinterpret_cast<float4*>(out)[i] = d;
}

__global__ void debug_encode_kernel(int kind, const float* x, long long n, void* out) {
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const float v = x[i];
    switch (kind) {
      case 0: static_cast<uint16_t*>(out)[i] = f32_to_bf16_bits(v); break;
      case 1: static_cast<uint8_t*>(out)[i] = f32_to_e4m3_bits(v); break;
      case 2: static_cast<uint16_t*>(out)[i] = __half_as_ushort(__float2half_rn(v)); break;
      default: static_cast<uint16_t*>(out)[i] = __half_as_ushort(__float2half_ru(v)); break;
    }
  }
}

}  // namespace
}  // namespace kvq

using namespace kvq;

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

extern "C" size_t kvq_tile_bytes(int32_t fmt, int32_t plane) {
  if (fmt < KVQ_FMT_BF16 || fmt > KVQ_FMT_INT8_DITHER_G32) return 0;
  switch (plane) {
    case 0: return static_cast<size_t>(tile_bytes_k(fmt));
    case 1: return static_cast<size_t>(tile_bytes_v(fmt));
    case 2:
    case 3: return fmt_has_scale(fmt) ? static_cast<size_t>(tile_bytes_s(fmt)) : 0;
    case 4: return static_cast<size_t>(kTileBytesW);
    case 5: return static_cast<size_t>(kTileBytesVW);
    case 6: return fmt == KVQ_FMT_INT8_DITHER ? static_cast<size_t>(outlier_tile_bytes(4)) : 0;
    case 7: return fmt == KVQ_FMT_INT8_DITHER ? static_cast<size_t>(outlier_tile_bytes(8)) : 0;
  }
  return 0;
}

extern "C" size_t kvq_sizeof(int32_t which) {
  switch (which) {
    case 0: return sizeof(kvq_cache);
    case 1: return sizeof(kvq_meter_params);
  }
  return 0;
}

namespace {
// The checks of kvq_append and kvq_append_rope, then the launch (rope: nullptr for post-RoPE keys).
kvq_status append_impl(const kvq_cache* c, const void* k, const void* v, int32_t in_dtype,
                       const int32_t* slot_mapping, int32_t num_tokens, int32_t* err, kvq_stream_t stream,
                       const RopeArgs* rope) {
  if (!c || num_tokens < 0 || (in_dtype != KVQ_DTYPE_F32 && in_dtype != KVQ_DTYPE_BF16)) return KVQ_ERR_INVALID_ARG;
  if (c->k_fmt < 0 || c->k_fmt > 4 || c->v_fmt < 0 || c->v_fmt > 4) return KVQ_ERR_UNSUPPORTED_LAYOUT;
  if ((c->k_fmt == KVQ_FMT_INT8_DITHER_G32) != (c->v_fmt == KVQ_FMT_INT8_DITHER_G32)) return KVQ_ERR_UNSUPPORTED_LAYOUT;
  if (c->num_kv_heads <= 0 || c->num_pages < 0 || c->reserved != 0) return KVQ_ERR_INVALID_ARG;
  if (num_tokens == 0) return KVQ_OK;
  if (!k || !v || !slot_mapping || !c->k_data || !c->v_data || !c->witness) return KVQ_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(c->k_data) || !aligned16(c->v_data) || !aligned16(c->witness))
    return KVQ_ERR_INVALID_ARG;
  if (fmt_has_scale(c->k_fmt) && (!c->k_scale || !aligned16(c->k_scale))) return KVQ_ERR_INVALID_ARG;
  if (fmt_has_scale(c->v_fmt) && (!c->v_scale || !aligned16(c->v_scale))) return KVQ_ERR_INVALID_ARG;
  if (c->v_witness && !aligned16(c->v_witness)) return KVQ_ERR_INVALID_ARG;
  if (c->n_outlier_pairs < 0 || c->n_outlier_pairs > kMaxOutlierPairs || c->reserved2 != 0) return KVQ_ERR_INVALID_ARG;
  if (c->n_outlier_pairs > 0) {
    if (c->k_fmt != KVQ_FMT_INT8_DITHER) return KVQ_ERR_UNSUPPORTED_LAYOUT;
    if (!c->outlier_pairs || !c->k_outlier || !aligned16(c->k_outlier)) return KVQ_ERR_INVALID_ARG;
  }
  if (rope && (!rope->positions || !rope->cos_sin || !aligned16(rope->cos_sin) || rope->max_pos <= 0))
    return KVQ_ERR_INVALID_ARG;
  const int in_bf16 = in_dtype == KVQ_DTYPE_BF16;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaErrorInvalidValue;
  const NewestArgs* no_newest = nullptr;
  switch (c->k_fmt) {
    case KVQ_FMT_BF16:
      e = dispatch_v<KVQ_FMT_BF16>(c->v_fmt, *c, k, v, in_bf16, slot_mapping, num_tokens, err, s, no_newest, rope);
      break;
    case KVQ_FMT_E4M3:
      e = dispatch_v<KVQ_FMT_E4M3>(c->v_fmt, *c, k, v, in_bf16, slot_mapping, num_tokens, err, s, no_newest, rope);
      break;
    case KVQ_FMT_E4M3_SCALED:
      e = dispatch_v<KVQ_FMT_E4M3_SCALED>(c->v_fmt, *c, k, v, in_bf16, slot_mapping, num_tokens, err, s, no_newest,
                                          rope);
      break;
    case KVQ_FMT_INT8_DITHER:
      e = dispatch_v<KVQ_FMT_INT8_DITHER>(c->v_fmt, *c, k, v, in_bf16, slot_mapping, num_tokens, err, s, no_newest,
                                          rope);
      break;
    case KVQ_FMT_INT8_DITHER_G32:
      e = dispatch_v<KVQ_FMT_INT8_DITHER_G32>(c->v_fmt, *c, k, v, in_bf16, slot_mapping, num_tokens, err, s,
                                              no_newest, rope);
      break;
  }
  return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}
}  // namespace

extern "C" kvq_status kvq_append(const kvq_cache* c, const void* k, const void* v, int32_t in_dtype,
                                 const int32_t* slot_mapping, int32_t num_tokens, int32_t* err,
                                 kvq_stream_t stream) {
  return append_impl(c, k, v, in_dtype, slot_mapping, num_tokens, err, stream, nullptr);
}

extern "C" kvq_status kvq_append_rope(const kvq_cache* c, const void* k_pre, const void* v, int32_t in_dtype,
                                      const int32_t* positions, const float* cos_sin, int32_t max_position,
                                      const int32_t* slot_mapping, int32_t num_tokens, int32_t* err,
                                      kvq_stream_t stream) {
  const RopeArgs rope{positions, cos_sin, max_position};
  return append_impl(c, k_pre, v, in_dtype, slot_mapping, num_tokens, err, stream, &rope);
}

namespace kvq {
// Library-internal: the append kernel of kvq_decode_attn_append (arguments checked by the caller).
cudaError_t launch_append_newest(const kvq_cache& c, const void* k, const void* v, int in_bf16,
                                 const int32_t* block_table, int max_pages, const int32_t* seq_lens, int batch,
                                 int32_t* err, cudaStream_t s) {
  const NewestArgs nw{block_table, max_pages, seq_lens, batch};
  switch (c.k_fmt) {
    case KVQ_FMT_BF16: return dispatch_v<KVQ_FMT_BF16>(c.v_fmt, c, k, v, in_bf16, nullptr, 0, err, s, &nw);
    case KVQ_FMT_E4M3: return dispatch_v<KVQ_FMT_E4M3>(c.v_fmt, c, k, v, in_bf16, nullptr, 0, err, s, &nw);
    case KVQ_FMT_E4M3_SCALED: return dispatch_v<KVQ_FMT_E4M3_SCALED>(c.v_fmt, c, k, v, in_bf16, nullptr, 0, err, s, &nw);
    case KVQ_FMT_INT8_DITHER: return dispatch_v<KVQ_FMT_INT8_DITHER>(c.v_fmt, c, k, v, in_bf16, nullptr, 0, err, s, &nw);
    case KVQ_FMT_INT8_DITHER_G32:
      return dispatch_v<KVQ_FMT_INT8_DITHER_G32>(c.v_fmt, c, k, v, in_bf16, nullptr, 0, err, s, &nw);
  }
  return cudaErrorInvalidValue;
}
}  // namespace kvq

extern "C" kvq_status kvq_zero_witness(const kvq_cache* c, const int32_t* slots, int32_t n, int32_t* err,
                                       kvq_stream_t stream) {
  if (!c || n < 0 || c->num_kv_heads <= 0 || c->num_pages < 0) return KVQ_ERR_INVALID_ARG;
  if (n == 0) return KVQ_OK;
  if (!slots || !c->witness) return KVQ_ERR_INVALID_ARG;
  const long long threads = static_cast<long long>(n) * c->num_kv_heads;
  zero_witness_kernel<<<static_cast<unsigned>((threads + 255) / 256), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      *c, slots, n, err);
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

extern "C" kvq_status kvq_debug_dither(uint64_t seed, int32_t layer, int32_t kv_head, const int32_t* slots, int32_t n,
                                       float* xi, kvq_stream_t stream) {
  if (n < 0 || (n > 0 && (!slots || !xi || !aligned16(xi)))) return KVQ_ERR_INVALID_ARG;
  if (n == 0) return KVQ_OK;
  const long long threads = static_cast<long long>(n) * 32;
  debug_dither_kernel<<<static_cast<unsigned>((threads + 255) / 256), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      seed, layer, kv_head, slots, n, xi);
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

extern "C" kvq_status kvq_debug_encode(int32_t kind, const float* x, int64_t n, void* out, kvq_stream_t stream) {
  if (kind < 0 || kind > 3 || n < 0 || (n > 0 && (!x || !out))) return KVQ_ERR_INVALID_ARG;
  if (n == 0) return KVQ_OK;
  long long blocks = (n + 255) / 256;
  if (blocks > 65535LL * 16) blocks = 65535LL * 16;
  debug_encode_kernel<<<static_cast<unsigned>(blocks), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(kind, x, n, out);
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}
