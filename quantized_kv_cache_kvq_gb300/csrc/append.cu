// append.cu -- quantize-on-append: K/V codes, fp16 scales and the band-norm witness written
// into the paged cache tiles (one warp per (token, kv head)).
//
// WitCert (arXiv 2607.28699) Sec. 4.2 "Subtractive dither": x_hat = s (round(x/s + xi) - xi),
// s = amax / (Q - 1/2), Q = 127.  Sec. 6.2.1: quantize with the stored fp16 scale.  Sec. 6.2.3:
// one scale per token (per channel group; here the whole 128-channel head), dither keyed by the
// slot.  Sec. 4.1 eq. (2): the witness w_{t,b} = ||r_{t,b}|| over 16 bands of RoPE pairs, fp16.
// "Compress the shared cartridge": BF16 keys, FP8 E4M3 values (K16/V8), E4M3 keys (K8/V8).
#include "kvq_common.cuh"

namespace kvq {
namespace {

struct Quantized4 {
  float xhat[4];   // exact reconstruction of the 4 channels (for the witness), K only
  float lo[4];     // lower bound of the residual x_hat - x (directed rounding)
  float hi[4];     // upper bound of the residual
};

// Store 4 consecutive channels c0..c0+3 of token t into a K tile (k16 or k8 layout).
template <int FMT>
__device__ __forceinline__ void store_k4(uint8_t* tile, int t, int c0, const uint32_t codes[4]) {
  if (FMT == KVQ_FMT_BF16) {
    uint2 w;
    w.x = codes[0] | (codes[1] << 16);
    w.y = codes[2] | (codes[3] << 16);
    *reinterpret_cast<uint2*>(tile + k16_offset(t, c0)) = w;  // c0 % 4 == 0: 8-byte aligned
  } else {
    const uint32_t w = codes[0] | (codes[1] << 8) | (codes[2] << 16) | (codes[3] << 24);
    *reinterpret_cast<uint32_t*>(tile + k8_offset(t, c0)) = w;
  }
}

template <int FMT>
__device__ __forceinline__ void store_v4(uint8_t* tile, int t, int c0, const uint32_t codes[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (FMT == KVQ_FMT_BF16)
      *reinterpret_cast<uint16_t*>(tile + v16_offset(t, c0 + i)) = static_cast<uint16_t>(codes[i]);
    else
      tile[v8_offset(t, c0 + i)] = static_cast<uint8_t>(codes[i]);
  }
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Quantize 4 channels of one row.  `amax` is the row's max |x| (exact), `xi` the dither (INT8).
// Returns codes (bit patterns) and the scale bits; fills the residual bounds when WANT_RES.
template <int FMT, bool WANT_RES>
__device__ __forceinline__ void quantize4(const float x[4], float amax, const float xi[4], uint32_t codes[4],
                                          uint16_t& scale_bits, Quantized4& q, int& flags) {
  if (FMT == KVQ_FMT_BF16 || FMT == KVQ_FMT_E4M3) {
    scale_bits = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float xh;
      if (FMT == KVQ_FMT_BF16) {
        codes[i] = f32_to_bf16_bits(x[i]);
        xh = bf16_bits_to_f32(codes[i]);
      } else {
        codes[i] = f32_to_e4m3_bits(x[i]);
        xh = e4m3_bits_to_f32(static_cast<uint8_t>(codes[i]));
      }
      if (WANT_RES) {
        q.xhat[i] = xh;
        q.hi[i] = __fsub_ru(xh, x[i]);
        q.lo[i] = __fsub_rd(xh, x[i]);
      }
    }
    return;
  }
  const float divisor = (FMT == KVQ_FMT_INT8_DITHER) ? 126.5f : 448.0f;
  const __half s16 = __float2half_rn(__fdiv_rn(amax, divisor));
  scale_bits = __half_as_ushort(s16);
  const float s = __half2float(s16);
  if (!(s <= 65504.0f)) flags |= 1;  // fp16 overflow (or NaN amax)
  if (FMT == KVQ_FMT_INT8_DITHER) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      int code = 0;
      if (s > 0.0f) {
        const float y = __fdiv_rn(x[i], s);
        const float y2 = __fadd_rn(y, xi[i]);
        code = __float2int_rn(y2);  // round half to even
        code = max(-127, min(127, code));
      }
      codes[i] = static_cast<uint32_t>(code) & 0xFFu;
      if (WANT_RES) {
        // residual r = s*code - s*xi - x, bracketed with directed-rounding FMAs
        const float fc = static_cast<float>(code);
        q.hi[i] = __fmaf_ru(-s, xi[i], __fmaf_ru(s, fc, -x[i]));
        q.lo[i] = __fmaf_rd(-s, xi[i], __fmaf_rd(s, fc, -x[i]));
        q.xhat[i] = 0.0f;
      }
    }
  } else {  // E4M3_SCALED
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t code = 0;
      if (s > 0.0f) code = f32_to_e4m3_bits(__fdiv_rn(x[i], s));
      codes[i] = code;
      if (WANT_RES) {
        const float xh = s * e4m3_bits_to_f32(static_cast<uint8_t>(code));  // exact: 11 x 4 bits
        q.hi[i] = __fsub_ru(xh, x[i]);
        q.lo[i] = __fsub_rd(xh, x[i]);
        q.xhat[i] = xh;
      }
    }
  }
}

template <int KF, int VF>
__global__ void __launch_bounds__(256) append_kernel(kvq_cache c, const void* __restrict__ kin,
                                                     const void* __restrict__ vin, int in_bf16,
                                                     const int32_t* __restrict__ slots, int num_tokens,
                                                     int32_t* err) {
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
  const int c0 = lane * 4;
  float k[4], v[4];
  const size_t base = static_cast<size_t>(row) * kHeadDim + c0;
  if (in_bf16) {
    const uint2 kw = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(kin) + base);
    const uint2 vw = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(vin) + base);
    k[0] = bf16_bits_to_f32(kw.x & 0xFFFFu); k[1] = bf16_bits_to_f32(kw.x >> 16);
    k[2] = bf16_bits_to_f32(kw.y & 0xFFFFu); k[3] = bf16_bits_to_f32(kw.y >> 16);
    v[0] = bf16_bits_to_f32(vw.x & 0xFFFFu); v[1] = bf16_bits_to_f32(vw.x >> 16);
    v[2] = bf16_bits_to_f32(vw.y & 0xFFFFu); v[3] = bf16_bits_to_f32(vw.y >> 16);
  } else {
    const float4 kf = *reinterpret_cast<const float4*>(static_cast<const float*>(kin) + base);
    const float4 vf = *reinterpret_cast<const float4*>(static_cast<const float*>(vin) + base);
    k[0] = kf.x; k[1] = kf.y; k[2] = kf.z; k[3] = kf.w;
    v[0] = vf.x; v[1] = vf.y; v[2] = vf.z; v[3] = vf.w;
  }
  bool finite = true;
#pragma unroll
  for (int i = 0; i < 4; ++i) finite = finite && isfinite(k[i]) && isfinite(v[i]);
  finite = __all_sync(0xffffffffu, finite);

  float xi[4] = {0.f, 0.f, 0.f, 0.f};
  if (KF == KVQ_FMT_INT8_DITHER || VF == KVQ_FMT_INT8_DITHER) {
    const float4 d = dither4(static_cast<uint32_t>(slot), static_cast<uint32_t>(c.layer), static_cast<uint32_t>(head),
                             static_cast<uint32_t>(lane), static_cast<uint32_t>(c.dither_seed),
                             static_cast<uint32_t>(c.dither_seed >> 32));
    xi[0] = d.x; xi[1] = d.y; xi[2] = d.z; xi[3] = d.w;
  }
  float kamax = 0.f, vamax = 0.f;
  if (fmt_has_scale(KF)) kamax = warp_max(fmaxf(fmaxf(fabsf(k[0]), fabsf(k[1])), fmaxf(fabsf(k[2]), fabsf(k[3]))));
  if (fmt_has_scale(VF)) vamax = warp_max(fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3]))));

  const size_t tile = static_cast<size_t>(page) * H + head;
  int flags = 0;
  Quantized4 qk;
  uint32_t kc[4], vc[4];
  uint16_t ks = 0, vs = 0;
  quantize4<KF, true>(k, kamax, xi, kc, ks, qk, flags);
  Quantized4 qv;
  quantize4<VF, false>(v, vamax, xi, vc, vs, qv, flags);
  store_k4<KF>(static_cast<uint8_t*>(c.k_data) + tile * tile_bytes_k(KF), t, c0, kc);
  store_v4<VF>(static_cast<uint8_t*>(c.v_data) + tile * tile_bytes_v(VF), t, c0, vc);
  if (lane == 0) {
    // scale planes are head-major: tile (page, head) at head * num_pages + page
    const size_t stile = static_cast<size_t>(head) * c.num_pages + page;
    if (fmt_has_scale(KF)) *reinterpret_cast<uint16_t*>(reinterpret_cast<uint8_t*>(c.k_scale) + stile * kTileBytesS + s_offset(t)) = ks;
    if (fmt_has_scale(VF)) {
      *reinterpret_cast<uint16_t*>(reinterpret_cast<uint8_t*>(c.v_scale) + stile * kTileBytesS + s_offset(t)) = vs;
      if (__half2float(__ushort_as_half(vs)) > KVQ_MAX_VALUE_SCALE) flags |= 2;
    }
  }
  // Witness: upper bound of each band norm.  Lane l holds channels 4l..4l+3, all in band l % 16;
  // lanes l and l + 16 share a band (channels 4b..4b+3 and 64+4b..64+4b+3).
  float ss = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float a = fmaxf(qk.hi[i], -qk.lo[i]);  // >= |r_i|
    ss = __fmaf_ru(a, a, ss);
  }
  ss = __fadd_ru(ss, __shfl_xor_sync(0xffffffffu, ss, 16));
  if (lane < 16) {
    const float w = __fsqrt_ru(ss);
    const uint16_t wb = __half_as_ushort(__float2half_ru(w));
    *reinterpret_cast<uint16_t*>(reinterpret_cast<uint8_t*>(c.witness) + tile * kTileBytesW + w_offset(t, lane)) = wb;
  }
  if (lane == 0) {
    if (!finite || (flags & 1)) report(err, KVQ_ERR_NONFINITE_INPUT);
    else if (flags & 2) report(err, KVQ_ERR_RANGE);
  }
}

template <int KF, int VF>
cudaError_t launch_append(const kvq_cache& c, const void* k, const void* v, int in_bf16, const int32_t* slots,
                          int n, int32_t* err, cudaStream_t s) {
  const long long rows = static_cast<long long>(n) * c.num_kv_heads;
  const int threads = 256;
  const long long blocks = (rows * 32 + threads - 1) / threads;
  append_kernel<KF, VF><<<static_cast<unsigned>(blocks), threads, 0, s>>>(c, k, v, in_bf16, slots, n, err);
  return cudaGetLastError();
}

template <int KF>
cudaError_t dispatch_v(int vf, const kvq_cache& c, const void* k, const void* v, int b, const int32_t* sl, int n,
                       int32_t* e, cudaStream_t s) {
  switch (vf) {
    case KVQ_FMT_BF16: return launch_append<KF, KVQ_FMT_BF16>(c, k, v, b, sl, n, e, s);
    case KVQ_FMT_E4M3: return launch_append<KF, KVQ_FMT_E4M3>(c, k, v, b, sl, n, e, s);
    case KVQ_FMT_E4M3_SCALED: return launch_append<KF, KVQ_FMT_E4M3_SCALED>(c, k, v, b, sl, n, e, s);
    case KVQ_FMT_INT8_DITHER: return launch_append<KF, KVQ_FMT_INT8_DITHER>(c, k, v, b, sl, n, e, s);
  }
  return cudaErrorInvalidValue;
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
  if (fmt < KVQ_FMT_BF16 || fmt > KVQ_FMT_INT8_DITHER) return 0;
  switch (plane) {
    case 0: return static_cast<size_t>(tile_bytes_k(fmt));
    case 1: return static_cast<size_t>(tile_bytes_v(fmt));
    case 2:
    case 3: return fmt_has_scale(fmt) ? static_cast<size_t>(kTileBytesS) : 0;
    case 4: return static_cast<size_t>(kTileBytesW);
  }
  return 0;
}

extern "C" kvq_status kvq_append(const kvq_cache* c, const void* k, const void* v, int32_t in_dtype,
                                 const int32_t* slot_mapping, int32_t num_tokens, int32_t* err,
                                 kvq_stream_t stream) {
  if (!c || num_tokens < 0 || (in_dtype != KVQ_DTYPE_F32 && in_dtype != KVQ_DTYPE_BF16)) return KVQ_ERR_INVALID_ARG;
  if (c->k_fmt < 0 || c->k_fmt > 3 || c->v_fmt < 0 || c->v_fmt > 3) return KVQ_ERR_UNSUPPORTED_LAYOUT;
  if (c->num_kv_heads <= 0 || c->num_pages < 0 || c->reserved != 0) return KVQ_ERR_INVALID_ARG;
  if (num_tokens == 0) return KVQ_OK;
  if (!k || !v || !slot_mapping || !c->k_data || !c->v_data || !c->witness) return KVQ_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(c->k_data) || !aligned16(c->v_data) || !aligned16(c->witness))
    return KVQ_ERR_INVALID_ARG;
  if (fmt_has_scale(c->k_fmt) && (!c->k_scale || !aligned16(c->k_scale))) return KVQ_ERR_INVALID_ARG;
  if (fmt_has_scale(c->v_fmt) && (!c->v_scale || !aligned16(c->v_scale))) return KVQ_ERR_INVALID_ARG;
  const int in_bf16 = in_dtype == KVQ_DTYPE_BF16;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaErrorInvalidValue;
  switch (c->k_fmt) {
    case KVQ_FMT_BF16: e = dispatch_v<KVQ_FMT_BF16>(c->v_fmt, *c, k, v, in_bf16, slot_mapping, num_tokens, err, s); break;
    case KVQ_FMT_E4M3: e = dispatch_v<KVQ_FMT_E4M3>(c->v_fmt, *c, k, v, in_bf16, slot_mapping, num_tokens, err, s); break;
    case KVQ_FMT_E4M3_SCALED: e = dispatch_v<KVQ_FMT_E4M3_SCALED>(c->v_fmt, *c, k, v, in_bf16, slot_mapping, num_tokens, err, s); break;
    case KVQ_FMT_INT8_DITHER: e = dispatch_v<KVQ_FMT_INT8_DITHER>(c->v_fmt, *c, k, v, in_bf16, slot_mapping, num_tokens, err, s); break;
  }
  return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
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
