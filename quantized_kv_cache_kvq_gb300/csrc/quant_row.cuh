// quant_row.cuh -- quantize-on-append of one (token, kv head) row by one warp: K / V codes, fp16
// scales and the band-norm witness, for the append kernel and for the decode that appends each
// sequence's newest token itself.  Lane l holds channels 4l .. 4l+3.
//
// WitCert (arXiv 2607.28699) Sec. 4.2 "Subtractive dither": x_hat = s (round(x/s + xi) - xi),
// s = amax / (Q - 1/2), Q = 127.  Sec. 6.2.1: quantize with the stored fp16 scale.  Sec. 6.2.3:
// one scale per token per channel group (the whole 128-channel head, or groups of 32 channels, the
// 8 lanes 8g..8g+7), dither keyed by the slot.  Sec. 4.1 eq. (2): the witness w_{t,b} = ||r_{t,b}||
// over 16 bands of RoPE pairs, fp16.
// "Compress the shared cartridge": BF16 keys, FP8 E4M3 values (K16/V8), E4M3 keys (K8/V8).
#pragma once

#include "kvq_common.cuh"

namespace kvq {

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
    *reinterpret_cast<uint32_t*>(tile + (fmt_group_scales(FMT) ? k8g_offset(t, c0) : k8_offset(t, c0))) = w;
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
// max over the 8 lanes of one 32-channel scale group
__device__ __forceinline__ float group_max(float v) {
#pragma unroll
  for (int o = 4; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
// the amax a lane's scale is taken over: its 32-channel group or the whole row
template <int FMT>
__device__ __forceinline__ float scale_amax(float v) {
  return fmt_group_scales(FMT) ? group_max(v) : warp_max(v);
}

// Quantize 4 channels of one row.  `amax` is the max |x| (exact) over the channels that share this
// lane's scale (the row, or its 32-channel group), `xi` the dither (INT8).
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
  const float divisor = fmt_is_int8(FMT) ? 126.5f : 448.0f;
  const __half s16 = __float2half_rn(__fdiv_rn(amax, divisor));
  scale_bits = __half_as_ushort(s16);
  const float s = __half2float(s16);
  if (!(s <= 65504.0f)) flags |= 1;  // fp16 overflow (or NaN amax)
  if (fmt_is_int8(FMT)) {
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

// The four channels of this lane from row-major [.., 128] K and V inputs (fp32 or bf16).
__device__ __forceinline__ void load_row4(const void* kin, const void* vin, int in_bf16, size_t base, float k[4],
                                          float v[4]) {
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
}

// One row's stored form, as held by the lanes of the warp.
struct RowCodes {
  uint32_t kc[4], vc[4];  // this lane's four K and V codes
  uint16_t ks, vs;        // scale bits (formats with a scale; with group scales, this lane's group)
  uint16_t wb;            // witness bits of band `lane` (lanes 0..15)
  uint16_t vrho, vnorm;   // value witness bits: ||v_hat - v|| and ||v||, rounded up (warp-uniform)
  uint16_t kob[4];        // fp16 bits of this lane's bypassed key channels ...
  int8_t kocol[4];        // ... and their outlier columns (-1: not bypassed)
  bool nonfinite;         // non-finite input or scale overflow (warp-uniform)
  bool range;             // value scale above KVQ_MAX_VALUE_SCALE (warp-uniform)
  bool bad_pair;          // a bypassed pair index outside 0..63 (warp-uniform)
};

// want_vw: compute the value witness (the cache has a value witness plane).  opairs / m: the head's
// bypassed RoPE pairs (INT8-dithered keys; WitCert Sec. 6.2.5), m = 0 for none.
template <int KF, int VF>
__device__ __forceinline__ RowCodes quantize_row(const float k[4], const float v[4], uint32_t slot, uint32_t layer,
                                                 uint32_t head, uint64_t seed, bool want_vw,
                                                 const int32_t* opairs = nullptr, int m = 0) {
  const int lane = threadIdx.x & 31;
  RowCodes rc;
  bool finite = true;
#pragma unroll
  for (int i = 0; i < 4; ++i) finite = finite && isfinite(k[i]) && isfinite(v[i]);
  finite = __all_sync(0xffffffffu, finite);
  float xi[4] = {0.f, 0.f, 0.f, 0.f};
  if (fmt_is_int8(KF) || fmt_is_int8(VF)) {
    const float4 d = dither4(slot, layer, head, static_cast<uint32_t>(lane), static_cast<uint32_t>(seed),
                             static_cast<uint32_t>(seed >> 32));
    xi[0] = d.x; xi[1] = d.y; xi[2] = d.z; xi[3] = d.w;
  }
  // bypassed channels of this lane: column 2i <- channel pairs[i], column 2i + 1 <- pairs[i] + 64
  bool bad_pair = false;
#pragma unroll
  for (int e = 0; e < 4; ++e) rc.kocol[e] = -1;
  if (KF == KVQ_FMT_INT8_DITHER) {
    for (int i = 0; i < m; ++i) {
      const int j = opairs[i];
      if (j < 0 || j >= kHeadDim / 2) { bad_pair = true; continue; }
      if ((j >> 2) == lane) rc.kocol[j & 3] = static_cast<int8_t>(2 * i);
      if (((j + kHeadDim / 2) >> 2) == lane) rc.kocol[j & 3] = static_cast<int8_t>(2 * i + 1);
    }
  }
  float kamax = 0.f, vamax = 0.f;
  if (fmt_has_scale(KF)) {
    float a = 0.f;  // bypassed channels are left out of the amax
#pragma unroll
    for (int e = 0; e < 4; ++e) a = rc.kocol[e] < 0 ? fmaxf(a, fabsf(k[e])) : a;
    kamax = scale_amax<KF>(a);
  }
  if (fmt_has_scale(VF))
    vamax = scale_amax<VF>(fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3]))));
  int flags = 0;
  Quantized4 qk, qv;
  rc.ks = 0;
  rc.vs = 0;
  quantize4<KF, true>(k, kamax, xi, rc.kc, rc.ks, qk, flags);
  quantize4<VF, true>(v, vamax, xi, rc.vc, rc.vs, qv, flags);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    rc.kob[e] = 0;
    if (rc.kocol[e] >= 0) {  // bypassed: code 0, fp16 value, residual of the fp16 rounding
      const __half h = __float2half_rn(k[e]);
      const float hv = __half2float(h);
      rc.kob[e] = __half_as_ushort(h);
      rc.kc[e] = 0;
      qk.hi[e] = __fsub_ru(hv, k[e]);
      qk.lo[e] = __fsub_rd(hv, k[e]);
      if (!isfinite(hv)) flags |= 1;
    }
  }
  if (__any_sync(0xffffffffu, (flags & 1) != 0)) flags |= 1;  // an overflowing bypassed channel flags the row
  if (bad_pair) flags |= 4;
  // every group's value scale is checked (with group scales the lanes hold different ones)
  if (__any_sync(0xffffffffu, fmt_has_scale(VF) && __half2float(__ushort_as_half(rc.vs)) > KVQ_MAX_VALUE_SCALE))
    flags |= 2;
  // Witness: upper bound of each band norm.  Lane l holds channels 4l..4l+3, all in band l % 16;
  // lanes l and l + 16 share a band (channels 4b..4b+3 and 64+4b..64+4b+3).
  float ss = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float a = fmaxf(qk.hi[i], -qk.lo[i]);  // >= |r_i|
    ss = __fmaf_ru(a, a, ss);
  }
  ss = __fadd_ru(ss, __shfl_xor_sync(0xffffffffu, ss, 16));
  rc.wb = __half_as_ushort(__float2half_ru(__fsqrt_ru(ss)));
  // Value witness: upper bounds of ||v_hat - v|| and ||v|| over all 128 channels (sums rounded up)
  rc.vrho = 0;
  rc.vnorm = 0;
  if (want_vw) {  // warp-uniform
    float rv = 0.0f, vv = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float a = fmaxf(qv.hi[i], -qv.lo[i]);
      rv = __fmaf_ru(a, a, rv);
      vv = __fmaf_ru(v[i], v[i], vv);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      rv = __fadd_ru(rv, __shfl_xor_sync(0xffffffffu, rv, o));
      vv = __fadd_ru(vv, __shfl_xor_sync(0xffffffffu, vv, o));
    }
    rc.vrho = __half_as_ushort(__float2half_ru(__fsqrt_ru(rv)));
    rc.vnorm = __half_as_ushort(__float2half_ru(__fsqrt_ru(vv)));
  }
  rc.bad_pair = (flags & 4) != 0;
  rc.nonfinite = !finite || (flags & 1);  // flags are warp-uniform: amax and the scales are
  rc.range = (flags & 2) != 0;
  return rc;
}

// Write a row at token t into a page's tiles (global cache or a staged copy).  Scale or witness
// pointers may be null (plane absent).
template <int KF, int VF>
__device__ __forceinline__ void store_row(const RowCodes& rc, int t, uint8_t* ktile, uint8_t* vtile, uint8_t* kstile,
                                          uint8_t* vstile, uint8_t* wtile, uint8_t* vwtile, uint8_t* kotile = nullptr,
                                          bool ko_wide = false) {
  const int lane = threadIdx.x & 31;
  store_k4<KF>(ktile, t, lane * 4, rc.kc);
  store_v4<VF>(vtile, t, lane * 4, rc.vc);
  if (lane == 0) {
    if (fmt_has_scale(KF) && !fmt_group_scales(KF) && kstile) *reinterpret_cast<uint16_t*>(kstile + s_offset(t)) = rc.ks;
    if (fmt_has_scale(VF) && !fmt_group_scales(VF) && vstile) *reinterpret_cast<uint16_t*>(vstile + s_offset(t)) = rc.vs;
  }
  if ((lane & 7) == 0) {  // group scales: lane 8g holds group g's
    if (fmt_group_scales(KF) && kstile) *reinterpret_cast<uint16_t*>(kstile + gs_offset(t, lane >> 3)) = rc.ks;
    if (fmt_group_scales(VF) && vstile) *reinterpret_cast<uint16_t*>(vstile + gs_offset(t, lane >> 3)) = rc.vs;
  }
  if (wtile && lane < 16) *reinterpret_cast<uint16_t*>(wtile + w_offset(t, lane)) = rc.wb;
  if (vwtile && lane == 0) {
    *reinterpret_cast<uint16_t*>(vwtile + vw_offset(t, 0)) = rc.vrho;
    *reinterpret_cast<uint16_t*>(vwtile + vw_offset(t, 1)) = rc.vnorm;
  }
  if (kotile) {
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (rc.kocol[e] >= 0) *reinterpret_cast<uint16_t*>(kotile + ko_offset(t, rc.kocol[e], ko_wide)) = rc.kob[e];
  }
}

__device__ __forceinline__ void report_row(const RowCodes& rc, int32_t* err) {
  if (rc.bad_pair) report(err, KVQ_ERR_DEVICE_BOUNDS);
  else if (rc.nonfinite) report(err, KVQ_ERR_NONFINITE_INPUT);
  else if (rc.range) report(err, KVQ_ERR_RANGE);
}

}  // namespace kvq
