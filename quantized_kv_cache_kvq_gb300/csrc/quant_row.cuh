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
  // exact reconstruction of the 4 channels (for the witnesses): x_hat = xa * xb, a product that is exact in
  // double precision (INT8: s (code - xi); every other format: the binary32 value times 1)
  float xa[4], xb[4];
};

// ---------------------------------------------------------------------------------------------
// Exact norms rounded up to fp16 (WitCert Sec. 4.1 eq. (2): the witness ||r_b|| stored in fp16, rounded
// up so that it never under-states the norm; the value witness the same over a token's 128 channels).
// The result is the smallest fp16 value h with h^2 >= sum_i r_i^2 in exact arithmetic, r_i = x_hat_i - x_i
// (both exact doubles: x a binary32 input, x_hat a decoded code).  The sum of squares is bracketed with
// directed-rounding double arithmetic; a bracket that holds an fp16 square between h's predecessor and h
// (a sum within ~2^-50 of such a square) is decided exactly with ExactAcc.

// Exact sum of doubles that are integer multiples of 2^-320 below 2^300 in magnitude (every r_i is a multiple
// of 2^-149, its square's exact parts multiples of 2^-298): twenty signed 64-bit limbs of 32-bit digits,
// value = sum_k d[k] 2^(32 k - 320).  Each add changes a limb by less than 2^32, so 2^31 adds cannot overflow.
struct ExactAcc {
  long long d[20];
};
__device__ __forceinline__ void exact_clear(ExactAcc& a) {
#pragma unroll
  for (int k = 0; k < 20; ++k) a.d[k] = 0;
}
// (every limb index below is a compile-time constant after unrolling, so the limbs stay in registers)
__device__ __forceinline__ void exact_add(ExactAcc& a, double x) {
  if (x == 0.0) return;
  int e;
  const double m = frexp(x, &e);                               // x = m 2^e, 1/2 <= |m| < 1
  const long long M = static_cast<long long>(ldexp(m, 53));    // x = M 2^(e - 53), |M| < 2^53, exact
  unsigned long long mag = static_cast<unsigned long long>(M < 0 ? -M : M);
  int sh = e - 53 + 320;
  if (sh < 0) { mag >>= -sh; sh = 0; }                         // the dropped bits are zero (multiple of 2^-320)
  const int k = sh >> 5;
  const unsigned __int128 t = static_cast<unsigned __int128>(mag) << (sh & 31);   // < 2^85
  long long d0 = static_cast<long long>(static_cast<uint32_t>(t));
  long long d1 = static_cast<long long>(static_cast<uint32_t>(t >> 32));
  long long d2 = static_cast<long long>(t >> 64);
  if (M < 0) { d0 = -d0; d1 = -d1; d2 = -d2; }
#pragma unroll
  for (int j = 0; j < 20; ++j) a.d[j] += j == k ? d0 : j == k + 1 ? d1 : j == k + 2 ? d2 : 0ll;
}
// sign (-1, 0, 1) of the exact sum
__device__ __forceinline__ int exact_sign(ExactAcc a) {
#pragma unroll
  for (int k = 0; k < 19; ++k) {  // carries upward; limbs 0..18 end in [0, 2^32)
    const long long c = a.d[k] >> 32;
    a.d[k] -= c * 4294967296ll;
    a.d[k + 1] += c;
  }
  if (a.d[19] != 0) return a.d[19] > 0 ? 1 : -1;
  bool any = false;
#pragma unroll
  for (int k = 0; k < 19; ++k) any = any || a.d[k] != 0;
  return any ? 1 : 0;
}
// add r^2, r = xh - x, exactly: r = s + e by TwoSum, r^2 = s^2 + 2se + e^2, each product split exactly by an FMA
__device__ __forceinline__ void exact_add_square(ExactAcc& a, double xh, double x) {
  const double s = __dsub_rn(xh, x);
  const double bp = __dsub_rn(s, xh);
  const double e = __dadd_rn(__dsub_rn(xh, __dsub_rn(s, bp)), __dsub_rn(-x, bp));
  const double p1 = __dmul_rn(s, s), p2 = __dmul_rn(2.0 * s, e), p3 = __dmul_rn(e, e);
  exact_add(a, p1); exact_add(a, __fma_rn(s, s, -p1));
  exact_add(a, p2); exact_add(a, __fma_rn(2.0 * s, e, -p2));
  exact_add(a, p3); exact_add(a, __fma_rn(e, e, -p3));
}
// This lane's part [t_lo, t_hi] of the sum of squares of r_i = xa_i xb_i - x_i (directed rounding), in
// binary32 (the common path) or in double precision (the rare path).  One fused multiply-add rounds the exact
// r_i once, up or down.
__device__ __forceinline__ void abs_bracket(float up, float dn, float& a_lo, float& a_hi) {  // dn <= r <= up
  if (dn > 0.f) { a_lo = dn; a_hi = up; }
  else if (up < 0.f) { a_lo = -up; a_hi = -dn; }
  else { a_lo = 0.f; a_hi = fmaxf(-dn, up); }
}
__device__ __forceinline__ void sumsq_bracket32(const float* xa, const float* xb, const float* x,
                                                float& t_lo, float& t_hi) {
  t_lo = 0.f;
  t_hi = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float a_lo, a_hi;
    abs_bracket(__fmaf_ru(xa[i], xb[i], -x[i]), __fmaf_rd(xa[i], xb[i], -x[i]), a_lo, a_hi);
    t_hi = __fmaf_ru(a_hi, a_hi, t_hi);
    t_lo = __fmaf_rd(a_lo, a_lo, t_lo);
  }
}
__device__ __forceinline__ void sumsq_bracket64(const float* xa, const float* xb, const float* x,
                                                double& t_lo, double& t_hi) {
  t_lo = 0.0;
  t_hi = 0.0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const double xh = static_cast<double>(xa[i]) * static_cast<double>(xb[i]);  // exact
    const double up = __dsub_ru(xh, x[i]), dn = __dsub_rd(xh, x[i]);
    double a_lo, a_hi;
    if (dn > 0.0) { a_lo = dn; a_hi = up; }
    else if (up < 0.0) { a_lo = -up; a_hi = -dn; }
    else { a_lo = 0.0; a_hi = fmax(-dn, up); }
    t_hi = __fma_ru(a_hi, a_hi, t_hi);
    t_lo = __fma_rd(a_lo, a_lo, t_lo);
  }
}
// From a bracket [t_lo, t_hi] of the full sum: h0 = the smallest fp16 value whose square is >= t_hi (+inf
// above 65504), its predecessor, and whether the bracket decides the result (else it is h0 or pred, by the
// sign of sum - pred^2).  Squares of fp16 values are exact in binary32 (22 significant bits, >= 2^-48).
struct Fp16Pick {
  uint16_t h0, pred;
  bool decided;
};
__device__ __forceinline__ Fp16Pick fp16_ru_pick(float t_lo, float t_hi) {
  Fp16Pick p{0, 0, true};
  if (t_hi == 0.f) return p;  // every r_i is 0 (a nonzero r_i gives t_lo > 0)
  // sqrt rounded up, then to fp16 rounded up: the smallest fp16 value >= sqrt(t_hi)
  p.h0 = __half_as_ushort(__float2half_ru(__fsqrt_ru(t_hi)));
  p.pred = static_cast<uint16_t>(p.h0 - 1);
  const float pv = __half2float(__ushort_as_half(p.pred));
  p.decided = pv * pv < t_lo;  // pred^2 < t_lo <= sum: pred is too small, so h0
  return p;
}
__device__ __forceinline__ Fp16Pick fp16_ru_pick(double t_lo, double t_hi) {
  Fp16Pick p{0, 0, true};
  if (t_hi == 0.0) return p;
  p.h0 = __half_as_ushort(__float2half_ru(__double2float_ru(__dsqrt_ru(t_hi))));
  p.pred = static_cast<uint16_t>(p.h0 - 1);
  const double pv = static_cast<double>(__half2float(__ushort_as_half(p.pred)));
  p.decided = pv * pv < t_lo;
  return p;
}
// The exact decision between pick.h0 and pick.pred: this lane's 4 residual squares plus those of the lanes
// that `reduce` combines (xor offsets), compared with pred^2.  Every lane of the warp calls it.
template <int MASKS>
__device__ __forceinline__ uint16_t exact_pick(const float* xa, const float* xb, const float* x,
                                            Fp16Pick pick, bool want) {
  ExactAcc acc;
  exact_clear(acc);
#pragma unroll
  for (int i = 0; i < 4; ++i)
    exact_add_square(acc, static_cast<double>(xa[i]) * static_cast<double>(xb[i]), static_cast<double>(x[i]));
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    if (!((MASKS >> (o == 16 ? 4 : o == 8 ? 3 : o == 4 ? 2 : o == 2 ? 1 : 0)) & 1)) continue;
#pragma unroll
    for (int j = 0; j < 20; ++j) acc.d[j] += __shfl_xor_sync(0xffffffffu, acc.d[j], o);
  }
  if (!want) return pick.h0;
  const double pv = static_cast<double>(__half2float(__ushort_as_half(pick.pred)));
  exact_add(acc, -(pv * pv));
  return exact_sign(acc) > 0 ? pick.h0 : pick.pred;
}
// fp16 bits of the exact norm of the residuals held by the lanes that the xor offsets in MASKS combine (bit 4:
// offset 16, ..., bit 0: offset 1), rounded up.  Binary32 bracket first; the double-precision bracket and then
// exact arithmetic only where the previous bracket leaves the result open.  Every lane of the warp calls it.
template <int MASKS>
__device__ __forceinline__ uint16_t norm_fp16_ru(const float* xa, const float* xb, const float* x) {
  float lo32, hi32;
  sumsq_bracket32(xa, xb, x, lo32, hi32);
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    if (!((MASKS >> (o == 16 ? 4 : o == 8 ? 3 : o == 4 ? 2 : o == 2 ? 1 : 0)) & 1)) continue;
    hi32 = __fadd_ru(hi32, __shfl_xor_sync(0xffffffffu, hi32, o));  // commutative: the same sum in the lanes
    lo32 = __fadd_rd(lo32, __shfl_xor_sync(0xffffffffu, lo32, o));
  }
  const Fp16Pick p32 = fp16_ru_pick(lo32, hi32);
  if (!__any_sync(0xffffffffu, !p32.decided)) return p32.h0;
  double lo64, hi64;
  sumsq_bracket64(xa, xb, x, lo64, hi64);
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    if (!((MASKS >> (o == 16 ? 4 : o == 8 ? 3 : o == 4 ? 2 : o == 2 ? 1 : 0)) & 1)) continue;
    hi64 = __dadd_ru(hi64, __shfl_xor_sync(0xffffffffu, hi64, o));
    lo64 = __dadd_rd(lo64, __shfl_xor_sync(0xffffffffu, lo64, o));
  }
  const Fp16Pick p64 = p32.decided ? p32 : fp16_ru_pick(lo64, hi64);
  if (!__any_sync(0xffffffffu, !p64.decided)) return p64.h0;
  return exact_pick<MASKS>(xa, xb, x, p64, !p64.decided);
}

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
      if (WANT_RES) { q.xa[i] = xh; q.xb[i] = 1.f; }
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
      codes[i] = static_cast<uint32_t>(code + 128);  // stored offset binary: byte = code + 128
      // x_hat = s (code - xi): code - xi has 18 significant bits (exact in binary32) and s 11, so their
      // product is exact in double precision and one fused multiply-add rounds x_hat - x once
      if (WANT_RES) { q.xa[i] = s; q.xb[i] = static_cast<float>(code) - xi[i]; }
    }
  } else {  // E4M3_SCALED
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t code = 0;
      if (s > 0.0f) code = f32_to_e4m3_bits(__fdiv_rn(x[i], s));
      codes[i] = code;
      if (WANT_RES) { q.xa[i] = s * e4m3_bits_to_f32(static_cast<uint8_t>(code)); q.xb[i] = 1.f; }  // exact: 11 x 4 bits
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
      rc.kc[e] = 0x80u;  // INT8 code 0, offset binary
      qk.xa[e] = hv;
      qk.xb[e] = 1.f;
      if (!isfinite(hv)) flags |= 1;
    }
  }
  if (__any_sync(0xffffffffu, (flags & 1) != 0)) flags |= 1;  // an overflowing bypassed channel flags the row
  if (bad_pair) flags |= 4;
  // every group's value scale is checked (with group scales the lanes hold different ones)
  if (__any_sync(0xffffffffu, fmt_has_scale(VF) && __half2float(__ushort_as_half(rc.vs)) > KVQ_MAX_VALUE_SCALE))
    flags |= 2;
  // Witness: each band norm of r = k_hat - k, exact and rounded up to fp16.  Lane l holds channels
  // 4l..4l+3, all in band l % 16; lanes l and l + 16 share a band (channels 4b..4b+3 and 64+4b..64+4b+3).
  rc.wb = norm_fp16_ru<0x10>(qk.xa, qk.xb, k);
  // Value witness: ||v_hat - v|| and ||v|| over all 128 channels, exact and rounded up to fp16
  rc.vrho = 0;
  rc.vnorm = 0;
  if (want_vw) {  // warp-uniform
    const float ones[4] = {1.f, 1.f, 1.f, 1.f}, zeros[4] = {0.f, 0.f, 0.f, 0.f};
    rc.vrho = norm_fp16_ru<0x1F>(qv.xa, qv.xb, v);
    rc.vnorm = norm_fp16_ru<0x1F>(v, ones, zeros);
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
