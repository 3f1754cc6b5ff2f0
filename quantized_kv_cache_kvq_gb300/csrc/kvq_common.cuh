// kvq_common.cuh -- constants, tile layouts, number conversions, Philox4x32-10 and device
// error reporting shared by the libkvq kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvq.h"

namespace kvq {

constexpr int kHeadDim = KVQ_HEAD_DIM;  // 128
constexpr int kPage = KVQ_PAGE_SIZE;    // 16 tokens per page
constexpr int kBands = KVQ_N_BANDS;     // 16 witness bands
constexpr int kMaxGroup = KVQ_MAX_GROUP;

// Fixed power-of-two factor folded into the fp16 / bf16 softmax weights of the P*V
// tensor-core product: it keeps p * s (s a per-token value scale of ~1e-2) in the
// fp16 normal range.  The accumulator is multiplied by its inverse in the merge.
constexpr float kPvShift = 256.0f;
constexpr float kPvShiftInv = 1.0f / 256.0f;

__host__ __device__ constexpr bool fmt_is_16bit(int f) { return f == KVQ_FMT_BF16; }
// subtractively dithered INT8, with one scale per token or one per token and 32-channel group
__host__ __device__ constexpr bool fmt_is_int8(int f) {
  return f == KVQ_FMT_INT8_DITHER || f == KVQ_FMT_INT8_DITHER_G32;
}
__host__ __device__ constexpr bool fmt_group_scales(int f) { return f == KVQ_FMT_INT8_DITHER_G32; }
__host__ __device__ constexpr bool fmt_has_scale(int f) {
  return f == KVQ_FMT_E4M3_SCALED || fmt_is_int8(f);
}
__host__ __device__ constexpr int tile_bytes_k(int f) { return fmt_is_16bit(f) ? 4096 : 2048; }
__host__ __device__ constexpr int tile_bytes_v(int f) { return fmt_is_16bit(f) ? 4096 : 2048; }
constexpr int kTileBytesW = 512;
constexpr int kTileBytesS = 32;
constexpr int kScaleGroup = 32;                        // channels per scale group (group-scaled INT8)
constexpr int kScaleGroups = kHeadDim / kScaleGroup;   // 4
__host__ __device__ constexpr int tile_bytes_s(int f) { return fmt_group_scales(f) ? kTileBytesS * kScaleGroups : kTileBytesS; }
constexpr int kTileBytesVW = 64;  // value witness: (rho^v, ||v||) per token
constexpr int kMaxOutlierPairs = 8;
// key outlier tile: 16 tokens x 8 fp16 columns (m <= 4) or x 16 (m <= 8), tensor-core A-fragment order
__host__ __device__ constexpr int outlier_tile_bytes(int m) { return m <= 0 ? 0 : (m <= 4 ? 256 : 512); }

// ---------------------------------------------------------------------------------------------
// Tile layouts (byte offsets inside one (page, kv head) tile; see include/kvq.h).
// K tiles hold, per 16-byte word, one token and 8 (16-bit) or 16 (8-bit) channels -- consecutive,
// or with 32-channel scale groups four runs of 4 from two groups -- the A fragments of S^T = K . Q^T.
// V tiles hold, per lane of a 16-channel block, the tokens 2c, 2c+1, 2c+8, 2c+9 of channels g and
// g+8: the A fragments of O^T = V^T . P^T.  Scales hold tokens t and t+8 side by side (the two
// tokens a lane owns in S^T), one pair per 4-byte word and, with group scales, the four groups of
// that pair in one 16-byte word.
__host__ __device__ __forceinline__ int k16_offset(int t, int c) {
  return 16 * ((((t >> 3) * 4 + (c >> 5)) * 32) + (t & 7) * 4 + ((c >> 3) & 3)) + 2 * (c & 7);
}
__host__ __device__ __forceinline__ int k8_offset(int t, int c) {
  return 16 * ((((t >> 3) * 2 + (c >> 6)) * 32) + (t & 7) * 4 + ((c >> 4) & 3)) + (c & 15);
}
// 8-bit keys with 32-channel scale groups: the 16-bit family's k-step order (k-step 2j + s <- channels
// 32j + 8c + 4s + {0..3} of lane c), so that every tensor-core k-step lies inside one scale group
__host__ __device__ __forceinline__ int k8g_offset(int t, int c) {
  return 16 * ((((t >> 3) * 2 + (c >> 6)) * 32) + (t & 7) * 4 + ((c >> 3) & 3)) + 4 * (2 * ((c >> 5) & 1) + ((c >> 2) & 1)) +
         (c & 3);
}
__host__ __device__ __forceinline__ int v16_offset(int t, int c) {
  return 16 * (32 * (c >> 4) + 4 * (c & 7) + ((t & 7) >> 1)) + 4 * (2 * (t >> 3) + ((c >> 3) & 1)) + 2 * (t & 1);
}
__host__ __device__ __forceinline__ int v8_offset(int t, int c) {
  return 16 * (32 * (c >> 5) + 4 * (c & 7) + ((t & 7) >> 1)) + 8 * ((c >> 4) & 1) +
         2 * (2 * (t >> 3) + ((c >> 3) & 1)) + (t & 1);
}
__host__ __device__ __forceinline__ int w_offset(int t, int b) {
  return 16 * (4 * (t & 7) + (b >> 2)) + 8 * (t >> 3) + 2 * (b & 3);
}
__host__ __device__ __forceinline__ int s_offset(int t) { return 2 * (2 * (t & 7) + (t >> 3)); }
// group scales: lane g of the decode reads the four groups of tokens g and g + 8 as one 16-byte word
__host__ __device__ __forceinline__ int gs_offset(int t, int grp) { return 16 * (t & 7) + 4 * grp + 2 * (t >> 3); }
// key outlier column col of token t (m16n8k8 A fragment for m <= 4, m16n8k16 for m <= 8)
__host__ __device__ __forceinline__ int ko_offset(int t, int col, bool wide) {
  return wide ? 16 * (4 * (t & 7) + ((col & 7) >> 1)) + 8 * (col >> 3) + 4 * (t >> 3) + 2 * (col & 1)
              : 8 * (4 * (t & 7) + (col >> 1)) + 4 * (t >> 3) + 2 * (col & 1);
}
// value witness: k = 0 rho^v, k = 1 ||v||; lane g of the decode reads tokens g and g + 8 as one 8-byte word
__host__ __device__ __forceinline__ int vw_offset(int t, int k) { return 8 * (t & 7) + 4 * k + 2 * (t >> 3); }

// Devices a process can drive (per-device caches of attributes and of kernel settings).
constexpr int kMaxDevices = 64;

// ---------------------------------------------------------------------------------------------
// Device error word: the first error code wins.
__device__ __forceinline__ void report(int32_t* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

// ---------------------------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11).  One round:
//   (hi0, lo0) = M0 * x0, (hi1, lo1) = M1 * x2, x' = (hi1 ^ x1 ^ k0, lo1, hi0 ^ x3 ^ k1, lo0),
// then the key is bumped by the Weyl constants W0, W1.
constexpr uint32_t kPhiloxM0 = 0xD2511F53u;
constexpr uint32_t kPhiloxM1 = 0xCD9E8D57u;
constexpr uint32_t kPhiloxW0 = 0x9E3779B9u;
constexpr uint32_t kPhiloxW1 = 0xBB67AE85u;

// 32 x 32 -> 64-bit product, written as plain arithmetic so the compiler can share equal products.
__device__ __forceinline__ void mul_wide(uint32_t a, uint32_t b, uint32_t& hi, uint32_t& lo) {
  const uint64_t p = static_cast<uint64_t>(a) * b;
  lo = static_cast<uint32_t>(p);
  hi = static_cast<uint32_t>(p >> 32);
}

__device__ __forceinline__ uint4 philox4x32_10(uint4 x, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    uint32_t hi0, lo0, hi1, lo1;
    mul_wide(kPhiloxM0, x.x, hi0, lo0);
    mul_wide(kPhiloxM1, x.z, hi1, lo1);
    x = make_uint4(hi1 ^ x.y ^ k0, lo1, hi0 ^ x.w ^ k1, lo0);
    k0 += kPhiloxW0;
    k1 += kPhiloxW1;
  }
  return x;
}

// Philox4x32-10 with the ten round keys precomputed (k0[r] = key0 + r * W0, k1[r] = key1 + r * W1);
// kernel-parameter arrays make every round key a constant operand.
__device__ __forceinline__ uint4 philox4x32_10_rk(uint4 x, const uint32_t (&k0)[10], const uint32_t (&k1)[10]) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    uint32_t hi0, lo0, hi1, lo1;
    mul_wide(kPhiloxM0, x.x, hi0, lo0);
    mul_wide(kPhiloxM1, x.z, hi1, lo1);
    x = make_uint4(hi1 ^ x.y ^ k0[r], lo1, hi0 ^ x.w ^ k1[r], lo0);
  }
  return x;
}

// The decode regenerates, per page and lane, Philox4x32-10 of the counters (slot, layer, kv_head,
// grp) for two slots and its groups of sixteen channels.  In the first three rounds several products depend
// only on (layer, kv_head) or only on the slot; they are computed once (PhiloxHead per page,
// PhiloxSlot per token) and each call finishes with two products in rounds 1-2 and seven full
// rounds.  With (H, L) the high and low words of a product and y, z, w the counters after rounds
// 0, 1, 2:
//   y = (H(M1 kvh) ^ layer ^ k0[0], L(M1 kvh), H(M0 slot) ^ grp ^ k1[0], L(M0 slot))
//   z = (H(M1 y2) ^ y1 ^ k0[1], L(M1 y2), H(M0 y0) ^ y3 ^ k1[1], L(M0 y0))
//   w = (H(M1 z2) ^ z1 ^ k0[2], L(M1 z2), H(M0 z0) ^ z3 ^ k1[2], L(M0 z0))
// where y0, y1, L(M0 y0) depend on (layer, kv_head) only and y3, z2, H(M1 z2), L(M1 z2) on the slot.
struct PhiloxHead {
  uint32_t c1;  // y1 ^ k0[1]
  uint32_t uB;  // H(M0 y0) ^ k1[1]
  uint32_t uD;  // L(M0 y0) ^ k1[2] = z3 ^ k1[2]
};
struct PhiloxSlot {
  uint32_t tA;  // H(M0 slot) ^ k1[0]            (y2 = tA ^ grp)
  uint32_t tC;  // H(M1 z2) ^ k0[2]              (w0 = tC ^ z1)
  uint32_t w1;  // L(M1 z2)
};

__device__ __forceinline__ PhiloxHead philox_head(uint32_t layer, uint32_t kv_head, const uint32_t (&k0)[10],
                                                  const uint32_t (&k1)[10]) {
  uint32_t h1, l1, h0, l0;
  mul_wide(kPhiloxM1, kv_head, h1, l1);
  mul_wide(kPhiloxM0, h1 ^ layer ^ k0[0], h0, l0);
  return PhiloxHead{l1 ^ k0[1], h0 ^ k1[1], l0 ^ k1[2]};
}

__device__ __forceinline__ PhiloxSlot philox_slot(uint32_t slot, const PhiloxHead& h, const uint32_t (&k0)[10],
                                                  const uint32_t (&k1)[10]) {
  uint32_t h0, l0, h1, l1;
  mul_wide(kPhiloxM0, slot, h0, l0);
  mul_wide(kPhiloxM1, l0 ^ h.uB, h1, l1);  // z2 = y3 ^ H(M0 y0) ^ k1[1]
  return PhiloxSlot{h0 ^ k1[0], h1 ^ k0[2], l1};
}

// Philox4x32-10 of (slot, layer, kv_head, grp) from its PhiloxHead / PhiloxSlot parts.
__device__ __forceinline__ uint4 philox_finish(uint32_t grp, const PhiloxSlot& t, const PhiloxHead& h,
                                               const uint32_t (&k0)[10], const uint32_t (&k1)[10]) {
  uint32_t ah, al, bh, bl;
  mul_wide(kPhiloxM1, t.tA ^ grp, ah, al);  // round 1: M1 y2
  mul_wide(kPhiloxM0, ah ^ h.c1, bh, bl);   // round 2: M0 z0
  uint4 x = make_uint4(t.tC ^ al, t.w1, bh ^ h.uD, bl);
#pragma unroll
  for (int r = 3; r < 10; ++r) {
    uint32_t hi0, lo0, hi1, lo1;
    mul_wide(kPhiloxM0, x.x, hi0, lo0);
    mul_wide(kPhiloxM1, x.z, hi1, lo1);
    x = make_uint4(hi1 ^ x.y ^ k0[r], lo1, hi0 ^ x.w ^ k1[r], lo0);
  }
  return x;
}

// Dither contract: the call (slot, layer, kv_head, channel >> 4) serves sixteen channels; output word
// w = (channel >> 2) & 3 carries four of them, one per byte: channel 4i + j in byte j of w; xi = byte * 2^-8 - 1/2
// (a 256-point grid of [-1/2, 1/2), every value exact in fp16).

// Dither of an 8-bit field: exact in binary32.
__device__ __forceinline__ float dither_of_field(uint32_t field) {
  return __fmaf_rn(static_cast<float>(field), 0.00390625f /* 2^-8 */, -0.5f);
}

// The decode's dither operand of a word's channels 4i, 4i + 1 (lo) or 4i + 2, 4i + 3 (hi): the fp16 pair
// -(xi + 9/2) = -(4 + byte 2^-8), whose bit pattern is 0xC400 | byte (low half: the lower channel), made by one
// byte permutation of the word with the constant 0xC4 bytes.  The products add 9/2 sum back through the
// accumulators' initial values (keys) or a lazy per-head correction (values).
constexpr float kDitherOffset = 4.5f;
constexpr uint32_t kDitherHighBytes = 0xC4C4C4C4u;
__device__ __forceinline__ uint32_t neg_offset_dither_lo_f16x2(uint32_t w) { return __byte_perm(w, kDitherHighBytes, 0x4140); }
__device__ __forceinline__ uint32_t neg_offset_dither_hi_f16x2(uint32_t w) { return __byte_perm(w, kDitherHighBytes, 0x4342); }

// Minus the dither of a channel pair as an fp16 pair: -xi = 9/2 - (4 + byte 2^-8), exact.
__device__ __forceinline__ uint32_t neg_dither_f16x2(uint32_t op) {
  const __half2 r = __hadd2(*reinterpret_cast<const __half2*>(&op), __half2(__half(kDitherOffset), __half(kDitherOffset)));
  return *reinterpret_cast<const uint32_t*>(&r);
}

// The four dithers of channels 4*quad .. 4*quad+3 of (slot, layer, kv_head): the bytes of word quad & 3 of the
// call (slot, layer, kv_head, quad >> 2).
__device__ __forceinline__ float4 dither4(uint32_t slot, uint32_t layer, uint32_t kv_head, uint32_t quad,
                                          uint32_t k0, uint32_t k1) {
  const uint4 v = philox4x32_10(make_uint4(slot, layer, kv_head, quad >> 2), k0, k1);
  const uint32_t q = quad & 3u;
  const uint32_t w = q == 0 ? v.x : q == 1 ? v.y : q == 2 ? v.z : v.w;
  return make_float4(dither_of_field(w & 0xFFu), dither_of_field((w >> 8) & 0xFFu),
                     dither_of_field((w >> 16) & 0xFFu), dither_of_field(w >> 24));
}

// ---------------------------------------------------------------------------------------------
// Number conversions (hardware conversion instructions).
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}
__device__ __forceinline__ uint8_t f32_to_e4m3_bits(float x) {
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3));
}
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }
__device__ __forceinline__ float e4m3_bits_to_f32(uint8_t b) {
  const __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(b), __NV_E4M3);
  return __half2float(__half(h));
}

}  // namespace kvq
