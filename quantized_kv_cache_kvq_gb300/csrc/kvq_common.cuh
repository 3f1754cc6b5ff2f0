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
__host__ __device__ constexpr bool fmt_has_scale(int f) {
  return f == KVQ_FMT_E4M3_SCALED || f == KVQ_FMT_INT8_DITHER;
}
__host__ __device__ constexpr int tile_bytes_k(int f) { return fmt_is_16bit(f) ? 4096 : 2048; }
__host__ __device__ constexpr int tile_bytes_v(int f) { return fmt_is_16bit(f) ? 4096 : 2048; }
constexpr int kTileBytesW = 512;
constexpr int kTileBytesS = 32;

// ---------------------------------------------------------------------------------------------
// Tile layouts (byte offsets inside one (page, kv head) tile; see include/kvq.h).
// K tiles hold, per 16-byte word, one token and 8 (16-bit) or 16 (8-bit) consecutive channels:
// the A fragments of S^T = K . Q^T.  V tiles hold, per lane of a 16-channel block, the tokens
// 2c, 2c+1, 2c+8, 2c+9 of channels g and g+8: the A fragments of O^T = V^T . P^T.  Scales hold
// tokens t and t+8 side by side (the two tokens a lane owns in S^T).
__host__ __device__ __forceinline__ int k16_offset(int t, int c) {
  return 16 * ((((t >> 3) * 4 + (c >> 5)) * 32) + (t & 7) * 4 + ((c >> 3) & 3)) + 2 * (c & 7);
}
__host__ __device__ __forceinline__ int k8_offset(int t, int c) {
  return 16 * ((((t >> 3) * 2 + (c >> 6)) * 32) + (t & 7) * 4 + ((c >> 4) & 3)) + (c & 15);
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

__device__ __forceinline__ void mul_wide(uint32_t a, uint32_t b, uint32_t& hi, uint32_t& lo) {
  uint64_t p;
  asm("mul.wide.u32 %0, %1, %2;" : "=l"(p) : "r"(a), "r"(b));
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

// Dither value of a Philox output word: ((w >> 8) + 1/2) * 2^-24 - 1/2, exact in binary32.
__device__ __forceinline__ float dither_from_word(uint32_t w) {
  return __fmaf_rn(static_cast<float>(w >> 8), 5.9604644775390625e-8f /* 2^-24 */,
                   -0.49999997019767761f /* 2^-25 - 1/2 */);
}

// Minus the dither of two words, rounded to an fp16 pair (low half from w0): the decode's tensor-core
// operand; -xi = 1/2 - 2^-25 - (w >> 8) * 2^-24 is exact in binary32 before the fp16 rounding.
__device__ __forceinline__ uint32_t neg_dither_f16x2(uint32_t w0, uint32_t w1) {
  const float a = __fmaf_rn(static_cast<float>(w0 >> 8), -5.9604644775390625e-8f, 0.49999997019767761f);
  const float b = __fmaf_rn(static_cast<float>(w1 >> 8), -5.9604644775390625e-8f, 0.49999997019767761f);
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// The four dithers of channels 4*group .. 4*group+3 of (slot, layer, kv_head).
__device__ __forceinline__ float4 dither4(uint32_t slot, uint32_t layer, uint32_t kv_head, uint32_t group,
                                          uint32_t k0, uint32_t k1) {
  const uint4 w = philox4x32_10(make_uint4(slot, layer, kv_head, group), k0, k1);
  return make_float4(dither_from_word(w.x), dither_from_word(w.y), dither_from_word(w.z), dither_from_word(w.w));
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
