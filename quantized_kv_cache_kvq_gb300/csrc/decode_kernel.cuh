// decode_kernel.cuh -- split-KV paged GQA decode attention with the WitCert meter fused in.
//
// Work decomposition.  A "unit" is one (sequence, kv head); its logical page list is the shared
// prefix pages followed by the sequence's live pages ("Compress the shared cartridge", "One kernel
// spans cartridge and live KV": one logical sequence, one online softmax).  All units' pages are
// laid end to end and cut into equal contiguous ranges, one per warp of a persistent grid (a warp
// range may cross unit boundaries).  Each warp streams its pages through its own ring of shared-
// memory stages filled by bulk asynchronous copies (cp.async.bulk + mbarrier complete_tx), runs
// q.K^T, the witness dot product and P.V on tensor cores (mma.sync m16n8k16; the page's 16 tokens
// are the M rows and the GQA group of up to 8 query heads the N columns), keeps one online-softmax
// state and the meter accumulators per query head, and
// writes a partial (m, l, acc, meter sums) for every (warp, unit) piece it covered.  The merge
// kernel combines the pieces of each unit with log-sum-exp weights -- WitCert Sec. 6.2.2: the
// certificate A is a p~-weighted average, so per-split values merged under the same LSE weights
// give the global A exactly.
//
// Meter (WitCert Sec. 3 Thm. 1, Sec. 4.1 Thm. 2, Sec. 4.2, Sec. 4.3): with x_t the compressed
// logit, c_t = sm_scale * sum_b ||q_b|| w_{t,b}, the kernel accumulates
//     A - 1 = sum_t e^{x_t} (e^{c_t} - 1) / sum_t e^{x_t} = sum_t e^{x_t + c_t} (1 - e^{-c_t}) / sum_t e^{x_t}
// as a running maximum and a scaled sum of e^{x_t + c_t - max} (1 - e^{-c_t}), i.e. in the log
// domain, so c is never clipped and A never overflows; Tier B does the same with
// u_t = sm_scale s_t (||q|| kappa + ||q||_1 2^-9), kappa = sqrt(2 ln(2S/delta_loc) / 12) (the second
// term covers the dither grid's bias), or with one scale per 32-channel group
// u_t = sm_scale (kappa sqrt(sum_g ||q_g||^2 s_{g,t}^2) + 2^-9 sum_g ||q_g||_1 s_{g,t}).
#pragma once

#include "kvq_common.cuh"

namespace kvq {
namespace dec {

// Warps per CTA (one CTA per SM) is a per-layout template parameter (decode_instances.inc); this is
// the largest value any layout uses, which sizes the workspace.
constexpr int kMaxWarps = 16;
constexpr int kQloBytes = 8 * 2 * 32 * 4;  // per-warp low parts of an fp32 query (only when q is fp32)
constexpr int kMaxStages = 16;
constexpr int kMaxBatch = KVQ_MAX_BATCH;  // sequences per call (prefix sums live in shared memory; 16 bits of a
                                         // page descriptor)
static_assert(KVQ_MAX_KV_HEADS <= 128 && KVQ_MAX_BATCH <= 65536, "page descriptor fields");
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;
constexpr int kNoPrefix = -1;
constexpr int kXiScratch = 16 * 128 * 2;  // per-warp fp16 dither tile (INT8 values)
// Extended meter state per lane in shared memory (so it costs no registers in the page loop), 8 floats:
// value side (sum_t e^{x_t - m} rho^v_t for heads 2c and 2c + 1, rescaled with l; max_t ||v_t||; 0) and
// alternative bound shapes (max_t c_t for heads 2c, 2c + 1; sum_t e^{x_t - m} (1 - e^{-c_t}) for both heads).
constexpr int kVStateBytes = 32 * 32;
// Group-scaled INT8 keys: per-warp table of the query's per-group terms, [kind][group][head] floats:
// kind 0 = 9/2 sum_c q_c (the fp16 query the key products use), 1 = (sm_scale kappa)^2 ||q_g||^2,
// 2 = sm_scale 2^-9 ||q_g||_1 (Tier B), for the 4 groups of 32 channels and the 8 heads of a unit.
constexpr int kGqBytes = 3 * 4 * 8 * 4;
constexpr int kExtValue = 1, kExtShapes = 2, kExtContrib = 4;
constexpr int kStatsFloats = 12;  // per (piece, head): m l mc sc | mu su vr vmax | cmax om 0 0
constexpr unsigned kFull = 0xffffffffu;
constexpr unsigned long long kWaitNs = 2000000000ull;  // a copy not landed after 2 s is reported as a timeout

struct Planes {
  const uint8_t* k;
  const uint8_t* v;
  const uint8_t* ks;
  const uint8_t* vs;
  const uint8_t* w;
  const uint8_t* vw;  // value witness plane (head-major) or nullptr
  const uint8_t* ko;  // key outlier plane (head-major) or nullptr
  const int32_t* opairs;  // [Hkv][n_out] bypassed RoPE pairs
  int n_out;          // bypassed pairs per head (0: none)
  int num_pages;
  uint32_t layer;
  uint32_t seed_lo, seed_hi;
  uint32_t rk0[10], rk1[10];  // Philox round keys of the dither stream (host-precomputed)
};

struct Args {
  Planes live, pre;
  int prefix_len, prefix_pages;
  int Hkv, G, Hq, B;
  const void* q;
  int q_bf16;
  const int32_t* bt;
  int max_pages;
  const int32_t* seq_lens;
  float sm_scale;
  int tier_b;
  float ln_delta_loc;
  int wait_append;   // the preceding grid appends each sequence's newest token (programmatic launch)
  float* out;        // [B][Hq][128]
  float* meter_state;  // [B][Hq][4] or nullptr
  int meter_on;
  int value_on;      // value side of the output bound (value witness read, R and Vmax accumulated)
  int shapes_on;     // alternative bound shapes (max radius, 1 - A^-)
  float* page_contrib;  // [B][Hq][contrib_stride] per-page log contributions to A - 1, or nullptr
  int contrib_stride;
  float* ws_stats;   // [slots][G][8]
  float* ws_acc;     // [slots][G][128]
  int w_max;
  int nwa;           // warps per CTA that stream pages (<= NW: fewer when NW warps' stages do not fit shared memory)
  int stages;
  int stage_bytes;
  int32_t* err;
};

// OUTL: the stage has room for a key outlier tile (fixed-channel bypass), 512 bytes reserved.
template <int KF, int VF, bool METER, bool OUTL = false>
struct Layout {
  static constexpr int kBytes = tile_bytes_k(KF);
  static constexpr int vBytes = tile_bytes_v(VF);
  static constexpr int kOff = 0;
  static constexpr int vOff = kBytes;
  static constexpr int wOff = kBytes + vBytes;
  static constexpr int ksOff = wOff + (METER ? kTileBytesW : 0);
  static constexpr int vsOff = ksOff + (fmt_has_scale(KF) ? tile_bytes_s(KF) : 0);
  static constexpr int koOff = vsOff + (fmt_has_scale(VF) ? tile_bytes_s(VF) : 0);
  // the value witness tile follows; it is copied (and the stage sized for it) only with the value
  // side on, so stages without it keep their size
  static constexpr int vwOff = koOff + (OUTL ? outlier_tile_bytes(kMaxOutlierPairs) : 0);
  static constexpr int total = vwOff + (METER ? kTileBytesVW : 0);
  static constexpr int unvalued = vwOff;  // bytes copied when the value side is off
};

// ------------------------------------------------------------------------------------------------
// PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Bounded wait: returns false if the phase did not complete within `limit_ns` of wall time.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned long long limit_ns = kWaitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (;;) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > limit_ns) return false;
  }
}
// L2 policy for the streamed pages of the live cache when a shared prefix is attended too: each live page
// is read once, so it goes first when L2 needs room and the prefix pages, read by every sequence, stay
// resident (measured: +1 % on a 632-token prefix; without a prefix the plain policy is kept).
__device__ __forceinline__ uint64_t stream_policy(bool evict_first) {
  uint64_t p;
  if (evict_first)
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  else
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Page copies are issued by the whole converged warp with the same operands, each operation predicated on the
// one lane that elect.sync picks (no lane-0 branch around them: ~34 fewer warp-instructions per page on the
// INT8 layout than issuing from lane 0 alone).
__device__ __forceinline__ uint32_t elect_one() {
  uint32_t r;
  asm volatile("{\n\t.reg .pred p;\n\t.reg .b32 t;\n\telect.sync t|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}" : "=r"(r));
  return r;
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes, uint32_t leader) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %2, 0;\n\t@p mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n\t}"
               ::"r"(smem_u32(bar)), "r"(bytes), "r"(leader) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar, uint32_t leader) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %1, 0;\n\t@p mbarrier.arrive.shared::cta.b64 _, [%0];\n\t}"
               ::"r"(smem_u32(bar)), "r"(leader) : "memory");
}
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t pol,
                                              uint32_t leader) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %5, 0;\n\t"
               "@p cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;\n\t}"
               ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol), "r"(leader) : "memory");
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint32_t leader) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
               "@p cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n\t}"
               ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)), "r"(leader) : "memory");
}
// A value every lane of the warp holds, returned through a warp reduction: the compiler then knows it is
// uniform and keeps it, and the addresses computed from it, on the uniform datapath.
__device__ __forceinline__ uint32_t uniform_u32(uint32_t v) { return __reduce_or_sync(kFull, v); }
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ uint4 lds128(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }
__device__ __forceinline__ uint2 lds64(const uint8_t* p) { return *reinterpret_cast<const uint2*>(p); }

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed binary32 pairs (lane 0 in the low word).  sm_100-family SMs issue add / sub / mul / fma on two
// binary32 values as one instruction and round each one exactly like the scalar instruction, so the
// pair forms below halve the issue cost of the per-lane arithmetic without changing any result bit.
using f2x = unsigned long long;
__device__ __forceinline__ f2x f2_pack(float lo, float hi) {
  f2x r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ f2x f2_splat(float v) { return f2_pack(v, v); }
__device__ __forceinline__ void f2_unpack(f2x x, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(x));
}
__device__ __forceinline__ f2x f2_fma(f2x a, f2x b, f2x c) {
  f2x d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ f2x f2_mul(f2x a, f2x b) {
  f2x d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f2x f2_add(f2x a, f2x b) {
  f2x d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f2x f2_sub(f2x a, f2x b) {
  f2x d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}

// two e4m3 bytes (low 16 bits of w) -> f16x2 (exact)
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t w) {
  uint32_t r;
  asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(r) : "r"(w));
  return r;
}
// INT8 codes are stored offset binary (byte = code + 128).  Two of them (sel: 0 -> bytes 0,1; 1 -> bytes
// 2,3 of w) -> f16x2 of code + 1152 (exact): 0x6400 | byte is the fp16 value 1024 + byte.  The products
// that take these operands remove the 1152 offset in their accumulator (keys: its initial value; values:
// one product with a constant operand).
constexpr uint32_t kInt8BiasF16x2 = 0xE480E480u;  // fp16 pair (-1152, -1152)
__device__ __forceinline__ uint32_t u8x2_to_f16x2_biased(uint32_t w, int sel) {
  return __byte_perm(w, 0x64646464u, sel ? 0x4342 : 0x4140);
}
// the same without the offset: f16x2 of the two codes themselves (exact)
__device__ __forceinline__ uint32_t u8x2_to_f16x2(uint32_t w, int sel) {
  const uint32_t h = u8x2_to_f16x2_biased(w, sel);
  const __half2 v = __hsub2(*reinterpret_cast<const __half2*>(&h), __half2(__half(1152.f), __half(1152.f)));
  return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ float2 unpack_bf16(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}
__device__ __forceinline__ float2 unpack_f16(uint32_t w) {
  const __half2 h = *reinterpret_cast<const __half2*>(&w);
  return __half22float2(h);
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}

// 1 - e^{-c} for c >= 0: Taylor series to c^8 below 1/2 (truncation < c^9/9! <= 5.4e-9), else via exp2.
__device__ __forceinline__ float one_minus_exp_neg(float c) {
  float p = -2.48015873015873e-05f;           // -1/8!
  p = __fmaf_rn(p, c, 1.98412698412698e-04f);  //  1/7!
  p = __fmaf_rn(p, c, -1.38888888888889e-03f); // -1/6!
  p = __fmaf_rn(p, c, 8.33333333333333e-03f);  //  1/5!
  p = __fmaf_rn(p, c, -4.16666666666667e-02f); // -1/4!
  p = __fmaf_rn(p, c, 1.66666666666667e-01f);  //  1/3!
  p = __fmaf_rn(p, c, -0.5f);                  // -1/2!
  p = __fmaf_rn(p, c, 1.0f);
  const float small = p * c;
  const float large = 1.0f - ex2(-c * kLog2e);
  return c < 0.5f ? small : large;
}

// e^c - 1 for 0 <= c: Taylor series to c^8 below 1/2 (truncation < c^9/9! * e^c), else via exp2.
__device__ __forceinline__ float expm1_pos(float c, bool all_small) {
  float p = 2.48015873015873e-05f;            // 1/8!
  p = __fmaf_rn(p, c, 1.98412698412698e-04f);  // 1/7!
  p = __fmaf_rn(p, c, 1.38888888888889e-03f);  // 1/6!
  p = __fmaf_rn(p, c, 8.33333333333333e-03f);  // 1/5!
  p = __fmaf_rn(p, c, 4.16666666666667e-02f);  // 1/4!
  p = __fmaf_rn(p, c, 1.66666666666667e-01f);  // 1/3!
  p = __fmaf_rn(p, c, 0.5f);                   // 1/2!
  p = __fmaf_rn(p, c, 1.0f);
  const float small = p * c;
  if (all_small) return small;
  const float large = ex2(c * kLog2e) - 1.0f;
  return c < 0.5f ? small : large;
}
// The same for a pair: the Taylor polynomial in packed arithmetic.
__device__ __forceinline__ f2x expm1_pos2(f2x c, bool all_small) {
  f2x p = f2_fma(f2_splat(2.48015873015873e-05f), c, f2_splat(1.98412698412698e-04f));
  p = f2_fma(p, c, f2_splat(1.38888888888889e-03f));
  p = f2_fma(p, c, f2_splat(8.33333333333333e-03f));
  p = f2_fma(p, c, f2_splat(4.16666666666667e-02f));
  p = f2_fma(p, c, f2_splat(1.66666666666667e-01f));
  p = f2_fma(p, c, f2_splat(0.5f));
  p = f2_fma(p, c, f2_splat(1.0f));
  const f2x small = f2_mul(p, c);
  if (all_small) return small;
  float s0, s1, c0, c1;
  f2_unpack(small, s0, s1);
  f2_unpack(c, c0, c1);
  return f2_pack(c0 < 0.5f ? s0 : ex2(c0 * kLog2e) - 1.0f, c1 < 0.5f ? s1 : ex2(c1 * kLog2e) - 1.0f);
}
constexpr float kFastRadius = 60.f;  // e^60 * 2^17 tokens stays far below the fp32 range

// ------------------------------------------------------------------------------------------------
// Fragment orientation.  The page's 16 tokens are the M dimension of every tensor-core product:
//   S^T [16 tok x 8 heads]  = K [16 x 128]      . Q^T [128 x 8]    (8 k-steps)
//   C^T [16 tok x 8 heads]  = W [16 x 16 bands] . QN^T [16 x 8]    (1 k-step; QN = band norms)
//   O^T [128 ch x 8 heads] += V^T [128 x 16 tok] . P^T [16 x 8]    (8 m-tiles of 16 channels)
// Lane (g, c) (g = lane / 4, c = lane % 4) holds S^T / C^T for tokens g and g+8 and query heads
// 2c and 2c+1 (heads >= G are padding), and O^T for channels 16mt+g, 16mt+g+8 of those heads.
// P^T, the B operand of the third product, is S^T's fragment transposed 8x8 by movmatrix.

__device__ __forceinline__ void mma_bf16_4(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                           uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_f16_4(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// m16n8k8 (fp16 inputs, fp32 accumulate): the key-outlier product of up to 8 bypassed channels
__device__ __forceinline__ void mma_f16_k8(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
  asm volatile("mma.sync.aligned.m16n8k8.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, {%0,%1,%2,%3};"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
               : "r"(a0), "r"(a1), "r"(b0));
}
// sum of squares of an fp16 pair, rounded up
__device__ __forceinline__ float sq2_ru(uint32_t h2, float acc) {
  const float2 v = unpack_f16(h2);
  return __fmaf_ru(v.y, v.y, __fmaf_ru(v.x, v.x, acc));
}
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}
__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}

// sum over the 4 lanes of one fragment row (lanes with the same g)
__device__ __forceinline__ float row_sum4(float v) {
  v += __shfl_xor_sync(kFull, v, 1);
  v += __shfl_xor_sync(kFull, v, 2);
  return v;
}
// max over the 8 lanes of one fragment column (lanes with the same c)
__device__ __forceinline__ float col_max8(float v) {
  v = fmaxf(v, __shfl_xor_sync(kFull, v, 4));
  v = fmaxf(v, __shfl_xor_sync(kFull, v, 8));
  v = fmaxf(v, __shfl_xor_sync(kFull, v, 16));
  return v;
}
__device__ __forceinline__ float col_sum8(float v) {
  v += __shfl_xor_sync(kFull, v, 4);
  v += __shfl_xor_sync(kFull, v, 8);
  v += __shfl_xor_sync(kFull, v, 16);
  return v;
}

struct QFrag {
  uint32_t hi[8][2];  // Q^T B fragments (b0, b1) per k-step: head g, channels of the K tile word order
  uint32_t* lo;       // q - hi per (k-step, word, lane) in the warp's shared memory (fp32 queries only)
  uint32_t qn_hi[2], qn_lo[2];  // QN^T B fragment: band norms of head g (normalised by 2^-e)
  bool has_lo;
  float cm_scale;    // c_t = cm_scale * (W . QN)  (natural units)
  float alpha_b[2];  // Tier B: u_t = alpha_b[h] * s_t for heads 2c, 2c+1 (natural units)
  float s_init[2];   // INT8 keys: 9/2 sum_c q_c - 1152 sum_c (q_c + lo_c) (fp16 query parts as the key products
                     // use them: the dither operand's 9/2 and the code operand's 1152 offsets), heads 2c, 2c+1
  float* gq;         // group-scaled INT8 keys: the warp's per-group query table (kGqBytes)
  // fixed-channel outlier bypass: B fragment of the bypassed channels (head g; fp16 hi / lo), and the
  // Tier B terms of heads 2c, 2c+1: u_t += beta_o[h] ||k_hat_{t,O}|| + gamma_o[h]
  uint32_t qo_hi[2], qo_lo[2];
  float beta_o[2], gamma_o[2];
};

struct SoftState {
  float m[2], l[2];    // per head (2c, 2c+1): running max (log2 units), lane-partial sum
  float mc[2], sc[2];  // Tier A accumulator: reference max (log2 units) and scaled sum
  float mu[2], su[2];  // Tier B accumulator
  float o[8][4];       // O^T fragments of the 8 channel blocks
  float pv[2];         // INT8 values: lane-partial sum of the fp16 P' weights per head (for the 9/2 correction)
  // While every radius seen in the unit is <= kFastRadius the meter sums share the softmax's
  // reference max (mc == m): sum p_t (e^{c_t} - 1).  The first larger radius switches the unit to
  // the general form with its own running max (warp-uniform, sticky until the unit ends).
  bool slow_a, slow_b;
};

__device__ __forceinline__ void reset_state(SoftState& s) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    s.m[h] = -INFINITY; s.l[h] = 0.f; s.mc[h] = -INFINITY; s.sc[h] = 0.f; s.mu[h] = -INFINITY; s.su[h] = 0.f;
    s.pv[h] = 0.f;
  }
  s.slow_a = false;
  s.slow_b = false;
#pragma unroll
  for (int i = 0; i < 8; ++i) { s.o[i][0] = 0.f; s.o[i][1] = 0.f; s.o[i][2] = 0.f; s.o[i][3] = 0.f; }
}

// Build the fragments of unit (seq, kv head).  Lane (g, c) supplies the B fragments of query head g:
// K16 family, k-step kb = 2j + s: b0 <- channels 32j + 8c + 4s + {0,1}, b1 <- + {2,3};
// K8 family, kb = 4jj + s: channels 64jj + 16c + 4s + {0,1} / {2,3}.  Band norms: b0 <- bands 4c, 4c+1,
// b1 <- 4c+2, 4c+3 (the witness tile's word order).
// OUTL: the live cache bypasses a fixed set of key channels (INT8 keys): those channels are zeroed in
// the INT8 fragments, gathered into qo_hi / qo_lo (column 2i <- channel pairs[i], 2i + 1 <- pairs[i] + 64;
// B fragment of m16n8k8, or m16n8k16 when m > 4), and Tier B splits ||q|| into the INT8 part (alpha_b)
// and the bypassed part (beta_o, gamma_o: the deterministic bound of the fp16 rounding).
// GS: group-scaled INT8 keys: the 16-bit family's channel order (k-steps 2j, 2j + 1 hold scale group j)
// with fp16 fragments, and the per-group table f.gq.
template <bool K16, bool METER, bool OUTL = false, bool GS = false>
__device__ void load_q(const Args& a, int seq, int kvh, int seq_total, QFrag& f) {
  const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  const bool real = g < a.G;
  const int qh = kvh * a.G + (real ? g : 0);
  const size_t qbase = (static_cast<size_t>(seq) * a.Hq + qh) * kHeadDim;
  // bypassed channels among this lane's channels 64 jj + 16 c + (0..15): bit e of omask[jj]
  uint32_t omask[2] = {0u, 0u};
  const int m_out = OUTL ? a.live.n_out : 0;
  const int32_t* pairs = OUTL ? a.live.opairs + static_cast<size_t>(kvh) * m_out : nullptr;
  if (OUTL) {
    for (int i = 0; i < m_out; ++i) {
      const int j = pairs[i];
      if (j < 0 || j >= kHeadDim / 2) continue;  // reported by the append
      if ((j >> 4) == c) omask[0] |= 1u << (j & 15);        // channel j < 64: jj = 0
      if (((j >> 4) & 3) == c) omask[1] |= 1u << (j & 15);  // channel j + 64: jj = 1, same 16-block
    }
  }
  auto q_at = [&](int ch) -> float {  // one channel of this lane's head
    if (!real) return 0.f;
    return a.q_bf16 ? __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(a.q)[qbase + ch]) << 16)
                    : static_cast<const float*>(a.q)[qbase + ch];
  };
  // 8 consecutive channels of this lane's head (ch % 8 == 0): one 16-byte (bf16) or two (fp32) loads
  auto load8 = [&](int ch, float (&v)[8]) {
    if (!real) {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = 0.f;
      return;
    }
    if (a.q_bf16) {
      const uint4 w = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.q) + qbase + ch);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) { v[2 * i] = __uint_as_float(ws[i] << 16); v[2 * i + 1] = __uint_as_float(ws[i] & 0xFFFF0000u); }
    } else {
      const float4 x0 = *reinterpret_cast<const float4*>(static_cast<const float*>(a.q) + qbase + ch);
      const float4 x1 = *reinterpret_cast<const float4*>(static_cast<const float*>(a.q) + qbase + ch + 4);
      v[0] = x0.x; v[1] = x0.y; v[2] = x0.z; v[3] = x0.w; v[4] = x1.x; v[5] = x1.y; v[6] = x1.z; v[7] = x1.w;
    }
  };
  const bool fp32q = !a.q_bf16;
  bool any_lo = false;
  float qsum = 0.f;  // sum of this lane's fp16 query channels (K8 family)
  float lsum = 0.f;  // sum of their fp16 low parts (fp32 queries)
  auto put = [&](int kb, const float* x) {  // channels x[0..3] of k-step kb: b0 <- x0, x1; b1 <- x2, x3
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float x0 = x[2 * h], x1 = x[2 * h + 1];
      uint32_t lo;
      if (K16) {
        f.hi[kb][h] = pack_bf16(x0, x1);
        const float2 r = unpack_bf16(f.hi[kb][h]);
        lo = pack_bf16(x0 - r.x, x1 - r.y);
      } else {
        // bf16 queries are exact in fp16 down to 2^-14 and within 2^-25 below it: no low part needed
        f.hi[kb][h] = pack_f16(x0, x1);
        const float2 r = unpack_f16(f.hi[kb][h]);
        lo = pack_f16(x0 - r.x, x1 - r.y);
        qsum += r.x + r.y;
        if (fp32q) {
          const float2 rl = unpack_f16(lo);
          lsum += rl.x + rl.y;
        }
      }
      if (fp32q) {
        f.lo[(kb * 2 + h) * 32 + lane] = lo;
        any_lo |= (lo & 0x7FFF7FFFu) != 0u;
      }
    }
  };
  float gsum[4], gsq[4], gl1[4];  // GS: this lane's part of group j's fp16 sum, ||q||^2 and ||q||_1
  if (K16 || GS) {
    // k-step 2j + s <- channels 32j + 8c + 4s + {0..3}
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float v[8];
      load8(32 * j + 8 * c, v);
      if (GS) qsum = lsum = 0.f;
      put(2 * j, v);
      put(2 * j + 1, v + 4);
      if (GS) {
        gsum[j] = kDitherOffset * qsum - 1152.f * (qsum + lsum);
        float sq = 0.f, l1 = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) { sq = __fmaf_rn(v[e], v[e], sq); l1 += fabsf(v[e]); }
        gsq[j] = sq;
        gl1[j] = l1;
      }
    }
  } else {
    // k-step 4jj + s <- channels 64jj + 16c + 4s + {0..3}
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      float v0[8], v1[8];
      load8(64 * jj + 16 * c, v0);
      load8(64 * jj + 16 * c + 8, v1);
      if (OUTL) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          if ((omask[jj] >> e) & 1u) v0[e] = 0.f;
          if ((omask[jj] >> (8 + e)) & 1u) v1[e] = 0.f;
        }
      }
      put(4 * jj, v0);
      put(4 * jj + 1, v0 + 4);
      put(4 * jj + 2, v1);
      put(4 * jj + 3, v1 + 4);
    }
  }
  f.has_lo = __any_sync(kFull, any_lo);
  {
    // the key products of dithered INT8 pages multiply -(xi + 9/2) by the fp16 query and the codes, as
    // code + 1152, by its fp16 high and low parts, so their accumulator starts at 9/2 sum_c q_c -
    // 1152 sum_c (q_c + lo_c) (heads 2c and 2c + 1; the sums live on the lanes of row g)
    const float qs_g = row_sum4(kDitherOffset * qsum - 1152.f * (qsum + lsum));
    f.s_init[0] = __shfl_sync(kFull, qs_g, 8 * c);
    f.s_init[1] = __shfl_sync(kFull, qs_g, 8 * c + 4);
  }
  __syncwarp();
  if (METER) {
    // band b = 4c + i holds channels 16c + 4i + {0..3} and 64 + 16c + 4i + {0..3}
    float u0[8], u1[8], w0[8], w1[8];
    load8(16 * c, u0);
    load8(16 * c + 8, u1);
    load8(64 + 16 * c, w0);
    load8(64 + 16 * c + 8, w1);
    float qn[4];
    float sq_all = 0.f, sq_int8 = 0.f;  // ||q||^2 and, with the bypass, its INT8-channel part
    float l1 = 0.f;                      // ||q||_1 over the INT8 channels (Tier B's dither-grid term)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float* u = (i < 2) ? (u0 + 4 * i) : (u1 + 4 * (i - 2));
      const float* w = (i < 2) ? (w0 + 4 * i) : (w1 + 4 * (i - 2));
      float s = 0.f, s8 = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        s = __fmaf_rn(u[e], u[e], s);
        s = __fmaf_rn(w[e], w[e], s);
        if (OUTL) {
          const int bit = 4 * i + e;  // channel 16c + bit (u) and 64 + 16c + bit (w)
          if (!((omask[0] >> bit) & 1u)) { s8 = __fmaf_rn(u[e], u[e], s8); l1 += fabsf(u[e]); }
          if (!((omask[1] >> bit) & 1u)) { s8 = __fmaf_rn(w[e], w[e], s8); l1 += fabsf(w[e]); }
        } else {
          l1 += fabsf(u[e]) + fabsf(w[e]);
        }
      }
      qn[i] = sqrtf(s);
      sq_all += s;
      sq_int8 += s8;
    }
    // one power-of-two normalisation for the unit (max over heads and bands < 2), hi/lo fp16 split
    float mx = fmaxf(fmaxf(qn[0], qn[1]), fmaxf(qn[2], qn[3]));
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
    int e2 = 0;
    if (mx > 0.f) frexpf(mx, &e2);
    const float inv = ldexpf(1.f, -e2);
    float hv[4], lv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float v = qn[i] * inv;
      hv[i] = __half2float(__float2half_rn(v));
      lv[i] = v - hv[i];
    }
    f.qn_hi[0] = pack_f16(hv[0], hv[1]);
    f.qn_hi[1] = pack_f16(hv[2], hv[3]);
    f.qn_lo[0] = pack_f16(lv[0], lv[1]);
    f.qn_lo[1] = pack_f16(lv[2], lv[3]);
    f.cm_scale = a.sm_scale * ldexpf(1.f, e2);
    // ||q_g|| lives on the lanes of row g; the C fragment needs heads 2c and 2c+1
    // the dither term uses the query on the INT8 channels only (the bypassed ones leave the variance)
    // u_t = sm_scale s_t (||q|| kappa + ||q||_1 2^-9): the sub-Gaussian radius of WitCert Sec. 4.2 plus
    // the largest mean of the dithered rounding error on the 256-point dither grid (2^-9 LSB)
    const float qnorm_g = sqrtf(row_sum4(OUTL ? sq_int8 : sq_all));
    const float l1_g = row_sum4(l1);
    const float kappa = sqrtf(2.f * (logf(2.f * static_cast<float>(seq_total)) - a.ln_delta_loc) / 12.f);
    const float b_g = __fmaf_rn(qnorm_g, kappa, l1_g * 0.001953125f /* 2^-9 */);
    f.alpha_b[0] = a.sm_scale * __shfl_sync(kFull, b_g, 8 * c);
    f.alpha_b[1] = a.sm_scale * __shfl_sync(kFull, b_g, 8 * c + 4);
  }
  if (OUTL) {
    // bypassed channels: B fragment columns 2c, 2c + 1 (pair c) and, when m > 4, 2c + 8, 2c + 9 (pair c + 4)
    float x[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int k2 = 0; k2 < 2; ++k2) {
      const int i = c + 4 * k2;
      if (i < m_out) {
        const int j = pairs[i];
        if (j >= 0 && j < kHeadDim / 2) { x[2 * k2] = q_at(j); x[2 * k2 + 1] = q_at(j + kHeadDim / 2); }
      }
    }
    f.qo_hi[0] = pack_f16(x[0], x[1]);
    f.qo_hi[1] = pack_f16(x[2], x[3]);
    const float2 r0 = unpack_f16(f.qo_hi[0]), r1 = unpack_f16(f.qo_hi[1]);
    f.qo_lo[0] = pack_f16(x[0] - r0.x, x[1] - r0.y);
    f.qo_lo[1] = pack_f16(x[2] - r1.x, x[3] - r1.y);
    // ||q_O|| of head g (rounded up), for the deterministic fp16 term of Tier B:
    // |q_O . r_O| <= ||q_O|| (2^-11 ||k_hat_O|| + sqrt(2m) 2^-25)
    float so = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) so = __fmaf_ru(x[e], x[e], so);
    so = __fadd_ru(so, __shfl_xor_sync(kFull, so, 1));
    so = __fadd_ru(so, __shfl_xor_sync(kFull, so, 2));
    const float qo_g = __fsqrt_ru(so);
    const float o0 = __shfl_sync(kFull, qo_g, 8 * c), o1 = __shfl_sync(kFull, qo_g, 8 * c + 4);
    const float rt = sqrtf(2.f * static_cast<float>(m_out)) * 1.0000001f;
    f.beta_o[0] = a.sm_scale * o0 * 0x1p-11f;
    f.beta_o[1] = a.sm_scale * o1 * 0x1p-11f;
    f.gamma_o[0] = a.sm_scale * o0 * rt * 0x1p-25f;
    f.gamma_o[1] = a.sm_scale * o1 * rt * 0x1p-25f;
  }
  if (GS) {
    // the per-group table, one entry per (kind, group, head g) from the lanes of row g
    const float kap = METER ? sqrtf(2.f * (logf(2.f * static_cast<float>(seq_total)) - a.ln_delta_loc) / 12.f) : 0.f;
    const float ka = a.sm_scale * kap;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float s1 = row_sum4(gsum[j]), s2 = row_sum4(gsq[j]), s3 = row_sum4(gl1[j]);
      if (c == 0) {
        f.gq[(0 * 4 + j) * 8 + g] = s1;  // 9/2 sum q - 1152 sum (q + lo) of the group (see gsum)
        f.gq[(1 * 4 + j) * 8 + g] = ka * ka * s2;
        f.gq[(2 * 4 + j) * 8 + g] = a.sm_scale * 0x1p-9f * s3;
      }
    }
    __syncwarp();
  }
}

// One page of a meter sum.  r[v]: radius (c_t or u_t, natural units) of token g + 8(v >> 1) for head
// 2c + (v & 1); x[v]: its logit (log2 units, -inf for padding); p[v] = 2^{x - mnew}.
// Fast form (mc == m): sum += sum_v p (e^r - 1), rescaled with the softmax's alpha.
// General form: own running max of x + r log2e, terms 2^{x + r log2e - max} (1 - e^{-r}).
// Returns true for the fast form, whose per-head terms of this lane's two tokens (p (e^r - 1) summed
// over tokens g and g + 8, under the softmax max) go to `terms` when it is given.
__device__ __forceinline__ bool accumulate_meter(const float (&r)[4], const float (&x)[4], const float (&p)[4],
                                                 const float (&alpha)[2], const float (&mnew)[2], float (&mc)[2],
                                                 float (&sc)[2], bool& slow, float* terms = nullptr) {
  const float rmax = __uint_as_float(__reduce_max_sync(
      kFull, __float_as_uint(fmaxf(fmaxf(r[0], r[1]), fmaxf(r[2], r[3])))));  // r >= 0: bit order = value order
  slow = slow || !(rmax <= kFastRadius);
  if (!slow) {
    // both heads at once: sc = sc alpha + (p_g (e^{r_g} - 1) + p_{g+8} (e^{r_{g+8}} - 1))
    const bool small = rmax < 0.5f;
    const f2x e0 = expm1_pos2(f2_pack(r[0], r[1]), small), e1 = expm1_pos2(f2_pack(r[2], r[3]), small);
    const f2x t = f2_fma(f2_pack(p[2], p[3]), e1, f2_mul(f2_pack(p[0], p[1]), e0));
    f2_unpack(f2_fma(f2_pack(sc[0], sc[1]), f2_pack(alpha[0], alpha[1]), t), sc[0], sc[1]);
    mc[0] = mnew[0];
    mc[1] = mnew[1];
    if (terms) f2_unpack(t, terms[0], terms[1]);
    return true;
  }
  float z[4];
#pragma unroll
  for (int v = 0; v < 4; ++v) z[v] = __fmaf_rn(r[v], kLog2e, x[v]);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const float mz = col_max8(fmaxf(z[h], z[2 + h]));
    const float mc_new = fmaxf(mc[h], mz);
    if (mc_new != -INFINITY) {
      const float t0 = ex2(z[h] - mc_new) * one_minus_exp_neg(r[h]);
      const float t1 = ex2(z[2 + h] - mc_new) * one_minus_exp_neg(r[2 + h]);
      sc[h] = sc[h] * ex2(mc[h] - mc_new) + (t0 + t1);
      mc[h] = mc_new;
    }
  }
  return false;
}

// ------------------------------------------------------------------------------------------------
// One page of 16 tokens for one kv head.  `st` is the stage holding the page's tiles.  LO = false: the
// query has no low part (f.has_lo is false), so the page body has no per-k-step test of it.
// Tokens past the end of the sequence (a partial last page) have had their K, V, witness and scale
// bytes zeroed in the stage; `xb0` / `xb1` are 0 for valid tokens g / g + 8 and -inf otherwise, added
// to the logits, so no per-element masking is needed here.
template <int KF, int VF, bool METER, bool OUTL = false, bool LO = true, bool VOTE = true>
__device__ __forceinline__ void process_page(const uint8_t* st, uint8_t* xi_tile, float xb0, float xb1, uint32_t phys,
                                             const Planes& pl, int kvh, const QFrag& f, SoftState& s,
                                             float qk_scale, bool tier_b, float* vstate, int ext,
                                             float* cdst = nullptr, int cstride = 0, int G = 0) {
  using L = Layout<KF, VF, METER, OUTL>;
  const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  constexpr bool K16 = fmt_is_16bit(KF);
  constexpr bool KDITHER = fmt_is_int8(KF);
  constexpr bool VDITHER = fmt_is_int8(VF);
  constexpr bool GS = fmt_group_scales(KF);  // keys and values both group-scaled INT8
  static_assert(fmt_group_scales(KF) == fmt_group_scales(VF), "group-scaled keys go with group-scaled values");

  // ---------------- S^T = K . Q^T: rows are tokens g (a0, a2) and g + 8 (a1, a3)
  float S[4] = {0.f, 0.f, 0.f, 0.f};
  if (K16) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 k0 = lds128(st + L::kOff + (j * 32 + lane) * 16);
      const uint4 k1 = lds128(st + L::kOff + ((4 + j) * 32 + lane) * 16);
      mma_bf16_4(S, k0.x, k1.x, k0.y, k1.y, f.hi[2 * j][0], f.hi[2 * j][1]);
      mma_bf16_4(S, k0.z, k1.z, k0.w, k1.w, f.hi[2 * j + 1][0], f.hi[2 * j + 1][1]);
      if (LO && f.has_lo) {
        const uint32_t* lo = f.lo + lane;
        mma_bf16_4(S, k0.x, k1.x, k0.y, k1.y, lo[(4 * j + 0) * 32], lo[(4 * j + 1) * 32]);
        mma_bf16_4(S, k0.z, k1.z, k0.w, k1.w, lo[(4 * j + 2) * 32], lo[(4 * j + 3) * 32]);
      }
    }
  } else if (GS) {
    // group-scaled INT8 keys: k-step kb = 4jj + sidx holds channels 32gr + 8c + 4(sidx & 1) + {0..3} of scale
    // group gr = 2jj + (sidx >> 1); group gr's product T (started at 9/2 sum of its q, undoing the -(xi + 9/2)
    // of the dither products) is multiplied by the token scales of the group into S
    // lanes c and c ^ 1 use the two halves of the same calls: the even lane makes token g's call, the odd lane
    // token g + 8's, and each passes its partner the half it needs
    const PhiloxHead ph = philox_head(pl.layer, static_cast<uint32_t>(kvh), pl.rk0, pl.rk1);
    const PhiloxSlot pt = philox_slot(phys * kPage + g + 8 * (c & 1), ph, pl.rk0, pl.rk1);
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      const uint4 k0 = lds128(st + L::kOff + (jj * 32 + lane) * 16);
      const uint4 k1 = lds128(st + L::kOff + ((2 + jj) * 32 + lane) * 16);
      const uint32_t w0[4] = {k0.x, k0.y, k0.z, k0.w};
      const uint32_t w1[4] = {k1.x, k1.y, k1.z, k1.w};
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int gr = 2 * jj + half;
        const float2 ti = *reinterpret_cast<const float2*>(f.gq + gr * 8 + 2 * c);  // undoes the 9/2, 1152 offsets
        float T[4] = {ti.x, ti.y, ti.x, ti.y};
        // one Philox call per token serves this lane's 8 channels 32gr + 8c + {0..7}: words 2(c & 1) and
        // 2(c & 1) + 1 of the call (slot, layer, kv head, (32gr + 8c) >> 4)
        const uint32_t grp = 2 * gr + (c >> 1);
        const uint4 d = philox_finish(grp, pt, ph, pl.rk0, pl.rk1);  // token g (even lanes) or g + 8 (odd lanes)
        const uint32_t keep0 = (c & 1) ? d.z : d.x, keep1 = (c & 1) ? d.w : d.y;  // this lane's half
        const uint32_t got0 = __shfl_xor_sync(kFull, (c & 1) ? d.x : d.z, 1);    // the partner's call, this half
        const uint32_t got1 = __shfl_xor_sync(kFull, (c & 1) ? d.y : d.w, 1);
        const uint32_t u0 = (c & 1) ? got0 : keep0, v0 = (c & 1) ? got1 : keep1;  // token g: channels +0..3, +4..7
        const uint32_t u1 = (c & 1) ? keep0 : got0, v1 = (c & 1) ? keep1 : got1;  // token g + 8
        const uint32_t n0[4] = {neg_offset_dither_lo_f16x2(u0), neg_offset_dither_hi_f16x2(u0),
                                neg_offset_dither_lo_f16x2(v0), neg_offset_dither_hi_f16x2(v0)};
        const uint32_t n1[4] = {neg_offset_dither_lo_f16x2(u1), neg_offset_dither_hi_f16x2(u1),
                                neg_offset_dither_lo_f16x2(v1), neg_offset_dither_hi_f16x2(v1)};
        if (VDITHER) {
          const int off = ((4 * gr + c) ^ g) << 4;
          *reinterpret_cast<uint4*>(xi_tile + g * 256 + off) =
              make_uint4(neg_dither_f16x2(n0[0]), neg_dither_f16x2(n0[1]), neg_dither_f16x2(n0[2]), neg_dither_f16x2(n0[3]));
          *reinterpret_cast<uint4*>(xi_tile + (g + 8) * 256 + off) =
              make_uint4(neg_dither_f16x2(n1[0]), neg_dither_f16x2(n1[1]), neg_dither_f16x2(n1[2]), neg_dither_f16x2(n1[3]));
        }
#pragma unroll
        for (int s2 = 0; s2 < 2; ++s2) {
          const int sidx = 2 * half + s2, kb = 4 * jj + sidx;
          const uint32_t a0 = u8x2_to_f16x2_biased(w0[sidx], 0), a2 = u8x2_to_f16x2_biased(w0[sidx], 1);
          const uint32_t a1 = u8x2_to_f16x2_biased(w1[sidx], 0), a3 = u8x2_to_f16x2_biased(w1[sidx], 1);
          mma_f16_4(T, a0, a1, a2, a3, f.hi[kb][0], f.hi[kb][1]);
          if (LO && f.has_lo) mma_f16_4(T, a0, a1, a2, a3, f.lo[(2 * kb) * 32 + lane], f.lo[(2 * kb + 1) * 32 + lane]);
          mma_f16_4(T, n0[2 * s2], n1[2 * s2], n0[2 * s2 + 1], n1[2 * s2 + 1], f.hi[kb][0], f.hi[kb][1]);
        }
        // scales of group gr for tokens g (low half) and g + 8 (high half)
        const float2 sg = unpack_f16(*reinterpret_cast<const uint32_t*>(st + L::ksOff + 16 * g + 4 * gr));
        f2_unpack(f2_fma(f2_pack(T[0], T[1]), f2_splat(sg.x), f2_pack(S[0], S[1])), S[0], S[1]);
        f2_unpack(f2_fma(f2_pack(T[2], T[3]), f2_splat(sg.y), f2_pack(S[2], S[3])), S[2], S[3]);
      }
    }
  } else {
    float S2[4] = {0.f, 0.f, 0.f, 0.f};  // the dither products: a second accumulator chain, added at the end
    PhiloxHead ph{};
    PhiloxSlot pt0{}, pt1{};
    if (KDITHER) {
      ph = philox_head(pl.layer, static_cast<uint32_t>(kvh), pl.rk0, pl.rk1);
      pt0 = philox_slot(phys * kPage + g, ph, pl.rk0, pl.rk1);
      pt1 = philox_slot(phys * kPage + g + 8, ph, pl.rk0, pl.rk1);
      // the products below use code + 1152 and -(xi + 9/2); the accumulator's initial value undoes both offsets
      S[0] = S[2] = f.s_init[0];
      S[1] = S[3] = f.s_init[1];
    }
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      const uint4 k0 = lds128(st + L::kOff + (jj * 32 + lane) * 16);
      const uint4 k1 = lds128(st + L::kOff + ((2 + jj) * 32 + lane) * 16);
      const uint32_t w0[4] = {k0.x, k0.y, k0.z, k0.w};
      const uint32_t w1[4] = {k1.x, k1.y, k1.z, k1.w};
      // one Philox call per token serves this lane's 16 channels 64jj + 16c + {0..15} (the call (slot, layer, kv
      // head, 4jj + c)); word sidx holds the k-step's channels 64jj + 16c + 4 sidx + {0..3}
      uint4 d0{}, d1{};
      if (KDITHER) {
        d0 = philox_finish(4 * jj + c, pt0, ph, pl.rk0, pl.rk1);
        d1 = philox_finish(4 * jj + c, pt1, ph, pl.rk0, pl.rk1);
      }
#pragma unroll
      for (int sidx = 0; sidx < 4; ++sidx) {
        uint32_t a0, a1, a2, a3;
        if (KDITHER) {
          a0 = u8x2_to_f16x2_biased(w0[sidx], 0); a2 = u8x2_to_f16x2_biased(w0[sidx], 1);
          a1 = u8x2_to_f16x2_biased(w1[sidx], 0); a3 = u8x2_to_f16x2_biased(w1[sidx], 1);
        } else {
          a0 = e4m3x2_to_f16x2(w0[sidx] & 0xFFFFu); a2 = e4m3x2_to_f16x2(w0[sidx] >> 16);
          a1 = e4m3x2_to_f16x2(w1[sidx] & 0xFFFFu); a3 = e4m3x2_to_f16x2(w1[sidx] >> 16);
        }
        const int kb = 4 * jj + sidx;
        mma_f16_4(S, a0, a1, a2, a3, f.hi[kb][0], f.hi[kb][1]);
        if (LO && f.has_lo) mma_f16_4(S, a0, a1, a2, a3, f.lo[(2 * kb) * 32 + lane], f.lo[(2 * kb + 1) * 32 + lane]);
        if (KDITHER) {
          // the key operand -(xi + 9/2) of channel pairs (+0, +1) and (+2, +3) of tokens g and g + 8
          const uint32_t w0s = sidx == 0 ? d0.x : sidx == 1 ? d0.y : sidx == 2 ? d0.z : d0.w;
          const uint32_t w1s = sidx == 0 ? d1.x : sidx == 1 ? d1.y : sidx == 2 ? d1.z : d1.w;
          const uint32_t e0 = neg_offset_dither_lo_f16x2(w0s), e2 = neg_offset_dither_hi_f16x2(w0s);
          const uint32_t e1 = neg_offset_dither_lo_f16x2(w1s), e3 = neg_offset_dither_hi_f16x2(w1s);
          if (VDITHER && (sidx & 1)) {
            // the value side's dither operand -(xi + 9/2) of channels 64jj + 16c + 8(sidx >> 1) + {0..7}: token-major
            // fp16 tile, 16-byte chunks xor-swizzled by row
            const uint32_t p0 = sidx == 1 ? d0.x : d0.z, p1 = sidx == 1 ? d1.x : d1.z;
            const int off = ((8 * jj + 2 * c + (sidx >> 1)) ^ g) << 4;
            *reinterpret_cast<uint4*>(xi_tile + g * 256 + off) =
                make_uint4(neg_offset_dither_lo_f16x2(p0), neg_offset_dither_hi_f16x2(p0), e0, e2);
            *reinterpret_cast<uint4*>(xi_tile + (g + 8) * 256 + off) =
                make_uint4(neg_offset_dither_lo_f16x2(p1), neg_offset_dither_hi_f16x2(p1), e1, e3);
          }
          mma_f16_4(S2, e0, e1, e2, e3, f.hi[kb][0], f.hi[kb][1]);
        }
      }
    }
    if (KDITHER) {
#pragma unroll
      for (int i = 0; i < 4; ++i) S[i] += S2[i];
    }
  }

  // ---------------- bypassed key channels (fixed-channel outlier bypass, WitCert Sec. 6.2.5): fp16 values
  // times the query's bypassed channels; kon = ||k_hat_O|| of tokens g and g + 8 (Tier B, rounded up)
  float So[4] = {0.f, 0.f, 0.f, 0.f};
  float kon[2] = {0.f, 0.f};
  if (OUTL) {
    float s0 = 0.f, s1 = 0.f;
    if (pl.n_out > 4) {
      const uint4 ko = lds128(st + L::koOff + lane * 16);
      mma_f16_4(So, ko.x, ko.y, ko.z, ko.w, f.qo_hi[0], f.qo_hi[1]);
      if (LO && f.has_lo) mma_f16_4(So, ko.x, ko.y, ko.z, ko.w, f.qo_lo[0], f.qo_lo[1]);
      s0 = sq2_ru(ko.z, sq2_ru(ko.x, 0.f));
      s1 = sq2_ru(ko.w, sq2_ru(ko.y, 0.f));
    } else {
      const uint2 ko = lds64(st + L::koOff + lane * 8);
      mma_f16_k8(So, ko.x, ko.y, f.qo_hi[0]);
      if (LO && f.has_lo) mma_f16_k8(So, ko.x, ko.y, f.qo_lo[0]);
      s0 = sq2_ru(ko.x, 0.f);
      s1 = sq2_ru(ko.y, 0.f);
    }
    if (METER && tier_b) {
      s0 = __fadd_ru(s0, __shfl_xor_sync(kFull, s0, 1));
      s0 = __fadd_ru(s0, __shfl_xor_sync(kFull, s0, 2));
      s1 = __fadd_ru(s1, __shfl_xor_sync(kFull, s1, 1));
      s1 = __fadd_ru(s1, __shfl_xor_sync(kFull, s1, 2));
      kon[0] = __fsqrt_ru(s0);
      kon[1] = __fsqrt_ru(s1);
    }
  }

  // ---------------- per-token scales of tokens g and g + 8
  float sk[2] = {1.f, 1.f}, sv[2] = {1.f, 1.f};  // (group scales are applied in the products instead)
  if (fmt_has_scale(KF) && !GS) {
    const float2 a = unpack_f16(*reinterpret_cast<const uint32_t*>(st + L::ksOff + 4 * g));
    sk[0] = a.x; sk[1] = a.y;
  }
  if (fmt_has_scale(VF) && !GS) {
    const float2 a = unpack_f16(*reinterpret_cast<const uint32_t*>(st + L::vsOff + 4 * g));
    sv[0] = a.x; sv[1] = a.y;
  }

  // ---------------- online softmax (log2 domain).  v = 2r + h: token g + 8r, head 2c + h
  // pair r holds token g + 8r for heads 2c, 2c + 1
  f2x xp[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const float sc = fmt_has_scale(KF) && !GS ? qk_scale * sk[r] : qk_scale;
    f2x base = f2_splat(r ? xb1 : xb0);
    if (OUTL) base = f2_fma(f2_pack(So[2 * r], So[2 * r + 1]), f2_splat(qk_scale), base);
    xp[r] = f2_fma(f2_pack(S[2 * r], S[2 * r + 1]), f2_splat(sc), base);
  }
  float x[4];
  f2_unpack(xp[0], x[0], x[1]);
  f2_unpack(xp[1], x[2], x[3]);
  // VOTE: the running max moves only when a logit of the page exceeds it, which one vote tells; otherwise the
  // column maxima below would give mnew = m and alpha = 1 exactly, so they are skipped (same results).  Measured per
  // launch: INT8 -2.5 %, group-scaled INT8 -3.2 %, cartridge -0.4 %, ragged +0.3 %; the 16-warp layouts at their
  // 128-register cap +0.3 % (FP8 raw) and the INT8 outlier-bypass body +2.0 %, so those keep the unconditional form.
  float alpha[2] = {1.f, 1.f}, mnew[2] = {s.m[0], s.m[1]};
  const bool grow =
      !VOTE || __any_sync(kFull, (x[0] > s.m[0]) | (x[2] > s.m[0]) | (x[1] > s.m[1]) | (x[3] > s.m[1]));
  if (grow) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float mx = col_max8(fmaxf(x[h], x[2 + h]));
      mnew[h] = fmaxf(s.m[h], mx);
      alpha[h] = ex2(s.m[h] - mnew[h]);  // 0 on the first page (m = -inf); every page has a valid token
    }
  }
  float p[4];
  {
    const f2x mn = f2_pack(mnew[0], mnew[1]);
    float d[4];
    f2_unpack(f2_sub(xp[0], mn), d[0], d[1]);
    f2_unpack(f2_sub(xp[1], mn), d[2], d[3]);
#pragma unroll
    for (int v = 0; v < 4; ++v) p[v] = ex2(d[v]);  // 0 for -inf logits
    f2_unpack(f2_fma(f2_pack(s.l[0], s.l[1]), f2_pack(alpha[0], alpha[1]),
                     f2_add(f2_pack(p[0], p[1]), f2_pack(p[2], p[3]))), s.l[0], s.l[1]);
  }
  if (METER && vstate && (ext & kExtValue)) {
    // value side: rho^v and ||v|| of tokens g and g + 8 (WitCert Sec. 3 output bound)
    const uint2 vw = lds64(st + L::vwOff + 8 * g);
    const float2 rho = unpack_f16(vw.x), vn = unpack_f16(vw.y);
    float4 v4 = *reinterpret_cast<const float4*>(vstate + 8 * lane);
    v4.x = __fmaf_rn(p[2], rho.y, __fmaf_rn(p[0], rho.x, v4.x * alpha[0]));
    v4.y = __fmaf_rn(p[3], rho.y, __fmaf_rn(p[1], rho.x, v4.y * alpha[1]));
    v4.z = fmaxf(v4.z, fmaxf(vn.x, vn.y));
    *reinterpret_cast<float4*>(vstate + 8 * lane) = v4;
  }
  if (grow && __any_sync(kFull, (alpha[0] != 1.f) | (alpha[1] != 1.f))) {
    const f2x al = f2_pack(alpha[0], alpha[1]);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      f2_unpack(f2_mul(f2_pack(s.o[i][0], s.o[i][1]), al), s.o[i][0], s.o[i][1]);
      f2_unpack(f2_mul(f2_pack(s.o[i][2], s.o[i][3]), al), s.o[i][2], s.o[i][3]);
    }
  }

  // ---------------- meter (Tier A witness bound; Tier B dither certificate)
  if (METER) {
    float C[4] = {0.f, 0.f, 0.f, 0.f};
    const uint4 wb = lds128(st + L::wOff + lane * 16);
    mma_f16_4(C, wb.x, wb.z, wb.y, wb.w, f.qn_hi[0], f.qn_hi[1]);
    mma_f16_4(C, wb.x, wb.z, wb.y, wb.w, f.qn_lo[0], f.qn_lo[1]);
    float cv[4];
    f2_unpack(f2_mul(f2_pack(C[0], C[1]), f2_splat(f.cm_scale)), cv[0], cv[1]);
    f2_unpack(f2_mul(f2_pack(C[2], C[3]), f2_splat(f.cm_scale)), cv[2], cv[3]);
#pragma unroll
    for (int v = 0; v < 4; ++v) cv[v] = fmaxf(cv[v], 0.f);
    float pt[2];
    const bool fast_a = accumulate_meter(cv, x, p, alpha, mnew, s.mc, s.sc, s.slow_a, cdst ? pt : nullptr);
    if (vstate && (ext & kExtShapes)) {
      // alternative shapes (WitCert Sec. 4.3 Prop. 1; det-tanh): max_t c_t and sum_t e^{x_t - m} (1 - e^{-c_t})
      float4 w4 = *reinterpret_cast<const float4*>(vstate + 8 * lane + 4);
      w4.x = fmaxf(w4.x, fmaxf(cv[0], cv[2]));
      w4.y = fmaxf(w4.y, fmaxf(cv[1], cv[3]));
      w4.z = __fmaf_rn(p[2], one_minus_exp_neg(cv[2]), __fmaf_rn(p[0], one_minus_exp_neg(cv[0]), w4.z * alpha[0]));
      w4.w = __fmaf_rn(p[3], one_minus_exp_neg(cv[3]), __fmaf_rn(p[1], one_minus_exp_neg(cv[1]), w4.w * alpha[1]));
      *reinterpret_cast<float4*>(vstate + 8 * lane + 4) = w4;
    }
    if (vstate && cdst && fast_a) {
      // gate support (WitCert Sec. 6.3.5): ln sum_{t in page} e^{x_t} (e^{c_t} - 1) for heads 2c, 2c + 1, from
      // the fast meter form's terms 2^{x_t - m} (e^{c_t} - 1) (m: the softmax's running max, log2 units)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float sum = col_sum8(pt[h]);
        const int head = 2 * (lane & 3) + h;
        if ((lane >> 2) == 0 && head < G)
          cdst[static_cast<size_t>(head) * cstride] = sum > 0.f ? logf(sum) + mnew[h] * kLn2 : -INFINITY;
      }
    } else if (vstate && cdst) {
      // the same in the general form (a radius above the fast form's range): per-page log-sum-exp
      float t[4];
#pragma unroll
      for (int v = 0; v < 4; ++v)
        t[v] = (x[v] == -INFINITY || cv[v] <= 0.f) ? -INFINITY : x[v] * kLn2 + cv[v] + logf(one_minus_exp_neg(cv[v]));
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float mx = col_max8(fmaxf(t[h], t[2 + h]));
        const float sum = col_sum8(mx == -INFINITY ? 0.f : expf(t[h] - mx) + expf(t[2 + h] - mx));
        const int head = 2 * (lane & 3) + h;
        if ((lane >> 2) == 0 && head < G) cdst[static_cast<size_t>(head) * cstride] = mx == -INFINITY ? -INFINITY
                                                                                              : mx + logf(sum);
      }
    }
    if (KDITHER && tier_b) {
      float uv[4];
      if (GS) {
        // u_t = sqrt(sum_g (sm_scale kappa)^2 ||q_g||^2 s_{g,t}^2) + sum_g sm_scale 2^-9 ||q_g||_1 s_{g,t}
        // (v = 2r + h: token g + 8r, head 2c + h)
        float var[4] = {0.f, 0.f, 0.f, 0.f}, bias[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int gr = 0; gr < kScaleGroups; ++gr) {
          const float2 A2 = *reinterpret_cast<const float2*>(f.gq + (4 + gr) * 8 + 2 * c);
          const float2 B1 = *reinterpret_cast<const float2*>(f.gq + (8 + gr) * 8 + 2 * c);
          const float2 sg = unpack_f16(*reinterpret_cast<const uint32_t*>(st + L::ksOff + 16 * g + 4 * gr));
          const float q0 = sg.x * sg.x, q1 = sg.y * sg.y;
          var[0] = __fmaf_rn(A2.x, q0, var[0]); var[1] = __fmaf_rn(A2.y, q0, var[1]);
          var[2] = __fmaf_rn(A2.x, q1, var[2]); var[3] = __fmaf_rn(A2.y, q1, var[3]);
          bias[0] = __fmaf_rn(B1.x, sg.x, bias[0]); bias[1] = __fmaf_rn(B1.y, sg.x, bias[1]);
          bias[2] = __fmaf_rn(B1.x, sg.y, bias[2]); bias[3] = __fmaf_rn(B1.y, sg.y, bias[3]);
        }
#pragma unroll
        for (int v = 0; v < 4; ++v) uv[v] = sqrtf(var[v]) + bias[v];
      } else {
        const f2x ab = f2_pack(f.alpha_b[0], f.alpha_b[1]);
        f2_unpack(f2_mul(ab, f2_splat(sk[0])), uv[0], uv[1]);
        f2_unpack(f2_mul(ab, f2_splat(sk[1])), uv[2], uv[3]);
      }
      if (OUTL) {
#pragma unroll
        for (int v = 0; v < 4; ++v) uv[v] = __fmaf_ru(f.beta_o[v & 1], kon[v >> 1], uv[v]) + f.gamma_o[v & 1];
      }
      accumulate_meter(uv, x, p, alpha, mnew, s.mu, s.su, s.slow_b);
    }
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) s.m[h] = mnew[h];

  // ---------------- O^T += V^T . P^T.  P'^T (B operand) = movmatrix of the S^T-shaped weights.
  float pw[4];
  f2_unpack(f2_mul(f2_pack(p[0], p[1]), f2_splat(kPvShift * sv[0])), pw[0], pw[1]);
  f2_unpack(f2_mul(f2_pack(p[2], p[3]), f2_splat(kPvShift * sv[1])), pw[2], pw[3]);
  if (GS) {
    // group-scaled INT8 values: the 32 channels of word block mm are scale group mm, so its two m-tiles take
    // P'^T built with the group's token scales; the dither product of the same m-tiles follows
    __syncwarp();  // the dither tile written in the key loop
#pragma unroll
    for (int mm = 0; mm < 4; ++mm) {
      const float2 sg = unpack_f16(*reinterpret_cast<const uint32_t*>(st + L::vsOff + 16 * g + 4 * mm));
      float pg[4];
      f2_unpack(f2_mul(f2_pack(p[0], p[1]), f2_splat(kPvShift * sg.x)), pg[0], pg[1]);
      f2_unpack(f2_mul(f2_pack(p[2], p[3]), f2_splat(kPvShift * sg.y)), pg[2], pg[3]);
      const uint32_t b0 = movmatrix_trans(pack_f16(pg[0], pg[1]));
      const uint32_t b1 = movmatrix_trans(pack_f16(pg[2], pg[3]));
      const uint4 vb = lds128(st + L::vOff + (mm * 32 + lane) * 16);
      const uint32_t words[4] = {vb.x, vb.y, vb.z, vb.w};
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const uint32_t x0 = words[2 * half], x1 = words[2 * half + 1];
        mma_f16_4(s.o[2 * mm + half], u8x2_to_f16x2(x0, 0), u8x2_to_f16x2(x0, 1), u8x2_to_f16x2(x1, 0),
                  u8x2_to_f16x2(x1, 1), b0, b1);
        const int mt = 2 * mm + half;
        const int mat = lane >> 3, r8 = lane & 7;
        const int row = ((mat >> 1) << 3) + r8;
        const int chunk = (2 * mt + (mat & 1)) ^ (row & 7);
        uint32_t fr[4];
        ldmatrix_x4_trans(fr, xi_tile + row * 256 + chunk * 16);
        mma_f16_4(s.o[mt], fr[0], fr[1], fr[2], fr[3], b0, b1);
      }
    }
  } else if (!fmt_is_16bit(VF)) {
    const uint32_t h01 = pack_f16(pw[0], pw[1]), h23 = pack_f16(pw[2], pw[3]);
    const uint32_t b0 = movmatrix_trans(h01);
    const uint32_t b1 = movmatrix_trans(h23);
    if (VDITHER) {
      // the operands below are code + 1152 (removed per page by a product with the constant -1152) and
      // -(xi + 9/2), whose 9/2 comes back as 9/2 sum_t P'_t per head when the piece is written: the lane's
      // part of that sum (tokens g, g + 8), rescaled like the accumulators
      const float2 q01 = unpack_f16(h01), q23 = unpack_f16(h23);
      f2_unpack(f2_fma(f2_pack(s.pv[0], s.pv[1]), f2_pack(alpha[0], alpha[1]), f2_pack(q01.x + q23.x, q01.y + q23.y)),
                s.pv[0], s.pv[1]);
    }
#pragma unroll
    for (int mm = 0; mm < 4; ++mm) {
      const uint4 vb = lds128(st + L::vOff + (mm * 32 + lane) * 16);
      const uint32_t words[4] = {vb.x, vb.y, vb.z, vb.w};
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const uint32_t u0 = words[2 * half], u1 = words[2 * half + 1];
        uint32_t a0, a1, a2, a3;
        if (VDITHER) {
          a0 = u8x2_to_f16x2_biased(u0, 0); a1 = u8x2_to_f16x2_biased(u0, 1);
          a2 = u8x2_to_f16x2_biased(u1, 0); a3 = u8x2_to_f16x2_biased(u1, 1);
        } else {
          a0 = e4m3x2_to_f16x2(u0 & 0xFFFFu); a1 = e4m3x2_to_f16x2(u0 >> 16);
          a2 = e4m3x2_to_f16x2(u1 & 0xFFFFu); a3 = e4m3x2_to_f16x2(u1 >> 16);
        }
        mma_f16_4(s.o[2 * mm + half], a0, a1, a2, a3, b0, b1);
        if (VDITHER) mma_f16_4(s.o[2 * mm + half], kInt8BiasF16x2, kInt8BiasF16x2, kInt8BiasF16x2, kInt8BiasF16x2, b0, b1);
      }
    }
    if (VDITHER) {
      // add (-(xi + 9/2))^T . P'^T: A fragments of the dither tile by transposed 8x8 loads
      __syncwarp();
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        // matrices: (tok 0-7, ch 16mt..+7), (tok 0-7, ch 16mt+8..), (tok 8-15, ch 16mt..), (tok 8-15, ch +8..)
        const int mat = lane >> 3, r8 = lane & 7;
        const int row = ((mat >> 1) << 3) + r8;
        const int chunk = (2 * mt + (mat & 1)) ^ (row & 7);
        uint32_t fr[4];
        ldmatrix_x4_trans(fr, xi_tile + row * 256 + chunk * 16);
        mma_f16_4(s.o[mt], fr[0], fr[1], fr[2], fr[3], b0, b1);
      }
    }
  } else {
    const uint32_t h01 = pack_bf16(pw[0], pw[1]), h23 = pack_bf16(pw[2], pw[3]);
    const float2 r01 = unpack_bf16(h01), r23 = unpack_bf16(h23);
    const uint32_t l01 = pack_bf16(pw[0] - r01.x, pw[1] - r01.y), l23 = pack_bf16(pw[2] - r23.x, pw[3] - r23.y);
    const uint32_t bh0 = movmatrix_trans(h01), bh1 = movmatrix_trans(h23);
    const uint32_t bl0 = movmatrix_trans(l01), bl1 = movmatrix_trans(l23);
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const uint4 vb = lds128(st + L::vOff + (mt * 32 + lane) * 16);
      mma_bf16_4(s.o[mt], vb.x, vb.y, vb.z, vb.w, bh0, bh1);
      mma_bf16_4(s.o[mt], vb.x, vb.y, vb.z, vb.w, bl0, bl1);
    }
  }
}

// ------------------------------------------------------------------------------------------------
// Page descriptors: lane l of a chunk describes page x0 + l of the warp's range.
struct Desc {
  int32_t phys;   // physical page in its cache (-1: out of range, skipped)
  uint32_t info;  // kv head (bits 0..6) | sequence (bits 7..22) | nvalid (bits 23..27) | prefix segment (bit 28)
                  // | present (bit 29) | last live page of the unit (bit 30)
};
// the unit's (sequence, kv head) pair as one key, and its parts
__device__ __forceinline__ uint32_t d_ukey(uint32_t i) { return i & 0x7FFFFFu; }
__device__ __forceinline__ int d_kvh(uint32_t i) { return static_cast<int>(i & 0x7Fu); }
__device__ __forceinline__ int d_seq(uint32_t i) { return static_cast<int>((i >> 7) & 0xFFFFu); }
__device__ __forceinline__ int d_nvalid(uint32_t i) { return static_cast<int>((i >> 23) & 31u); }
__device__ __forceinline__ bool d_prefix(uint32_t i) { return (i >> 28) & 1u; }
__device__ __forceinline__ bool d_present(uint32_t i) { return (i >> 29) & 1u; }
__device__ __forceinline__ bool d_last(uint32_t i) { return (i >> 30) & 1u; }

__device__ __forceinline__ Desc make_desc(const Args& a, const int32_t* cum, long long x, long long x_end) {
  Desc d{-1, 0u};
  if (x >= x_end) return d;
  // sequence: first s with Hkv * cum[s + 1] > x
  int lo = 0, hi = a.B - 1;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (static_cast<long long>(a.Hkv) * cum[mid + 1] > x) hi = mid; else lo = mid + 1;
  }
  const int s = lo;
  const int r = static_cast<int>(x - static_cast<long long>(a.Hkv) * cum[s]);  // < Hkv * pages of s (32-bit)
  const int P = cum[s + 1] - cum[s];
  const int kvh = r / P;
  const int p = r - kvh * P;
  int nvalid, phys;
  uint32_t pre = 0;
  if (p < a.prefix_pages) {
    pre = 1;
    phys = p;
    nvalid = min(kPage, a.prefix_len - p * kPage);
  } else {
    const int qp = p - a.prefix_pages;
    const int len = min(max(a.seq_lens[s], 0), a.max_pages * kPage);
    nvalid = min(kPage, len - qp * kPage);
    phys = a.bt[static_cast<size_t>(s) * a.max_pages + qp];
    if (phys < 0 || phys >= a.live.num_pages) {
      report(a.err, KVQ_ERR_DEVICE_BOUNDS);
      phys = -1;
    }
  }
  const uint32_t last = (!pre && p == P - 1) ? 1u : 0u;
  d.phys = phys;
  d.info = static_cast<uint32_t>(kvh) | (static_cast<uint32_t>(s) << 7) | (static_cast<uint32_t>(nvalid) << 23) |
           (pre << 28) | (1u << 29) | (last << 30);
  return d;
}

__device__ __forceinline__ Desc uniform_desc(Desc d) {
  return Desc{static_cast<int32_t>(uniform_u32(static_cast<uint32_t>(d.phys))), uniform_u32(d.info)};
}

// The copies of one page into a stage.  Every lane of the converged warp calls it with the same descriptor;
// the elected lane performs the barrier and copy operations.  A page without data (a block-table entry reported
// as out of range) only arrives.  PRED: that case is predicated instead of branched around (the operands are then
// computed either way and used only when valid); measured better for the 16-warp layouts, whose bodies sit at the
// 128-register cap (FP8 raw -5 % per launch, fewer spills), and worse for the 12-warp ones (INT8 +4 %).
template <int KF, int VF, int PKF, int PVF, bool METER, bool VALUE, bool OUTL, bool PRED>
__device__ __forceinline__ void issue_page(const Args& a, uint8_t* stage, uint64_t* bar, Desc d, uint64_t pol,
                                           uint32_t elected) {
  uint32_t leader = elected;
  if (PRED) {
    const uint32_t valid = d.phys >= 0 ? 1u : 0u;
    mbar_arrive(bar, elected & (valid ^ 1u));
    leader = elected & valid;
  } else if (d.phys < 0) {
    mbar_arrive(bar, elected);
    return;
  }
  const int kvh = d_kvh(d.info);
  const bool pre = d_prefix(d.info);
  if (PKF != kNoPrefix && pre) {
    using L = Layout<(PKF < 0 ? 0 : PKF), (PVF < 0 ? 0 : PVF), METER>;
    constexpr int pk = (PKF < 0 ? 0 : PKF), pv = (PVF < 0 ? 0 : PVF);
    const size_t tile = static_cast<size_t>(d.phys) * a.Hkv + kvh;
    mbar_arrive_expect_tx(bar, VALUE && a.value_on ? L::total : L::unvalued, leader);
    bulk_g2s(stage + L::kOff, a.pre.k + tile * L::kBytes, L::kBytes, bar, leader);
    bulk_g2s(stage + L::vOff, a.pre.v + tile * L::vBytes, L::vBytes, bar, leader);
    if (METER) bulk_g2s(stage + L::wOff, a.pre.w + tile * kTileBytesW, kTileBytesW, bar, leader);
    const size_t stile = static_cast<size_t>(kvh) * a.pre.num_pages + d.phys;
    if (fmt_has_scale(pk)) bulk_g2s(stage + L::ksOff, a.pre.ks + stile * tile_bytes_s(pk), tile_bytes_s(pk), bar, leader);
    if (fmt_has_scale(pv)) bulk_g2s(stage + L::vsOff, a.pre.vs + stile * tile_bytes_s(pv), tile_bytes_s(pv), bar, leader);
    if (METER && VALUE && a.value_on) bulk_g2s(stage + L::vwOff, a.pre.vw + stile * kTileBytesVW, kTileBytesVW, bar, leader);
  } else {
    using L = Layout<KF, VF, METER, OUTL>;
    const size_t tile = static_cast<size_t>(d.phys) * a.Hkv + kvh;
    if (a.wait_append && d_last(d.info)) {
      // the page holding the sequence's newest token: the append grid must have completed
      asm volatile("griddepcontrol.wait;" ::: "memory");
      asm volatile("fence.proxy.async.global;" ::: "memory");
    }
    const int ko_bytes = OUTL ? outlier_tile_bytes(a.live.n_out) : 0;
    mbar_arrive_expect_tx(bar, L::koOff + ko_bytes + (VALUE && a.value_on ? kTileBytesVW : 0), leader);
    bulk_g2s_hint(stage + L::kOff, a.live.k + tile * L::kBytes, L::kBytes, bar, pol, leader);
    bulk_g2s_hint(stage + L::vOff, a.live.v + tile * L::vBytes, L::vBytes, bar, pol, leader);
    if (METER) bulk_g2s_hint(stage + L::wOff, a.live.w + tile * kTileBytesW, kTileBytesW, bar, pol, leader);
    // scale planes are head-major, so consecutive pages of a unit share a 128-byte line
    const size_t stile = static_cast<size_t>(kvh) * a.live.num_pages + d.phys;
    if (fmt_has_scale(KF)) bulk_g2s(stage + L::ksOff, a.live.ks + stile * tile_bytes_s(KF), tile_bytes_s(KF), bar, leader);
    if (fmt_has_scale(VF)) bulk_g2s(stage + L::vsOff, a.live.vs + stile * tile_bytes_s(VF), tile_bytes_s(VF), bar, leader);
    if (OUTL) bulk_g2s_hint(stage + L::koOff, a.live.ko + stile * ko_bytes, ko_bytes, bar, pol, leader);
    if (METER && VALUE && a.value_on)
      bulk_g2s_hint(stage + L::vwOff, a.live.vw + stile * kTileBytesVW, kTileBytesVW, bar, pol, leader);
  }
}

// Partial of one (warp, unit) piece: per real head, (m, l, mc, sc, mu, su) and the 128 O^T values.
// PV: the value products used the dither operand -(xi + 9/2); 9/2 sum_t P'_t of each head is added back here.
template <bool PV>
__device__ __forceinline__ void write_piece(const Args& a, size_t slot, SoftState& s, float* vstate) {
  const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  float l[2], sc[2], su[2], vr[2] = {0.f, 0.f}, corr[2] = {0.f, 0.f};
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    l[h] = col_sum8(s.l[h]);
    sc[h] = col_sum8(s.sc[h]);
    su[h] = col_sum8(s.su[h]);
    if (PV) corr[h] = kDitherOffset * col_sum8(s.pv[h]);
  }
  float vmax = 0.f, cmax[2] = {0.f, 0.f}, om[2] = {0.f, 0.f};
  if (vstate) {
    const float4 v4 = *reinterpret_cast<const float4*>(vstate + 8 * lane);
    const float4 w4 = *reinterpret_cast<const float4*>(vstate + 8 * lane + 4);
    vr[0] = col_sum8(v4.x);
    vr[1] = col_sum8(v4.y);
    vmax = v4.z;
#pragma unroll
    for (int o = 16; o; o >>= 1) vmax = fmaxf(vmax, __shfl_xor_sync(kFull, vmax, o));
    cmax[0] = col_max8(w4.x);
    cmax[1] = col_max8(w4.y);
    om[0] = col_sum8(w4.z);
    om[1] = col_sum8(w4.w);
    // the next unit starts empty
    *reinterpret_cast<float4*>(vstate + 8 * lane) = make_float4(0.f, 0.f, 0.f, 0.f);
    *reinterpret_cast<float4*>(vstate + 8 * lane + 4) = make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int head = 2 * c + h;
    if (head < a.G) {
      float* acc = a.ws_acc + (slot * a.G + head) * kHeadDim;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        acc[16 * mt + g] = PV ? s.o[mt][h] + corr[h] : s.o[mt][h];
        acc[16 * mt + g + 8] = PV ? s.o[mt][2 + h] + corr[h] : s.o[mt][2 + h];
      }
      if (g == 0) {
        float* st = a.ws_stats + (slot * a.G + head) * kStatsFloats;
        *reinterpret_cast<float4*>(st) = make_float4(s.m[h], l[h], s.mc[h], sc[h]);
        *reinterpret_cast<float4*>(st + 4) = make_float4(s.mu[h], su[h], vr[h], vmax);
        *reinterpret_cast<float4*>(st + 8) = make_float4(cmax[h], om[h], 0.f, 0.f);
      }
    }
  }
}

// Zero the bytes of tokens nvalid..15 in a stage (a partial last page): the slots past the end of a
// sequence may hold anything, and zeros make their logit exactly the -inf bias, their value and
// radius exactly 0.  Runs once per unit at most; all lanes take part.
// vw_on: the stage holds a value witness tile (only then does the stage have room for it); OUTL: a key
// outlier tile of 8 (ko_wide: 16) columns.
template <int KF, int VF, bool METER, bool VALUE, bool OUTL = false>
__device__ void zero_tail(uint8_t* st, int nvalid, bool vw_on, bool ko_wide = false) {
  using L = Layout<KF, VF, METER, OUTL>;
  const int lane = threadIdx.x & 31;
  const int n = (kPage - nvalid) * kHeadDim;
  for (int e = lane; e < n; e += 32) {
    const int t = nvalid + e / kHeadDim, c = e % kHeadDim;
    // INT8 codes are offset binary: 0x80 is code 0
    if (fmt_is_16bit(KF)) *reinterpret_cast<uint16_t*>(st + L::kOff + k16_offset(t, c)) = 0;
    else st[L::kOff + (fmt_group_scales(KF) ? k8g_offset(t, c) : k8_offset(t, c))] = fmt_is_int8(KF) ? 0x80 : 0;
    if (fmt_is_16bit(VF)) *reinterpret_cast<uint16_t*>(st + L::vOff + v16_offset(t, c)) = 0;
    else st[L::vOff + v8_offset(t, c)] = fmt_is_int8(VF) ? 0x80 : 0;
  }
  for (int e = lane; e < (kPage - nvalid) * kBands; e += 32) {
    const int t = nvalid + e / kBands, b = e % kBands;
    if (METER) *reinterpret_cast<uint16_t*>(st + L::wOff + w_offset(t, b)) = 0;
  }
  for (int t = nvalid + lane; t < kPage; t += 32) {
    if (fmt_group_scales(KF)) {
      for (int gr = 0; gr < kScaleGroups; ++gr) *reinterpret_cast<uint16_t*>(st + L::ksOff + gs_offset(t, gr)) = 0;
    } else if (fmt_has_scale(KF)) {
      *reinterpret_cast<uint16_t*>(st + L::ksOff + s_offset(t)) = 0;
    }
    if (fmt_group_scales(VF)) {
      for (int gr = 0; gr < kScaleGroups; ++gr) *reinterpret_cast<uint16_t*>(st + L::vsOff + gs_offset(t, gr)) = 0;
    } else if (fmt_has_scale(VF)) {
      *reinterpret_cast<uint16_t*>(st + L::vsOff + s_offset(t)) = 0;
    }
    if (METER && VALUE && vw_on) {
      *reinterpret_cast<uint16_t*>(st + L::vwOff + vw_offset(t, 0)) = 0;
      *reinterpret_cast<uint16_t*>(st + L::vwOff + vw_offset(t, 1)) = 0;
    }
    if (OUTL)
      for (int col = 0; col < (ko_wide ? 16 : 8); ++col)
        *reinterpret_cast<uint16_t*>(st + L::koOff + ko_offset(t, col, ko_wide)) = 0;
  }
  __syncwarp();
}

// VALUE: the extended meter is compiled in (value side of the output bound and alternative bound
// shapes, chosen at run time; the value witness is staged only when the value side is on); without it
// no trace of either is left in the kernel.
// OUTL: the live cache stores a fixed set of key channels in fp16 (outlier bypass, INT8 keys).
template <int KF, int VF, int PKF, int PVF, int NW, bool METER, bool VALUE, bool OUTL>
__global__ void __launch_bounds__(NW * 32, 1) decode_split_kernel(const Args a) {
  extern __shared__ __align__(128) uint8_t smem[];
  // let the merge grid (programmatic dependent launch) be scheduled as soon as SMs free up
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  constexpr bool K16 = fmt_is_16bit(KF);
  constexpr bool XI = fmt_is_int8(KF) && fmt_is_int8(VF);
  constexpr bool GS = fmt_group_scales(KF);
  constexpr bool PV = XI && !GS;  // value products with the -(xi + 9/2) dither operand
  int32_t* cum = reinterpret_cast<int32_t*>(smem);
  const int cum_bytes = ((a.B + 1) * 4 + 127) & ~127;
  // UNI: the warp index and each page's descriptor go through uniform_u32, so the per-warp stage, barrier and copy
  // addresses live on the uniform datapath.  Measured for the 12-warp layouts: INT8 -9.2 % per launch (51 fewer
  // warp-instructions per page), cartridge -1.3 %; for the 16-warp ones +7 % (FP8 raw), so they keep plain values.
  constexpr bool UNI = NW != 16;
  constexpr bool VOTE = NW != 16 && !OUTL;  // the page's max update taken only on a vote (process_page)
  const int warp = UNI ? static_cast<int>(uniform_u32(threadIdx.x >> 5)) : static_cast<int>(threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;

  // ---- prefix sums of pages per sequence (block-wide scan)
  {
    __shared__ int32_t warp_tot[NW];
    const int per = (a.B + blockDim.x - 1) / blockDim.x;
    const int s0 = threadIdx.x * per;
    int loc = 0;
    for (int i = 0; i < per; ++i) {
      const int s = s0 + i;
      if (s < a.B) {
        int len = a.seq_lens[s];
        if (len < 0 || len > a.max_pages * kPage) {
          report(a.err, KVQ_ERR_DEVICE_BOUNDS);
          len = min(max(len, 0), a.max_pages * kPage);
        }
        loc += a.prefix_pages + (len + kPage - 1) / kPage;
      }
    }
    int inc = loc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(kFull, inc, o);
      if (lane >= o) inc += t;
    }
    if (lane == 31) warp_tot[warp] = inc;
    __syncthreads();
    int off = 0;
    for (int w = 0; w < warp; ++w) off += warp_tot[w];
    int run = off + inc - loc;  // exclusive prefix of this thread's first sequence
    for (int i = 0; i < per; ++i) {
      const int s = s0 + i;
      if (s < a.B) {
        if (s == 0) cum[0] = 0;
        int len = min(max(a.seq_lens[s], 0), a.max_pages * kPage);
        run += a.prefix_pages + (len + kPage - 1) / kPage;
        cum[s + 1] = run;
      }
    }
    __syncthreads();
  }

  const long long T = static_cast<long long>(a.Hkv) * cum[a.B];
  const long long W = min(static_cast<long long>(a.w_max), T);
  if (warp >= a.nwa) return;  // no block-wide barrier follows
  const int wid = blockIdx.x * a.nwa + warp;
  if (wid >= W) return;
  const long long x_begin = T * wid / W, x_end = T * (wid + 1) / W;
  const int n = static_cast<int>(x_end - x_begin);

  // ---- per-warp shared memory: stages, dither tile, query low parts, barriers
  const int lo_bytes = a.q_bf16 ? 0 : kQloBytes;
  static_assert(METER || !VALUE, "the extended meter rides on the meter");
  const int v_bytes = VALUE ? kVStateBytes : 0;
  const int gq_bytes = GS ? kGqBytes : 0;
  const int per_warp =
      a.stages * a.stage_bytes + (XI ? kXiScratch : 0) + lo_bytes + v_bytes + gq_bytes + kMaxStages * 8;
  uint8_t* wbase = smem + cum_bytes + warp * per_warp;
  uint8_t* xi_tile = wbase + a.stages * a.stage_bytes;
  float* vstate = VALUE ? reinterpret_cast<float*>(xi_tile + (XI ? kXiScratch : 0) + lo_bytes) : nullptr;
  float* gq = GS ? reinterpret_cast<float*>(xi_tile + (XI ? kXiScratch : 0) + lo_bytes + v_bytes) : nullptr;
  uint64_t* bars = reinterpret_cast<uint64_t*>(wbase + a.stages * a.stage_bytes + (XI ? kXiScratch : 0) + lo_bytes +
                                               v_bytes + gq_bytes);
  if (vstate) {
    *reinterpret_cast<float4*>(vstate + 8 * lane) = make_float4(0.f, 0.f, 0.f, 0.f);
    *reinterpret_cast<float4*>(vstate + 8 * lane + 4) = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const int ext = (a.value_on ? kExtValue : 0) | (a.shapes_on ? kExtShapes : 0);
  if (lane == 0) {
    for (int i = 0; i < a.stages; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
  }
  __syncwarp();

  const uint64_t pol = stream_policy(PKF != kNoPrefix && a.prefix_pages > 0);  // L2 policy of the live pages
  Desc cur = make_desc(a, cum, x_begin + lane, x_end);
  Desc nxt = make_desc(a, cum, x_begin + 32 + lane, x_end);
  // prologue: fill the ring
  for (int j = 0; j < a.stages && j < n; ++j) {
    const int32_t ph = __shfl_sync(kFull, cur.phys, j);
    const uint32_t in = __shfl_sync(kFull, cur.info, j);
    const Desc d{ph, in};
    issue_page<KF, VF, PKF, PVF, METER, VALUE, OUTL, NW == 16>(a, wbase + j * a.stage_bytes, &bars[j],
                                                               UNI ? uniform_desc(d) : d, pol, elect_one());
  }

  QFrag f;
  f.lo = reinterpret_cast<uint32_t*>(wbase + a.stages * a.stage_bytes + (XI ? kXiScratch : 0));
  f.has_lo = false;
  f.gq = gq;
  SoftState s;
  reset_state(s);
  int unit = -1;               // the current unit's index (sequence * Hkv + kv head)
  uint32_t ukey = 0xFFFFFFFFu;  // and its descriptor key
  long long unit_x0 = 0;   // gate support: global index of the current unit's first page
  float* crow = nullptr;   // gate support: the current unit's contribution row
  const float qk_scale = a.sm_scale * kLog2e;
  bool ok = true;
  int timeout_at = 0;

  const int g8 = lane >> 2;
  int stage = 0;
  uint32_t parity = 0;
  for (int j = 0; j < n; ++j) {
    if (j > 0 && (j & 31) == 0) {
      cur = nxt;
      nxt = make_desc(a, cum, x_begin + j + 32 + lane, x_end);
    }
    const int32_t phys = __shfl_sync(kFull, cur.phys, j & 31);
    const uint32_t info = __shfl_sync(kFull, cur.info, j & 31);
    if (d_ukey(info) != ukey) {
      if (unit >= 0) { write_piece<PV>(a, static_cast<size_t>(wid) + unit, s, vstate); reset_state(s); }
      ukey = d_ukey(info);
      const int seq = d_seq(info), kvh = d_kvh(info);
      unit = seq * a.Hkv + kvh;
      const int total = a.prefix_len + min(max(a.seq_lens[seq], 0), a.max_pages * kPage);
      load_q<K16, METER, OUTL, GS>(a, seq, kvh, total, f);
      if (VALUE && a.page_contrib) {
        // this unit's row of contributions, and the global index of its first page
        unit_x0 = static_cast<long long>(a.Hkv) * cum[seq] + static_cast<long long>(kvh) * (cum[seq + 1] - cum[seq]);
        crow = a.page_contrib + (static_cast<size_t>(seq) * a.Hq + static_cast<size_t>(kvh) * a.G) * a.contrib_stride;
      }
    }
    // every lane polls; the verdict is made warp-uniform before anyone leaves the loop
    if (!__all_sync(kFull, mbar_wait(&bars[stage], parity))) { ok = false; timeout_at = j; break; }
    uint8_t* st = wbase + stage * a.stage_bytes;
    if (phys >= 0) {
      const int kvh = d_kvh(info);
      const int nvalid = d_nvalid(info);
      const float xb0 = g8 < nvalid ? 0.f : -INFINITY, xb1 = g8 + 8 < nvalid ? 0.f : -INFINITY;
      if (PKF != kNoPrefix && d_prefix(info)) {
        constexpr int pk = (PKF < 0 ? 0 : PKF), pv = (PVF < 0 ? 0 : PVF);
        if (nvalid < kPage) zero_tail<pk, pv, METER, VALUE>(st, nvalid, a.value_on != 0);
        if (f.has_lo)
          process_page<pk, pv, METER, false, true, VOTE>(st, xi_tile, xb0, xb1, static_cast<uint32_t>(phys), a.pre, kvh, f,
                                                   s, qk_scale, a.tier_b != 0, vstate, ext,
                                                   crow ? crow + (x_begin + j - unit_x0) : nullptr, a.contrib_stride,
                                                   a.G);
        else
          process_page<pk, pv, METER, false, false, VOTE>(st, xi_tile, xb0, xb1, static_cast<uint32_t>(phys), a.pre, kvh,
                                                    f, s, qk_scale, a.tier_b != 0, vstate, ext,
                                                    crow ? crow + (x_begin + j - unit_x0) : nullptr, a.contrib_stride,
                                                    a.G);
      } else {
        if (nvalid < kPage) zero_tail<KF, VF, METER, VALUE, OUTL>(st, nvalid, a.value_on != 0, a.live.n_out > 4);
        // one test per page instead of one per k-step (measured per launch: FP8 raw -5.7 %, cartridge -1.0 %,
        // INT8 -0.9 %: the per-k-step form also loads the query's low parts whether or not it uses them)
        if (f.has_lo)
          process_page<KF, VF, METER, OUTL, true, VOTE>(st, xi_tile, xb0, xb1, static_cast<uint32_t>(phys), a.live, kvh, f,
                                                  s, qk_scale, a.tier_b != 0, vstate, ext,
                                                  crow ? crow + (x_begin + j - unit_x0) : nullptr, a.contrib_stride,
                                                  a.G);
        else
          process_page<KF, VF, METER, OUTL, false, VOTE>(st, xi_tile, xb0, xb1, static_cast<uint32_t>(phys), a.live, kvh, f,
                                                   s, qk_scale, a.tier_b != 0, vstate, ext,
                                                   crow ? crow + (x_begin + j - unit_x0) : nullptr, a.contrib_stride,
                                                   a.G);
      }
    }
    __syncwarp();
    const int jn = j + a.stages;
    if (jn < n) {
      const bool in_cur = (jn >> 5) == (j >> 5);
      const int32_t pc = __shfl_sync(kFull, cur.phys, jn & 31), pn = __shfl_sync(kFull, nxt.phys, jn & 31);
      const uint32_t ic = __shfl_sync(kFull, cur.info, jn & 31), inx = __shfl_sync(kFull, nxt.info, jn & 31);
      fence_proxy_async();
      const Desc d = in_cur ? Desc{pc, ic} : Desc{pn, inx};
      issue_page<KF, VF, PKF, PVF, METER, VALUE, OUTL, NW == 16>(a, st, &bars[stage], UNI ? uniform_desc(d) : d, pol,
                                                                 elect_one());
    }
    if (++stage == a.stages) { stage = 0; parity ^= 1u; }
  }
  if (!ok) {
    if (lane == 0) report(a.err, KVQ_ERR_TIMEOUT);
    // drain: wait (bounded) for the copies this warp issued and has not consumed (pages
    // timeout_at .. timeout_at + stages - 1), so no bulk copy lands after the warp exits
    for (int k = timeout_at; k < n && k < timeout_at + a.stages; ++k)
      (void)mbar_wait(&bars[k % a.stages], static_cast<uint32_t>((k / a.stages) & 1));
    return;
  }
  if (unit >= 0) write_piece<PV>(a, static_cast<size_t>(wid) + unit, s, vstate);
}

}  // namespace dec
}  // namespace kvq

namespace kvq {
namespace dec {

// Host launcher of one instantiation (the dynamic shared-memory limit is raised once per kernel and device:
// the setting belongs to the device's context).
// `programmatic`: launch as a programmatic dependent of the preceding grid in the stream (the
// fused append), which the kernel waits for where it reads that grid's output.
template <int KF, int VF, int PKF, int PVF, int NW, bool METER, bool VALUE, bool OUTL>
cudaError_t launch_decode(const Args& a, int grid, size_t smem, cudaStream_t s, bool programmatic) {
  auto kern = decode_split_kernel<KF, VF, PKF, PVF, NW, METER, VALUE, OUTL>;
  static size_t configured[kMaxDevices] = {};  // largest dynamic smem size set so far, per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices || smem > configured[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kMaxDevices) configured[dev] = smem;
  }
  if (!programmatic) {
    kern<<<grid, NW * 32, smem, s>>>(a);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(NW * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace dec
}  // namespace kvq

// Explicit instantiations are listed once, in decode_instances.inc, and split across translation
// units so they compile in parallel.
#define KVQ_DECODE_INSTANCE(KF, VF, PKF, PVF, NW, M, V, O)                                                      \
  template cudaError_t kvq::dec::launch_decode<KF, VF, PKF, PVF, NW, M, V, O>(const kvq::dec::Args&, int, size_t, \
                                                                               cudaStream_t, bool);
#define KVQ_DECODE_EXTERN(KF, VF, PKF, PVF, NW, M, V, O)                                                      \
  extern template cudaError_t kvq::dec::launch_decode<KF, VF, PKF, PVF, NW, M, V, O>(const kvq::dec::Args&, int, \
                                                                                      size_t, cudaStream_t, bool);
// meter off, meter on, meter with the extended meter (O: with the key outlier bypass)
#define KVQ_DECODE_INSTANCES3(KF, VF, PKF, PVF, NW, O)                                                     \
  KVQ_DECODE_INSTANCE(KF, VF, PKF, PVF, NW, false, false, O)                                              \
  KVQ_DECODE_INSTANCE(KF, VF, PKF, PVF, NW, true, false, O) KVQ_DECODE_INSTANCE(KF, VF, PKF, PVF, NW, true, true, O)
#define KVQ_DECODE_EXTERNS3(KF, VF, PKF, PVF, NW, O)                                                       \
  KVQ_DECODE_EXTERN(KF, VF, PKF, PVF, NW, false, false, O)                                                \
  KVQ_DECODE_EXTERN(KF, VF, PKF, PVF, NW, true, false, O) KVQ_DECODE_EXTERN(KF, VF, PKF, PVF, NW, true, true, O)
#define KVQ_DECODE_INSTANCES(KF, VF, PKF, PVF, NW) KVQ_DECODE_INSTANCES3(KF, VF, PKF, PVF, NW, false)
#define KVQ_DECODE_EXTERNS(KF, VF, PKF, PVF, NW) KVQ_DECODE_EXTERNS3(KF, VF, PKF, PVF, NW, false)
