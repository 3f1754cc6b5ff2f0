// decode_kernel.cuh -- split-KV paged GQA decode attention with the WitCert meter fused in.
//
// Work decomposition.  A "unit" is one (sequence, kv head); its logical page list is the shared
// prefix pages followed by the sequence's live pages ("Compress the shared cartridge", "One kernel
// spans cartridge and live KV": one logical sequence, one online softmax).  All units' pages are
// laid end to end and cut into equal contiguous ranges, one per warp of a persistent grid (a warp
// range may cross unit boundaries).  Each warp streams its pages through its own ring of shared-
// memory stages filled by bulk asynchronous copies (cp.async.bulk + mbarrier complete_tx), runs
// q.K^T, the witness dot product and P.V on tensor cores (mma.sync m16n8k16; the GQA group fills
// the M = 16 rows), keeps one online-softmax state and the meter accumulators per query head, and
// writes a partial (m, l, acc, meter sums) for every (warp, unit) piece it covered.  The merge
// kernel combines the pieces of each unit with log-sum-exp weights -- WitCert Sec. 6.2.2: the
// certificate A is a p~-weighted average, so per-split values merged under the same LSE weights
// give the global A exactly.
//
// Meter (WitCert Sec. 3 Thm. 1, Sec. 4.1 Thm. 2, Sec. 4.2, Sec. 4.3): with x_t the compressed
// logit, c_t = sm_scale * sum_b ||q_b|| w_{t,b}, the kernel accumulates
//     A - 1 = sum_t e^{x_t} (e^{c_t} - 1) / sum_t e^{x_t} = sum_t e^{x_t + c_t} (1 - e^{-c_t}) / sum_t e^{x_t}
// as a running maximum and a scaled sum of e^{x_t + c_t - max} (1 - e^{-c_t}), i.e. in the log
// domain ("we never truncate the error parameter"); Tier B does the same with
// u_t = sm_scale ||q|| s_t sqrt(2 ln(2S/delta_loc) / 12).
#pragma once

#include "kvq_common.cuh"

namespace kvq {
namespace dec {

constexpr int kWarps = 8;        // warps per CTA (one CTA per SM)
constexpr int kMaxStages = 8;
constexpr int kMaxBatch = 1024;  // sequences per call (prefix sums live in shared memory)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;
constexpr int kNoPrefix = -1;
constexpr int kXiScratch = 16 * 128 * 2;  // per-warp fp16 dither tile (INT8 values)
constexpr unsigned kFull = 0xffffffffu;
constexpr unsigned long long kWaitNs = 2000000000ull;  // a copy not landed after 2 s is reported as a timeout

struct Planes {
  const uint8_t* k;
  const uint8_t* v;
  const uint8_t* ks;
  const uint8_t* vs;
  const uint8_t* w;
  int num_pages;
  uint32_t layer;
  uint32_t seed_lo, seed_hi;
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
  int32_t* ws_cum;   // [B + 1] prefix sums of pages per sequence (written by CTA 0)
  float* ws_stats;   // [slots][G][8]
  float* ws_acc;     // [slots][G][128]
  int w_max;
  int stages;
  int stage_bytes;
  int32_t* err;
};

template <int KF, int VF, bool METER>
struct Layout {
  static constexpr int kBytes = tile_bytes_k(KF);
  static constexpr int vBytes = tile_bytes_v(VF);
  static constexpr int kOff = 0;
  static constexpr int vOff = kBytes;
  static constexpr int wOff = kBytes + vBytes;
  static constexpr int ksOff = wOff + (METER ? kTileBytesW : 0);
  static constexpr int vsOff = ksOff + (fmt_has_scale(KF) ? kTileBytesS : 0);
  static constexpr int total = vsOff + (fmt_has_scale(VF) ? kTileBytesS : 0);
};

// ------------------------------------------------------------------------------------------------
// PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
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
// Bounded wait: returns false if the phase did not complete within kWaitNs of wall time.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (;;) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > kWaitNs) return false;
  }
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
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
// two int8 codes (bytes sel: 0 -> bytes 0,1; 1 -> bytes 2,3 of w) -> f16x2 (exact):
// 0x6400 | (b ^ 0x80) is the fp16 value 1024 + b + 128.
__device__ __forceinline__ uint32_t s8x2_to_f16x2(uint32_t w_xor80, int sel) {
  const uint32_t h = __byte_perm(w_xor80, 0x64646464u, sel ? 0x4342 : 0x4140);
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

// ------------------------------------------------------------------------------------------------
// Per-warp state
struct QFrag {
  uint32_t hi[8][2];  // A fragment words a0, a2 per k-step (rows g; rows g+8 are zero)
  uint32_t lo[8][2];  // low parts (q - hi) when q is not exactly representable in the MMA type
  uint32_t qn_hi[2], qn_lo[2];  // band-norm A fragment (meter)
  bool has_lo;
  float cm_scale;   // c_t = cm_scale * (QN . W)  (natural units)
  float alpha_b;    // Tier B: u_t = alpha_b * s_t (natural units)
};

struct SoftState {
  float m;      // running max of the logits (log2 units), per row g
  float l;      // lane-partial sum of 2^{x - m}
  float mc, sc; // Tier A: running max of x + c*log2e, lane-partial sum
  float mu, su; // Tier B
  float o[16][4];
};

__device__ __forceinline__ void reset_state(SoftState& s) {
  s.m = -INFINITY; s.l = 0.f; s.mc = -INFINITY; s.sc = 0.f; s.mu = -INFINITY; s.su = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) { s.o[i][0] = 0.f; s.o[i][1] = 0.f; s.o[i][2] = 0.f; s.o[i][3] = 0.f; }
}

__device__ __forceinline__ float row_max4(float v) {
  v = fmaxf(v, __shfl_xor_sync(kFull, v, 1));
  v = fmaxf(v, __shfl_xor_sync(kFull, v, 2));
  return v;
}
__device__ __forceinline__ float row_sum4(float v) {
  v += __shfl_xor_sync(kFull, v, 1);
  v += __shfl_xor_sync(kFull, v, 2);
  return v;
}

// Build the q fragments of unit (seq, kv head).  K16 family: k-step kb = 2j + s covers channels
// 32j + 8c + 4s + {0,1} (slots 2c, 2c+1) and + {2,3} (slots 2c+8, 2c+9).  K8 family: kb = 4jj + s
// covers 64jj + 16c + 4s + {0..3}.  Band norms: slots (2c, 2c+1) <-> bands 4c, 4c+1 and
// (2c+8, 2c+9) <-> 4c+2, 4c+3.
template <bool K16, bool METER>
__device__ void load_q(const Args& a, int seq, int kvh, int seq_total, QFrag& f) {
  const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  const bool real = g < a.G;
  const int qh = kvh * a.G + (real ? g : 0);
  const size_t qbase = (static_cast<size_t>(seq) * a.Hq + qh) * kHeadDim;
  auto qv = [&](int ch) -> float {
    if (!real) return 0.f;
    if (a.q_bf16) return bf16_bits_to_f32(static_cast<const uint16_t*>(a.q)[qbase + ch]);
    return static_cast<const float*>(a.q)[qbase + ch];
  };
  bool any_lo = false;
#pragma unroll
  for (int kb = 0; kb < 8; ++kb) {
    const int ch0 = K16 ? (32 * (kb >> 1) + 8 * c + 4 * (kb & 1)) : (64 * (kb >> 2) + 16 * c + 4 * (kb & 3));
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float x0 = qv(ch0 + 2 * h), x1 = qv(ch0 + 2 * h + 1);
      if (K16) {
        f.hi[kb][h] = pack_bf16(x0, x1);
        const float2 r = unpack_bf16(f.hi[kb][h]);
        f.lo[kb][h] = pack_bf16(x0 - r.x, x1 - r.y);
      } else {
        f.hi[kb][h] = pack_f16(x0, x1);
        const float2 r = unpack_f16(f.hi[kb][h]);
        f.lo[kb][h] = pack_f16(x0 - r.x, x1 - r.y);
      }
      any_lo |= (f.lo[kb][h] & 0x7FFF7FFFu) != 0u;
    }
  }
  f.has_lo = __any_sync(kFull, any_lo);
  // band norms of q (for Tier A) and ||q|| (Tier B)
  float qn[4];
  float sq_all = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int b = 4 * c + i;
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float u = qv(4 * b + e), w = qv(64 + 4 * b + e);
      s = __fmaf_rn(u, u, s);
      s = __fmaf_rn(w, w, s);
    }
    qn[i] = sqrtf(s);
    sq_all += s;
  }
  if (METER) {
    // normalise the row's band norms by a power of two so that max < 2 (fp16 range), split hi/lo
    float mx = fmaxf(fmaxf(qn[0], qn[1]), fmaxf(qn[2], qn[3]));
    mx = row_max4(mx);
    int e2 = 0;
    if (mx > 0.f) frexpf(mx, &e2);  // mx = f * 2^e2, f in [0.5, 1)
    const float inv = ldexpf(1.f, -e2);
    float hv[4], lv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float v = qn[i] * inv;
      const __half h = __float2half_rn(v);
      hv[i] = __half2float(h);
      lv[i] = v - hv[i];
    }
    f.qn_hi[0] = pack_f16(hv[0], hv[1]);
    f.qn_hi[1] = pack_f16(hv[2], hv[3]);
    f.qn_lo[0] = pack_f16(lv[0], lv[1]);
    f.qn_lo[1] = pack_f16(lv[2], lv[3]);
    f.cm_scale = a.sm_scale * ldexpf(1.f, e2);
    const float qnorm = sqrtf(row_sum4(sq_all));
    // kappa = sqrt(2 ln(2S / delta_loc) / 12)
    const float kappa = sqrtf(2.f * (logf(2.f * static_cast<float>(seq_total)) - a.ln_delta_loc) / 12.f);
    f.alpha_b = a.sm_scale * qnorm * kappa;
  }
}

// ------------------------------------------------------------------------------------------------
// One page of 16 tokens for one kv head.  `st` is the stage holding the page's tiles.
template <int KF, int VF, bool METER>
__device__ __forceinline__ void process_page(const uint8_t* st, uint8_t* xi_tile, int nvalid, uint32_t phys,
                                             const Planes& pl, int kvh, const QFrag& f, SoftState& s,
                                             float qk_scale, bool tier_b) {
  using L = Layout<KF, VF, METER>;
  const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  constexpr bool K16 = fmt_is_16bit(KF);
  constexpr bool KDITHER = KF == KVQ_FMT_INT8_DITHER;
  constexpr bool VDITHER = VF == KVQ_FMT_INT8_DITHER;

  // ---------------- logits S = q . k (tensor cores); columns are tokens 8nt + 2c, 8nt + 2c + 1
  float S[2][4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) { S[nt][0] = S[nt][1] = S[nt][2] = S[nt][3] = 0.f; }
  if (K16) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 kb = lds128(st + L::kOff + ((nt * 4 + j) * 32 + lane) * 16);
        mma_bf16(S[nt], f.hi[2 * j][0], f.hi[2 * j][1], kb.x, kb.y);
        mma_bf16(S[nt], f.hi[2 * j + 1][0], f.hi[2 * j + 1][1], kb.z, kb.w);
        if (f.has_lo) {
          mma_bf16(S[nt], f.lo[2 * j][0], f.lo[2 * j][1], kb.x, kb.y);
          mma_bf16(S[nt], f.lo[2 * j + 1][0], f.lo[2 * j + 1][1], kb.z, kb.w);
        }
      }
    }
  } else {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        const uint4 kb = lds128(st + L::kOff + ((nt * 2 + jj) * 32 + lane) * 16);
        const uint32_t words[4] = {kb.x, kb.y, kb.z, kb.w};
#pragma unroll
        for (int sidx = 0; sidx < 4; ++sidx) {
          uint32_t b0, b1;
          if (KDITHER) {
            const uint32_t wx = words[sidx] ^ 0x80808080u;
            b0 = s8x2_to_f16x2(wx, 0);
            b1 = s8x2_to_f16x2(wx, 1);
          } else {
            b0 = e4m3x2_to_f16x2(words[sidx] & 0xFFFFu);
            b1 = e4m3x2_to_f16x2(words[sidx] >> 16);
          }
          const int kb_i = 4 * jj + sidx;
          mma_f16(S[nt], f.hi[kb_i][0], f.hi[kb_i][1], b0, b1);
          if (f.has_lo) mma_f16(S[nt], f.lo[kb_i][0], f.lo[kb_i][1], b0, b1);
          if (KDITHER) {
            // subtract q . xi: dither of token 8nt + g, channels 64jj + 16c + 4sidx + {0..3}
            const uint32_t slot = phys * kPage + 8 * nt + g;
            const uint32_t grp = 16 * jj + 4 * c + sidx;
            const float4 d = dither4(slot, pl.layer, static_cast<uint32_t>(kvh), grp, pl.seed_lo, pl.seed_hi);
            const uint32_t nb0 = pack_f16(-d.x, -d.y), nb1 = pack_f16(-d.z, -d.w);
            mma_f16(S[nt], f.hi[kb_i][0], f.hi[kb_i][1], nb0, nb1);
            if (VDITHER) {
              // stage the dither for the value side (token-major fp16 tile, 16-byte chunks xor-swizzled)
              const int row = 8 * nt + g;
              const int ch = 64 * jj + 16 * c + 4 * sidx;
              const int chunk = (ch >> 3) ^ (row & 7);
              uint2 w2;
              w2.x = pack_f16(d.x, d.y);
              w2.y = pack_f16(d.z, d.w);
              *reinterpret_cast<uint2*>(xi_tile + row * 256 + chunk * 16 + (ch & 7) * 2) = w2;
            }
          }
        }
      }
    }
  }

  // ---------------- per-token scales of the lane's four columns (tokens 2c, 2c+1, 2c+8, 2c+9)
  float sk[4] = {1.f, 1.f, 1.f, 1.f}, sv[4] = {1.f, 1.f, 1.f, 1.f};
  if (fmt_has_scale(KF)) {
    const uint2 w = lds64(st + L::ksOff + c * 8);
    const float2 a0 = unpack_f16(w.x), a1 = unpack_f16(w.y);
    sk[0] = a0.x; sk[1] = a0.y; sk[2] = a1.x; sk[3] = a1.y;
  }
  if (fmt_has_scale(VF)) {
    const uint2 w = lds64(st + L::vsOff + c * 8);
    const float2 a0 = unpack_f16(w.x), a1 = unpack_f16(w.y);
    sv[0] = a0.x; sv[1] = a0.y; sv[2] = a1.x; sv[3] = a1.y;
  }

  // ---------------- online softmax (log2 domain); v = 2 nt + e <-> token 8nt + 2c + e
  bool valid[4];
  float x[4];
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    const int tok = 8 * (v >> 1) + 2 * c + (v & 1);
    valid[v] = tok < nvalid;
    float sc = qk_scale;
    if (fmt_has_scale(KF)) sc *= sk[v];
    x[v] = valid[v] ? S[v >> 1][v & 1] * sc : -INFINITY;
  }
  const float mx = row_max4(fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3])));
  const float m_new = fmaxf(s.m, mx);
  const float alpha = (m_new == -INFINITY) ? 1.f : ex2(s.m - m_new);
  float p[4];
#pragma unroll
  for (int v = 0; v < 4; ++v) p[v] = valid[v] ? ex2(x[v] - m_new) : 0.f;
  s.l = s.l * alpha + ((p[0] + p[1]) + (p[2] + p[3]));
  if (__any_sync(kFull, alpha != 1.f)) {
#pragma unroll
    for (int i = 0; i < 16; ++i) { s.o[i][0] *= alpha; s.o[i][1] *= alpha; }
  }
  s.m = m_new;

  // ---------------- meter (Tier A witness bound; Tier B dither certificate)
  if (METER) {
    float Cm[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) { Cm[nt][0] = Cm[nt][1] = Cm[nt][2] = Cm[nt][3] = 0.f; }
    const uint4 wb = lds128(st + L::wOff + lane * 16);
    mma_f16(Cm[0], f.qn_hi[0], f.qn_hi[1], wb.x, wb.y);
    mma_f16(Cm[0], f.qn_lo[0], f.qn_lo[1], wb.x, wb.y);
    mma_f16(Cm[1], f.qn_hi[0], f.qn_hi[1], wb.z, wb.w);
    mma_f16(Cm[1], f.qn_lo[0], f.qn_lo[1], wb.z, wb.w);
    float cz[4], cv[4];
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      cv[v] = valid[v] ? Cm[v >> 1][v & 1] * f.cm_scale : 0.f;
      cz[v] = valid[v] ? __fmaf_rn(cv[v], kLog2e, x[v]) : -INFINITY;
    }
    const float mz = row_max4(fmaxf(fmaxf(cz[0], cz[1]), fmaxf(cz[2], cz[3])));
    const float mc_new = fmaxf(s.mc, mz);
    if (mc_new != -INFINITY) {
      float acc = 0.f;
#pragma unroll
      for (int v = 0; v < 4; ++v) acc += valid[v] ? ex2(cz[v] - mc_new) * one_minus_exp_neg(cv[v]) : 0.f;
      s.sc = s.sc * ex2(s.mc - mc_new) + acc;
      s.mc = mc_new;
    }
    if (KDITHER && tier_b) {
      float uz[4], uv[4];
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        uv[v] = valid[v] ? f.alpha_b * sk[v] : 0.f;
        uz[v] = valid[v] ? __fmaf_rn(uv[v], kLog2e, x[v]) : -INFINITY;
      }
      const float mu = row_max4(fmaxf(fmaxf(uz[0], uz[1]), fmaxf(uz[2], uz[3])));
      const float mu_new = fmaxf(s.mu, mu);
      if (mu_new != -INFINITY) {
        float acc = 0.f;
#pragma unroll
        for (int v = 0; v < 4; ++v) acc += valid[v] ? ex2(uz[v] - mu_new) * one_minus_exp_neg(uv[v]) : 0.f;
        s.su = s.su * ex2(s.mu - mu_new) + acc;
        s.mu = mu_new;
      }
    }
  }

  // ---------------- P . V (tensor cores).  A rows g = query heads, k = the page's 16 tokens.
  float pw[4];
#pragma unroll
  for (int v = 0; v < 4; ++v) pw[v] = valid[v] ? p[v] * (kPvShift * sv[v]) : 0.f;
  // partial pages: zero the value codes of invalid tokens (their bytes may hold NaN patterns)
  const bool partial = nvalid < kPage;
  if (!fmt_is_16bit(VF)) {
    const uint32_t a0 = pack_f16(pw[0], pw[1]), a2 = pack_f16(pw[2], pw[3]);
    uint32_t mask = 0xFFFFFFFFu;
    if (partial) {
      mask = (valid[0] ? 0xFFu : 0u) | (valid[1] ? 0xFF00u : 0u) | (valid[2] ? 0xFF0000u : 0u) |
             (valid[3] ? 0xFF000000u : 0u);
    }
#pragma unroll
    for (int m4 = 0; m4 < 4; ++m4) {
      const uint4 vb = lds128(st + L::vOff + (m4 * 32 + lane) * 16);
      const uint32_t words[4] = {vb.x & mask, vb.y & mask, vb.z & mask, vb.w & mask};
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        uint32_t b0, b1;
        if (VDITHER) {
          const uint32_t wx = words[r] ^ 0x80808080u;
          b0 = s8x2_to_f16x2(wx, 0);
          b1 = s8x2_to_f16x2(wx, 1);
        } else {
          b0 = e4m3x2_to_f16x2(words[r] & 0xFFFFu);
          b1 = e4m3x2_to_f16x2(words[r] >> 16);
        }
        mma_f16(s.o[4 * m4 + r], a0, a2, b0, b1);
      }
    }
    if (VDITHER) {
      // subtract p' . xi: B fragments of the dither tile via transposed 8x8 loads
      __syncwarp();
      const uint32_t na0 = a0 ^ 0x80008000u, na2 = a2 ^ 0x80008000u;
#pragma unroll
      for (int np = 0; np < 8; ++np) {
        // matrices: (tokens 0-7, chunk 2np), (8-15, 2np), (0-7, 2np+1), (8-15, 2np+1)
        const int mat = lane >> 3, r8 = lane & 7;
        const int row = ((mat & 1) << 3) + r8;
        const int chunk = (2 * np + (mat >> 1)) ^ (row & 7);
        uint32_t fr[4];
        ldmatrix_x4_trans(fr, xi_tile + row * 256 + chunk * 16);
        mma_f16(s.o[2 * np], na0, na2, fr[0], fr[1]);
        mma_f16(s.o[2 * np + 1], na0, na2, fr[2], fr[3]);
      }
    }
  } else {
    const uint32_t h0 = pack_bf16(pw[0], pw[1]), h2 = pack_bf16(pw[2], pw[3]);
    const float2 r0 = unpack_bf16(h0), r2 = unpack_bf16(h2);
    const uint32_t l0 = pack_bf16(pw[0] - r0.x, pw[1] - r0.y), l2 = pack_bf16(pw[2] - r2.x, pw[3] - r2.y);
    uint32_t mlo = 0xFFFFFFFFu, mhi = 0xFFFFFFFFu;
    if (partial) {
      mlo = (valid[0] ? 0xFFFFu : 0u) | (valid[1] ? 0xFFFF0000u : 0u);
      mhi = (valid[2] ? 0xFFFFu : 0u) | (valid[3] ? 0xFFFF0000u : 0u);
    }
#pragma unroll
    for (int m8 = 0; m8 < 8; ++m8) {
      const uint4 vb = lds128(st + L::vOff + (m8 * 32 + lane) * 16);
      const uint32_t b00 = vb.x & mlo, b01 = vb.y & mhi, b10 = vb.z & mlo, b11 = vb.w & mhi;
      mma_bf16(s.o[2 * m8], h0, h2, b00, b01);
      mma_bf16(s.o[2 * m8], l0, l2, b00, b01);
      mma_bf16(s.o[2 * m8 + 1], h0, h2, b10, b11);
      mma_bf16(s.o[2 * m8 + 1], l0, l2, b10, b11);
    }
  }
}

// ------------------------------------------------------------------------------------------------
// Page descriptors: lane l of a chunk describes page x0 + l of the warp's range.
struct Desc {
  int32_t phys;   // physical page in its cache (-1: out of range, skipped)
  uint32_t info;  // unit (bits 0..22) | nvalid (bits 23..27) | prefix segment (bit 28) | present (bit 29)
};
__device__ __forceinline__ int d_unit(uint32_t i) { return static_cast<int>(i & 0x7FFFFFu); }
__device__ __forceinline__ int d_nvalid(uint32_t i) { return static_cast<int>((i >> 23) & 31u); }
__device__ __forceinline__ bool d_prefix(uint32_t i) { return (i >> 28) & 1u; }
__device__ __forceinline__ bool d_present(uint32_t i) { return (i >> 29) & 1u; }

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
  const long long r = x - static_cast<long long>(a.Hkv) * cum[s];
  const int P = cum[s + 1] - cum[s];
  const int kvh = static_cast<int>(r / P);
  const int p = static_cast<int>(r - static_cast<long long>(kvh) * P);
  const int unit = s * a.Hkv + kvh;
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
  d.phys = phys;
  d.info = static_cast<uint32_t>(unit) | (static_cast<uint32_t>(nvalid) << 23) | (pre << 28) | (1u << 29);
  return d;
}

template <int KF, int VF, int PKF, int PVF, bool METER>
__device__ __forceinline__ void issue_page(const Args& a, uint8_t* stage, uint64_t* bar, Desc d) {
  // lane 0 only
  if (d.phys < 0) {
    mbar_arrive(bar);
    return;
  }
  const int kvh = d_unit(d.info) % a.Hkv;
  const bool pre = d_prefix(d.info);
  if (PKF != kNoPrefix && pre) {
    using L = Layout<(PKF < 0 ? 0 : PKF), (PVF < 0 ? 0 : PVF), METER>;
    constexpr int pk = (PKF < 0 ? 0 : PKF), pv = (PVF < 0 ? 0 : PVF);
    const size_t tile = static_cast<size_t>(d.phys) * a.Hkv + kvh;
    mbar_arrive_expect_tx(bar, L::total);
    bulk_g2s(stage + L::kOff, a.pre.k + tile * L::kBytes, L::kBytes, bar);
    bulk_g2s(stage + L::vOff, a.pre.v + tile * L::vBytes, L::vBytes, bar);
    if (METER) bulk_g2s(stage + L::wOff, a.pre.w + tile * kTileBytesW, kTileBytesW, bar);
    if (fmt_has_scale(pk)) bulk_g2s(stage + L::ksOff, a.pre.ks + tile * kTileBytesS, kTileBytesS, bar);
    if (fmt_has_scale(pv)) bulk_g2s(stage + L::vsOff, a.pre.vs + tile * kTileBytesS, kTileBytesS, bar);
  } else {
    using L = Layout<KF, VF, METER>;
    const size_t tile = static_cast<size_t>(d.phys) * a.Hkv + kvh;
    mbar_arrive_expect_tx(bar, L::total);
    bulk_g2s(stage + L::kOff, a.live.k + tile * L::kBytes, L::kBytes, bar);
    bulk_g2s(stage + L::vOff, a.live.v + tile * L::vBytes, L::vBytes, bar);
    if (METER) bulk_g2s(stage + L::wOff, a.live.w + tile * kTileBytesW, kTileBytesW, bar);
    if (fmt_has_scale(KF)) bulk_g2s(stage + L::ksOff, a.live.ks + tile * kTileBytesS, kTileBytesS, bar);
    if (fmt_has_scale(VF)) bulk_g2s(stage + L::vsOff, a.live.vs + tile * kTileBytesS, kTileBytesS, bar);
  }
}

__device__ __forceinline__ void flush(const Args& a, int warp_id, int unit, SoftState& s) {
  const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  const float l = row_sum4(s.l), sc = row_sum4(s.sc), su = row_sum4(s.su);
  const size_t slot = static_cast<size_t>(warp_id) + unit;
  if (g < a.G) {
    float* acc = a.ws_acc + (slot * a.G + g) * kHeadDim;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
      *reinterpret_cast<float2*>(acc + 8 * nt + 2 * c) = make_float2(s.o[nt][0], s.o[nt][1]);
    if (c == 0) {
      float* st = a.ws_stats + (slot * a.G + g) * 8;
      *reinterpret_cast<float4*>(st) = make_float4(s.m, l, s.mc, sc);
      *reinterpret_cast<float4*>(st + 4) = make_float4(s.mu, su, 0.f, 0.f);
    }
  }
}

template <int KF, int VF, int PKF, int PVF, bool METER>
__global__ void __launch_bounds__(kWarps * 32, 1) decode_split_kernel(const Args a) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr bool K16 = fmt_is_16bit(KF);
  constexpr bool XI = (KF == KVQ_FMT_INT8_DITHER && VF == KVQ_FMT_INT8_DITHER);
  int32_t* cum = reinterpret_cast<int32_t*>(smem);
  const int cum_bytes = ((a.B + 1) * 4 + 127) & ~127;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- prefix sums of pages per sequence (block-wide scan)
  {
    __shared__ int32_t warp_tot[kWarps];
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
    if (blockIdx.x == 0)
      for (int i = threadIdx.x; i <= a.B; i += blockDim.x) a.ws_cum[i] = cum[i];
  }

  const long long T = static_cast<long long>(a.Hkv) * cum[a.B];
  const long long W = min(static_cast<long long>(a.w_max), T);
  const int wid = blockIdx.x * kWarps + warp;
  if (wid >= W) return;
  const long long x_begin = T * wid / W, x_end = T * (wid + 1) / W;
  const int n = static_cast<int>(x_end - x_begin);

  // ---- per-warp shared memory: stages, dither tile, barriers
  const int per_warp = a.stages * a.stage_bytes + (XI ? kXiScratch : 0) + kMaxStages * 8;
  uint8_t* wbase = smem + cum_bytes + warp * per_warp;
  uint8_t* xi_tile = wbase + a.stages * a.stage_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(wbase + a.stages * a.stage_bytes + (XI ? kXiScratch : 0));
  if (lane == 0) {
    for (int i = 0; i < a.stages; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
  }
  __syncwarp();

  Desc cur = make_desc(a, cum, x_begin + lane, x_end);
  Desc nxt = make_desc(a, cum, x_begin + 32 + lane, x_end);
  // prologue: fill the ring
  for (int j = 0; j < a.stages && j < n; ++j) {
    const int32_t ph = __shfl_sync(kFull, cur.phys, j);
    const uint32_t in = __shfl_sync(kFull, cur.info, j);
    if (lane == 0) issue_page<KF, VF, PKF, PVF, METER>(a, wbase + j * a.stage_bytes, &bars[j], Desc{ph, in});
  }

  QFrag f;
  SoftState s;
  reset_state(s);
  int unit = -1;
  const float qk_scale = a.sm_scale * kLog2e;
  bool ok = true;
  int timeout_at = 0;

  for (int j = 0; j < n; ++j) {
    if (j > 0 && (j & 31) == 0) {
      cur = nxt;
      nxt = make_desc(a, cum, x_begin + j + 32 + lane, x_end);
    }
    const int32_t phys = __shfl_sync(kFull, cur.phys, j & 31);
    const uint32_t info = __shfl_sync(kFull, cur.info, j & 31);
    const int u = d_unit(info);
    if (u != unit) {
      if (unit >= 0) { flush(a, wid, unit, s); reset_state(s); }
      unit = u;
      const int seq = u / a.Hkv, kvh = u % a.Hkv;
      const int total = a.prefix_len + min(max(a.seq_lens[seq], 0), a.max_pages * kPage);
      load_q<K16, METER>(a, seq, kvh, total, f);
    }
    const int stage = j % a.stages;
    const uint32_t parity = static_cast<uint32_t>((j / a.stages) & 1);
    // every lane polls; the verdict is made warp-uniform before anyone leaves the loop
    if (!__all_sync(kFull, mbar_wait(&bars[stage], parity))) { ok = false; timeout_at = j; break; }
    if (phys >= 0) {
      const uint8_t* st = wbase + stage * a.stage_bytes;
      const int kvh = u % a.Hkv;
      if (PKF != kNoPrefix && d_prefix(info)) {
        constexpr int pk = (PKF < 0 ? 0 : PKF), pv = (PVF < 0 ? 0 : PVF);
        process_page<pk, pv, METER>(st, xi_tile, d_nvalid(info), static_cast<uint32_t>(phys), a.pre, kvh, f, s,
                                    qk_scale, a.tier_b != 0);
      } else {
        process_page<KF, VF, METER>(st, xi_tile, d_nvalid(info), static_cast<uint32_t>(phys), a.live, kvh, f, s,
                                    qk_scale, a.tier_b != 0);
      }
    }
    __syncwarp();
    const int jn = j + a.stages;
    if (jn < n) {
      const bool in_cur = (jn >> 5) == (j >> 5);
      const int32_t pc = __shfl_sync(kFull, cur.phys, jn & 31), pn = __shfl_sync(kFull, nxt.phys, jn & 31);
      const uint32_t ic = __shfl_sync(kFull, cur.info, jn & 31), inx = __shfl_sync(kFull, nxt.info, jn & 31);
      if (lane == 0) {
        fence_proxy_async();
        issue_page<KF, VF, PKF, PVF, METER>(a, wbase + stage * a.stage_bytes, &bars[stage],
                                            in_cur ? Desc{pc, ic} : Desc{pn, inx});
      }
    }
  }
  if (!ok) {
    if (lane == 0) report(a.err, KVQ_ERR_TIMEOUT);
    // drain: wait (bounded) for the copies this warp issued and has not consumed (pages
    // timeout_at .. timeout_at + stages - 1), so no bulk copy lands after the warp exits
    for (int k = timeout_at; k < n && k < timeout_at + a.stages; ++k)
      (void)mbar_wait(&bars[k % a.stages], static_cast<uint32_t>((k / a.stages) & 1));
    return;
  }
  if (unit >= 0) flush(a, wid, unit, s);
}

}  // namespace dec
}  // namespace kvq

namespace kvq {
namespace dec {

// Host launcher of one instantiation (the dynamic shared-memory limit is raised once per kernel).
template <int KF, int VF, int PKF, int PVF, bool METER>
cudaError_t launch_decode(const Args& a, int grid, size_t smem, cudaStream_t s) {
  auto kern = decode_split_kernel<KF, VF, PKF, PVF, METER>;
  static size_t configured = 0;  // largest dynamic smem size set so far
  if (smem > configured) {
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    configured = smem;
  }
  kern<<<grid, kWarps * 32, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace dec
}  // namespace kvq

// Explicit instantiations are listed once, in decode_instances.inc, and split across translation
// units so they compile in parallel.
#define KVQ_DECODE_INSTANCE(KF, VF, PKF, PVF, M) \
  template cudaError_t kvq::dec::launch_decode<KF, VF, PKF, PVF, M>(const kvq::dec::Args&, int, size_t, cudaStream_t);
#define KVQ_DECODE_EXTERN(KF, VF, PKF, PVF, M) \
  extern template cudaError_t kvq::dec::launch_decode<KF, VF, PKF, PVF, M>(const kvq::dec::Args&, int, size_t, cudaStream_t);
