// decode.cu -- kvq_decode_attn / kvq_decode_workspace_size: argument checks, workspace layout,
// shared-memory stage sizing, and dispatch to the decode and merge kernels.
#include <cmath>
#include <mutex>

#include "decode_kernel.cuh"

#define KVQ_X(KF, VF, PKF, PVF, NW) KVQ_DECODE_EXTERNS(KF, VF, PKF, PVF, NW)
#include "decode_instances.inc"
#undef KVQ_X
KVQ_DECODE_EXTERNS3(KVQ_FMT_INT8_DITHER, KVQ_FMT_INT8_DITHER, -1, -1, 12, true)

namespace kvq {
cudaError_t launch_append_newest(const kvq_cache& c, const void* k, const void* v, int in_bf16,
                                 const int32_t* block_table, int max_pages, const int32_t* seq_lens, int batch,
                                 int32_t* err, cudaStream_t s);  // append.cu

namespace dec {

// ------------------------------------------------------------------------------------------------
// Merge of the (warp, unit) pieces: one warp per (sequence, query head).  Piece statistics are
// loaded lane-parallel and combined by shuffles; the O^T partials are read with independent
// loads.  WitCert Sec. 6.2.2: the certificate A is a p~-weighted average, so per-piece sums
// merged under the same log-sum-exp weights give the global A exactly.
__device__ __forceinline__ void lse_combine(float& m, float& s, float m2, float s2) {
  const float mm = fmaxf(m, m2);
  if (mm == -INFINITY) return;
  s = (m == -INFINITY ? 0.f : s * ex2(m - mm)) + (m2 == -INFINITY ? 0.f : s2 * ex2(m2 - mm));
  m = mm;
}

// (m, l, r, u): r and u are merged with the same weights as l (the extended meter's p~-weighted sums:
// sum_t e^{x_t} rho^v_t and sum_t e^{x_t} (1 - e^{-c_t}))
__device__ __forceinline__ void lse_combine3(float& m, float& l, float& r, float& u, float m2, float l2, float r2,
                                             float u2) {
  const float mm = fmaxf(m, m2);
  if (mm == -INFINITY) return;
  const float a = m == -INFINITY ? 0.f : ex2(m - mm), b = m2 == -INFINITY ? 0.f : ex2(m2 - mm);
  l = l * a + l2 * b;
  r = r * a + r2 * b;
  u = u * a + u2 * b;
  m = mm;
}

__global__ void __launch_bounds__(256) merge_kernel(const Args a) {
  const int lane = threadIdx.x & 31;
  const long long gw = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (gw >= static_cast<long long>(a.B) * a.Hq) return;
  const int seq = static_cast<int>(gw / a.Hq), qh = static_cast<int>(gw % a.Hq);
  const int kvh = qh / a.G, row = qh % a.G;
  const int unit = seq * a.Hkv + kvh;
  // inputs of the call are read before the wait (the decode grid's outputs only after it): the
  // sequence's page range [c0, c1) and the total cB, by the decode's own clamping of the lengths
  const int total = a.prefix_len + min(max(a.seq_lens[seq], 0), a.max_pages * kPage);
  int c0 = 0, cB = 0;
  for (int s = lane; s < a.B; s += 32) {
    const int n = a.prefix_pages + (min(max(a.seq_lens[s], 0), a.max_pages * kPage) + kPage - 1) / kPage;
    cB += n;
    if (s < seq) c0 += n;
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) {
    c0 += __shfl_xor_sync(kFull, c0, off);
    cB += __shfl_xor_sync(kFull, cB, off);
  }
  const int c1 = c0 + a.prefix_pages + (total - a.prefix_len + kPage - 1) / kPage;
  float* o = a.out + static_cast<size_t>(gw) * kHeadDim;
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the decode grid's pieces are complete and visible
  const long long T = static_cast<long long>(a.Hkv) * cB;
  const int P = c1 - c0;
  if (P == 0) {
    *reinterpret_cast<float4*>(o + 4 * lane) = make_float4(0.f, 0.f, 0.f, 0.f);
    if (a.meter_state && lane == 0) {
      float* ms = a.meter_state + gw * KVQ_METER_STATE_FLOATS;
      *reinterpret_cast<float4*>(ms) = make_float4(-INFINITY, a.tier_b ? -INFINITY : NAN, -INFINITY,
                                                   static_cast<float>(total));
      *reinterpret_cast<float4*>(ms + 4) = make_float4(a.value_on ? 0.f : NAN, a.value_on ? 0.f : NAN,
                                                       a.shapes_on ? 0.f : NAN, a.shapes_on ? 0.f : NAN);
    }
    return;
  }
  // page indices fit in 32 bits (checked by the host)
  const int Ti = static_cast<int>(T);
  const int W = min(a.w_max, Ti);
  const int b_u = a.Hkv * c0 + kvh * P, e_u = b_u + P;
  // warp w covers pages [T w / W, T (w + 1) / W); with T = q W + r that start is q w + (r w) / W.  The
  // warp holding page x: a binary32 estimate of x W / T, corrected against the exact starts.
  const int qd = Ti / W, rd = Ti % W;
  auto start_of = [&](int w) { return qd * w + (rd * w) / W; };
  auto warp_of = [&](int x) {
    int w = min(W - 1, static_cast<int>(static_cast<float>(x) * (static_cast<float>(W) / static_cast<float>(Ti))));
    while (w + 1 < W && start_of(w + 1) <= x) ++w;
    while (w > 0 && start_of(w) > x) --w;
    return w;
  };
  const int w_lo = warp_of(b_u), w_hi = warp_of(e_u - 1);
  const int np = w_hi - w_lo + 1;
  const size_t p0 = static_cast<size_t>(w_lo) + unit;  // piece slot of the unit's first piece
  auto stats = [&](int i) { return a.ws_stats + ((p0 + i) * a.G + row) * kStatsFloats; };
  auto accp = [&](int i) { return a.ws_acc + ((p0 + i) * a.G + row) * kHeadDim + 4 * lane; };

  // one round of loads: every piece's statistics (lane-parallel) and the first kU pieces' partial
  // outputs (this lane's four channels), all independent of each other
  constexpr int kU = 16;
  float4 v[kU];
#pragma unroll
  for (int k = 0; k < kU; ++k)
    if (k < np) v[k] = *reinterpret_cast<const float4*>(accp(k));
  // this lane's pieces (lane, lane + 32, ...) merged locally; then one max and one weighted sum over
  // the lanes.  (m, l), (mc, sc), (mu, su): running max (log2 units) and scaled sums; r (value side) and
  // u (1 - A^- of the shapes) ride on l's weights.
  const bool ext = a.value_on | a.shapes_on;
  float m = -INFINITY, l = 0.f, mc = -INFINITY, sc = 0.f, mu = -INFINITY, su = 0.f, vr = 0.f, om = 0.f;
  float vmax = 0.f, cmax = 0.f;
  float m_mine = -INFINITY;  // the running max of piece `lane` (pieces < 32), for the weights below
  for (int i = lane; i < np; i += 32) {
    const float4 s4 = *reinterpret_cast<const float4*>(stats(i));
    const float2 t2 = *reinterpret_cast<const float2*>(stats(i) + 4);
    float r2 = 0.f, u2 = 0.f;
    if (ext) {
      const float2 q2 = *reinterpret_cast<const float2*>(stats(i) + 6);
      const float2 e2 = *reinterpret_cast<const float2*>(stats(i) + 8);
      r2 = q2.x;
      u2 = e2.y;
      vmax = fmaxf(vmax, q2.y);
      cmax = fmaxf(cmax, e2.x);
    }
    if (i < 32) m_mine = s4.x;
    lse_combine3(m, l, vr, om, s4.x, s4.y, r2, u2);
    lse_combine(mc, sc, s4.z, s4.w);
    lse_combine(mu, su, t2.x, t2.y);
  }
  // the maxima over the lanes, then every lane's sums rescaled to them and added up
  float gm = m, gc = mc, gu = mu;
#pragma unroll
  for (int off = 16; off; off >>= 1) {
    gm = fmaxf(gm, __shfl_xor_sync(kFull, gm, off));
    gc = fmaxf(gc, __shfl_xor_sync(kFull, gc, off));
    gu = fmaxf(gu, __shfl_xor_sync(kFull, gu, off));
  }
  {
    const float wl = m == -INFINITY ? 0.f : ex2(m - gm);
    const float wc = mc == -INFINITY ? 0.f : ex2(mc - gc);
    const float wu = mu == -INFINITY ? 0.f : ex2(mu - gu);
    l *= wl; vr *= wl; om *= wl; sc *= wc; su *= wu;
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) {
    l += __shfl_xor_sync(kFull, l, off);
    sc += __shfl_xor_sync(kFull, sc, off);
    if (a.tier_b) su += __shfl_xor_sync(kFull, su, off);
    if (ext) {
      vr += __shfl_xor_sync(kFull, vr, off);
      om += __shfl_xor_sync(kFull, om, off);
      vmax = fmaxf(vmax, __shfl_xor_sync(kFull, vmax, off));
      cmax = fmaxf(cmax, __shfl_xor_sync(kFull, cmax, off));
    }
  }
  m = gm; mc = gc; mu = gu;
  if (!a.tier_b) { mu = -INFINITY; su = 0.f; }
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const float wt_mine = m_mine == -INFINITY ? 0.f : ex2(m_mine - m);
#pragma unroll
  for (int k = 0; k < kU; ++k) {
    const float wt = __shfl_sync(kFull, wt_mine, k);
    if (k < np && wt != 0.f) {
      acc.x += v[k].x * wt; acc.y += v[k].y * wt; acc.z += v[k].z * wt; acc.w += v[k].w * wt;
    }
  }
  for (int i = kU; i < np; ++i) {  // units split over more than kU warps (few, long sequences)
    const float wt = i < 32 ? __shfl_sync(kFull, wt_mine, i) : [&] {
      const float mi = stats(i)[0];
      return mi == -INFINITY ? 0.f : ex2(mi - m);
    }();
    if (wt != 0.f) {
      const float4 vi = *reinterpret_cast<const float4*>(accp(i));
      acc.x += vi.x * wt; acc.y += vi.y * wt; acc.z += vi.z * wt; acc.w += vi.w * wt;
    }
  }
  const float inv = kPvShiftInv / l;
  *reinterpret_cast<float4*>(o + 4 * lane) = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  if (a.meter_state && lane == 0) {
    const float lse2 = m + log2f(l);
    const float la = (a.meter_on && sc > 0.f) ? (mc + log2f(sc) - lse2) * kLn2 : -INFINITY;
    const float lb = a.tier_b ? ((su > 0.f) ? (mu + log2f(su) - lse2) * kLn2 : -INFINITY) : NAN;
    float* ms = a.meter_state + gw * KVQ_METER_STATE_FLOATS;
    *reinterpret_cast<float4*>(ms) = make_float4(la, lb, lse2 * kLn2, static_cast<float>(total));
    *reinterpret_cast<float4*>(ms + 4) = make_float4(a.value_on ? vr / l : NAN, a.value_on ? vmax : NAN,
                                                     a.shapes_on ? cmax : NAN, a.shapes_on ? om / l : NAN);
  }
}

}  // namespace dec
}  // namespace kvq

using namespace kvq;
using namespace kvq::dec;

namespace {


int device_sm_count() {
  static int cache[kMaxDevices] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  if (!cache[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev] = n;
  }
  return cache[dev];
}

int device_smem_optin() {
  static int cache[kMaxDevices] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  if (!cache[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return 0;
    cache[dev] = n;
  }
  return cache[dev];
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct WsLayout {
  size_t stats, acc, total;
};

WsLayout ws_layout(int batch, int hkv, int hq, int w_max) {
  const int G = hq / hkv;
  const size_t slots = static_cast<size_t>(w_max) + static_cast<size_t>(batch) * hkv;
  WsLayout l;
  l.stats = 0;
  l.acc = l.stats + align256(slots * G * kStatsFloats * sizeof(float));
  l.total = l.acc + align256(slots * G * kHeadDim * sizeof(float));
  return l;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Stage bytes of a page: the Layout<kf, vf, meter, outl> bytes up to the value witness, plus the value
// witness tile with the value side on.
int page_bytes(int kf, int vf, bool meter, bool value, bool outl = false) {
  return tile_bytes_k(kf) + tile_bytes_v(vf) + (meter ? kTileBytesW : 0) + (value ? kTileBytesVW : 0) +
         (fmt_has_scale(kf) ? tile_bytes_s(kf) : 0) + (fmt_has_scale(vf) ? tile_bytes_s(vf) : 0) +
         (outl ? outlier_tile_bytes(kMaxOutlierPairs) : 0);
}

kvq_status check_cache(const kvq_cache* c, bool meter) {
  if (!c) return KVQ_ERR_INVALID_ARG;
  if (c->k_fmt < 0 || c->k_fmt > 4 || c->v_fmt < 0 || c->v_fmt > 4) return KVQ_ERR_UNSUPPORTED_LAYOUT;
  if (fmt_group_scales(c->k_fmt) != fmt_group_scales(c->v_fmt)) return KVQ_ERR_UNSUPPORTED_LAYOUT;
  if (c->num_kv_heads <= 0 || c->num_pages < 0 || c->reserved != 0) return KVQ_ERR_INVALID_ARG;
  if (!c->k_data || !c->v_data || !aligned16(c->k_data) || !aligned16(c->v_data)) return KVQ_ERR_INVALID_ARG;
  if (fmt_has_scale(c->k_fmt) && (!c->k_scale || !aligned16(c->k_scale))) return KVQ_ERR_INVALID_ARG;
  if (fmt_has_scale(c->v_fmt) && (!c->v_scale || !aligned16(c->v_scale))) return KVQ_ERR_INVALID_ARG;
  if (meter && (!c->witness || !aligned16(c->witness))) return KVQ_ERR_INVALID_ARG;
  if (c->n_outlier_pairs < 0 || c->n_outlier_pairs > kMaxOutlierPairs || c->reserved2 != 0) return KVQ_ERR_INVALID_ARG;
  if (c->n_outlier_pairs > 0) {
    if (c->k_fmt != KVQ_FMT_INT8_DITHER) return KVQ_ERR_UNSUPPORTED_LAYOUT;
    if (!c->outlier_pairs || !c->k_outlier || !aligned16(c->k_outlier)) return KVQ_ERR_INVALID_ARG;
  }
  return KVQ_OK;
}

Planes planes_of(const kvq_cache* c) {
  Planes p{};
  if (!c) return p;
  p.k = static_cast<const uint8_t*>(c->k_data);
  p.v = static_cast<const uint8_t*>(c->v_data);
  p.ks = reinterpret_cast<const uint8_t*>(c->k_scale);
  p.vs = reinterpret_cast<const uint8_t*>(c->v_scale);
  p.w = reinterpret_cast<const uint8_t*>(c->witness);
  p.vw = reinterpret_cast<const uint8_t*>(c->v_witness);
  p.ko = reinterpret_cast<const uint8_t*>(c->k_outlier);
  p.opairs = c->outlier_pairs;
  p.n_out = c->n_outlier_pairs;
  p.num_pages = c->num_pages;
  p.layer = static_cast<uint32_t>(c->layer);
  p.seed_lo = static_cast<uint32_t>(c->dither_seed);
  p.seed_hi = static_cast<uint32_t>(c->dither_seed >> 32);
  for (int r = 0; r < 10; ++r) {
    p.rk0[r] = p.seed_lo + static_cast<uint32_t>(r) * kPhiloxW0;
    p.rk1[r] = p.seed_hi + static_cast<uint32_t>(r) * kPhiloxW1;
  }
  return p;
}

using Launcher = cudaError_t (*)(const Args&, int, size_t, cudaStream_t, bool);

struct Pick {
  Launcher launch;
  int warps;
};

Pick pick(int kf, int vf, int pkf, int pvf, bool meter, bool value, bool outl) {
  if (outl) {  // the fixed-channel key outlier bypass exists for the INT8-dithered layout without a prefix
    constexpr int I8 = KVQ_FMT_INT8_DITHER;
    if (kf != I8 || vf != I8 || pkf != kNoPrefix || pvf != kNoPrefix) return Pick{nullptr, 0};
    return Pick{!meter  ? &launch_decode<I8, I8, -1, -1, 12, false, false, true>
                : value ? &launch_decode<I8, I8, -1, -1, 12, true, true, true>
                        : &launch_decode<I8, I8, -1, -1, 12, true, false, true>,
                12};
  }
#define KVQ_X(KF, VF, PKF, PVF, NW)                                                                       \
  if (kf == (KF) && vf == (VF) && pkf == (PKF) && pvf == (PVF))                                           \
    return Pick{!meter  ? &launch_decode<KF, VF, PKF, PVF, NW, false, false, false>                        \
                : value ? &launch_decode<KF, VF, PKF, PVF, NW, true, true, false>                          \
                        : &launch_decode<KF, VF, PKF, PVF, NW, true, false, false>,                        \
                NW};
#include "decode_instances.inc"
#undef KVQ_X
  return Pick{nullptr, 0};
}

}  // namespace

extern "C" size_t kvq_decode_workspace_size(int32_t batch, int32_t num_kv_heads, int32_t num_q_heads) {
  if (batch < 0 || num_kv_heads <= 0 || num_q_heads <= 0 || num_q_heads % num_kv_heads) return 0;
  const int sms = device_sm_count();
  if (sms <= 0) return 0;
  return ws_layout(batch, num_kv_heads, num_q_heads, sms * kMaxWarps).total;
}

namespace {

// Measurement hook (kvq_debug_time_decode): events recorded around the decode kernel's launch.
thread_local cudaEvent_t g_time_start = nullptr, g_time_stop = nullptr;

kvq_status decode_impl(const kvq_cache* cache, const void* k_new, const void* v_new, int32_t kv_dtype,
                       const kvq_cache* prefix, int32_t prefix_len, const void* q, int32_t q_dtype, int32_t batch,
                       int32_t num_q_heads, const int32_t* block_table, int32_t max_pages_per_seq,
                       const int32_t* seq_lens, float sm_scale, const kvq_meter_params* mp, float* out,
                       float* meter_state, void* workspace, size_t ws_bytes, int32_t* err_word, cudaStream_t s,
                       const kvq_decode_extras* extras = nullptr) {
  const bool meter = mp != nullptr;
  const bool contrib = extras && extras->page_log_contrib;
  if (extras && extras->reserved != 0) return KVQ_ERR_INVALID_ARG;
  if (contrib) {
    if (!meter) return KVQ_ERR_INVALID_ARG;
    const long long need = (static_cast<long long>(prefix && prefix_len > 0 ? prefix_len : 0) + kPage - 1) / kPage +
                           max_pages_per_seq;
    if (extras->contrib_stride < need) return KVQ_ERR_INVALID_ARG;
  }
  kvq_status st = check_cache(cache, meter);
  if (st != KVQ_OK) return st;
  const bool fused_append = k_new != nullptr || v_new != nullptr;
  if (fused_append) {
    if (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new)) return KVQ_ERR_INVALID_ARG;
    if (kv_dtype != KVQ_DTYPE_F32 && kv_dtype != KVQ_DTYPE_BF16) return KVQ_ERR_INVALID_ARG;
    if (!cache->witness || !aligned16(cache->witness)) return KVQ_ERR_INVALID_ARG;
  }
  if (prefix && prefix_len > 0) {
    if ((st = check_cache(prefix, meter)) != KVQ_OK) return st;
    if (prefix->num_kv_heads != cache->num_kv_heads) return KVQ_ERR_INVALID_ARG;
    if (static_cast<long long>(prefix->num_pages) * kPage < prefix_len) return KVQ_ERR_INVALID_ARG;
    if (fmt_is_16bit(prefix->k_fmt) != fmt_is_16bit(cache->k_fmt)) return KVQ_ERR_UNSUPPORTED_LAYOUT;
  }
  if (prefix_len < 0 || (prefix_len > 0 && !prefix)) return KVQ_ERR_INVALID_ARG;
  const int hkv = cache->num_kv_heads;
  if (hkv > KVQ_MAX_KV_HEADS) return KVQ_ERR_INVALID_ARG;
  if (batch < 0 || batch > kMaxBatch || num_q_heads <= 0 || num_q_heads % hkv) return KVQ_ERR_INVALID_ARG;
  const int G = num_q_heads / hkv;
  if (G > kMaxGroup) return KVQ_ERR_UNSUPPORTED_LAYOUT;
  if (q_dtype != KVQ_DTYPE_F32 && q_dtype != KVQ_DTYPE_BF16) return KVQ_ERR_INVALID_ARG;
  if (max_pages_per_seq < 0 || !std::isfinite(sm_scale)) return KVQ_ERR_INVALID_ARG;
  if (meter) {
    if (!(mp->tiers & KVQ_TIER_A) || (mp->tiers & ~15u) || mp->reserved != 0) return KVQ_ERR_INVALID_ARG;
    if (mp->tiers & KVQ_TIER_V) {
      if (!cache->v_witness || !aligned16(cache->v_witness)) return KVQ_ERR_INVALID_ARG;
      if (prefix && prefix_len > 0 && (!prefix->v_witness || !aligned16(prefix->v_witness)))
        return KVQ_ERR_INVALID_ARG;
    }
    if (mp->tiers & KVQ_TIER_B) {
      if (!fmt_is_int8(cache->k_fmt) || (prefix && prefix_len > 0)) return KVQ_ERR_INVALID_ARG;
      if (!(mp->delta_req > 0.0 && mp->delta_req < 1.0) || mp->n_layers <= 0 || mp->n_q_heads <= 0 || mp->n_steps <= 0)
        return KVQ_ERR_INVALID_ARG;
    }
    if (!meter_state) return KVQ_ERR_INVALID_ARG;
  }
  if (batch == 0) return KVQ_OK;
  if (!q || !seq_lens || !out || !workspace || (max_pages_per_seq > 0 && !block_table)) return KVQ_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(workspace) || (meter_state && !aligned16(meter_state))) return KVQ_ERR_INVALID_ARG;
  const int sms = device_sm_count();
  const int smem_max = device_smem_optin();
  if (sms <= 0 || smem_max <= 0) return KVQ_ERR_CUDA;
  const WsLayout wl = ws_layout(batch, hkv, num_q_heads, sms * kMaxWarps);
  if (ws_bytes < wl.total) return KVQ_ERR_WORKSPACE_TOO_SMALL;
  // page indices of the flattened (unit, page) space are 32-bit
  if (static_cast<long long>(batch) * hkv * ((prefix && prefix_len > 0 ? (prefix_len + kPage - 1) / kPage : 0) +
                                             static_cast<long long>(max_pages_per_seq)) > 0x7FFFFFFFll)
    return KVQ_ERR_INVALID_ARG;

  const bool has_prefix = prefix && prefix_len > 0;
  const int pkf = has_prefix ? prefix->k_fmt : kNoPrefix;
  const int pvf = has_prefix ? prefix->v_fmt : kNoPrefix;
  const bool outl = cache->n_outlier_pairs > 0;
  const bool ext_meter = meter && ((mp->tiers & (KVQ_TIER_V | KVQ_TIER_S)) || contrib);
  const Pick pk = pick(cache->k_fmt, cache->v_fmt, pkf, pvf, meter, ext_meter, outl);
  if (!pk.launch) return KVQ_ERR_UNSUPPORTED_LAYOUT;
  const int nw = pk.warps;

  Args a{};
  a.live = planes_of(cache);
  a.pre = planes_of(has_prefix ? prefix : nullptr);
  a.prefix_len = has_prefix ? prefix_len : 0;
  a.prefix_pages = (a.prefix_len + kPage - 1) / kPage;
  a.Hkv = hkv;
  a.G = G;
  a.Hq = num_q_heads;
  a.B = batch;
  a.q = q;
  a.q_bf16 = q_dtype == KVQ_DTYPE_BF16;
  a.wait_append = fused_append ? 1 : 0;
  a.bt = block_table;
  a.max_pages = max_pages_per_seq;
  a.seq_lens = seq_lens;
  a.sm_scale = sm_scale;
  a.tier_b = meter && (mp->tiers & KVQ_TIER_B) ? 1 : 0;
  a.ln_delta_loc = 0.f;
  if (a.tier_b)
    a.ln_delta_loc = static_cast<float>(
        std::log(mp->delta_req / (static_cast<double>(mp->n_layers) * mp->n_q_heads * mp->n_steps)));
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.out = out;
  a.meter_state = meter_state;
  a.meter_on = meter ? 1 : 0;
  a.value_on = meter && (mp->tiers & KVQ_TIER_V) ? 1 : 0;
  a.shapes_on = meter && (mp->tiers & KVQ_TIER_S) ? 1 : 0;
  a.page_contrib = contrib ? extras->page_log_contrib : nullptr;
  a.contrib_stride = contrib ? extras->contrib_stride : 0;
  a.ws_stats = reinterpret_cast<float*>(ws + wl.stats);
  a.ws_acc = reinterpret_cast<float*>(ws + wl.acc);
  a.err = err_word;

  // stage size: the larger of the two segments' page footprints (16-byte multiple by construction)
  int sb = page_bytes(cache->k_fmt, cache->v_fmt, meter, a.value_on, outl);
  if (has_prefix) sb = std::max(sb, page_bytes(prefix->k_fmt, prefix->v_fmt, meter, a.value_on));
  const bool xi = fmt_is_int8(cache->k_fmt) && fmt_is_int8(cache->v_fmt);
  const bool gs = fmt_group_scales(cache->k_fmt);
  const int cum_bytes = ((batch + 1) * 4 + 127) & ~127;
  const int lo_bytes = q_dtype == KVQ_DTYPE_F32 ? kQloBytes : 0;
  const bool ext = ext_meter;  // the extended-meter kernel variant and its per-lane state
  // warps that stream pages: the layout's warps per CTA, fewer when their two page stages do not fit shared
  // memory (large pages with an fp32 query's low parts)
  const int per_warp_fixed =
      (xi ? kXiScratch : 0) + lo_bytes + (ext ? kVStateBytes : 0) + (gs ? kGqBytes : 0) + kMaxStages * 8;
  int nwa = nw, stages = 0;
  for (; nwa >= 4; --nwa) {
    stages = (smem_max - 1024 - cum_bytes - nwa * per_warp_fixed) / (nwa * sb);
    if (stages >= 2) break;
  }
  if (stages < 2) return KVQ_ERR_UNSUPPORTED_LAYOUT;
  if (stages > kMaxStages) stages = kMaxStages;
  const int w_max = sms * nwa;
  a.w_max = w_max;
  a.nwa = nwa;
  a.stages = stages;
  a.stage_bytes = sb;
  const int fixed = cum_bytes + nwa * per_warp_fixed;
  const size_t smem = static_cast<size_t>(fixed) + static_cast<size_t>(nwa) * stages * sb;

  if (fused_append) {
    // the newest tokens first; the decode is a programmatic dependent of that grid and waits for it
    // only before it loads a page that holds one of them
    if (launch_append_newest(*cache, k_new, v_new, kv_dtype == KVQ_DTYPE_BF16, block_table, max_pages_per_seq,
                             seq_lens, batch, err_word, s) != cudaSuccess)
      return KVQ_ERR_CUDA;
  }
  if (g_time_start && cudaEventRecord(g_time_start, s) != cudaSuccess) return KVQ_ERR_CUDA;
  if (pk.launch(a, sms, smem, s, fused_append && !g_time_start) != cudaSuccess) return KVQ_ERR_CUDA;
  if (g_time_stop && cudaEventRecord(g_time_stop, s) != cudaSuccess) return KVQ_ERR_CUDA;
  // merge: programmatic dependent launch, so its launch overlaps the decode grid's tail
  const long long merge_threads = static_cast<long long>(batch) * num_q_heads * 32;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((merge_threads + 255) / 256));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, merge_kernel, a) != cudaSuccess) return KVQ_ERR_CUDA;
  return KVQ_OK;
}

}  // namespace

extern "C" kvq_status kvq_debug_time_decode(void* start_event, void* stop_event) {
  if ((start_event == nullptr) != (stop_event == nullptr)) return KVQ_ERR_INVALID_ARG;
  g_time_start = static_cast<cudaEvent_t>(start_event);
  g_time_stop = static_cast<cudaEvent_t>(stop_event);
  return KVQ_OK;
}

extern "C" kvq_status kvq_decode_attn(const kvq_cache* cache, const kvq_cache* prefix, int32_t prefix_len,
                                      const void* q, int32_t q_dtype, int32_t batch, int32_t num_q_heads,
                                      const int32_t* block_table, int32_t max_pages_per_seq,
                                      const int32_t* seq_lens, float sm_scale, const kvq_meter_params* mp,
                                      float* out, float* meter_state, void* workspace, size_t ws_bytes,
                                      int32_t* err_word, kvq_stream_t stream) {
  return decode_impl(cache, nullptr, nullptr, KVQ_DTYPE_F32, prefix, prefix_len, q, q_dtype, batch, num_q_heads,
                     block_table, max_pages_per_seq, seq_lens, sm_scale, mp, out, meter_state, workspace, ws_bytes,
                     err_word, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" kvq_status kvq_decode_attn_ex(const kvq_cache* cache, const void* k_new, const void* v_new, int32_t kv_dtype,
                                         const kvq_cache* prefix, int32_t prefix_len, const void* q, int32_t q_dtype,
                                         int32_t batch, int32_t num_q_heads, const int32_t* block_table,
                                         int32_t max_pages_per_seq, const int32_t* seq_lens, float sm_scale,
                                         const kvq_meter_params* mp, const kvq_decode_extras* extras, float* out,
                                         float* meter_state, void* workspace, size_t ws_bytes, int32_t* err_word,
                                         kvq_stream_t stream) {
  if ((k_new == nullptr) != (v_new == nullptr)) return KVQ_ERR_INVALID_ARG;
  return decode_impl(cache, k_new, v_new, kv_dtype, prefix, prefix_len, q, q_dtype, batch, num_q_heads, block_table,
                     max_pages_per_seq, seq_lens, sm_scale, mp, out, meter_state, workspace, ws_bytes, err_word,
                     reinterpret_cast<cudaStream_t>(stream), extras);
}

extern "C" kvq_status kvq_decode_attn_append(const kvq_cache* cache, const void* k_new, const void* v_new,
                                             int32_t kv_dtype, const kvq_cache* prefix, int32_t prefix_len,
                                             const void* q, int32_t q_dtype, int32_t batch, int32_t num_q_heads,
                                             const int32_t* block_table, int32_t max_pages_per_seq,
                                             const int32_t* seq_lens, float sm_scale, const kvq_meter_params* mp,
                                             float* out, float* meter_state, void* workspace, size_t ws_bytes,
                                             int32_t* err_word, kvq_stream_t stream) {
  if (!k_new || !v_new) return KVQ_ERR_INVALID_ARG;
  return decode_impl(cache, k_new, v_new, kv_dtype, prefix, prefix_len, q, q_dtype, batch, num_q_heads, block_table,
                     max_pages_per_seq, seq_lens, sm_scale, mp, out, meter_state, workspace, ws_bytes, err_word,
                     reinterpret_cast<cudaStream_t>(stream));
}

// ------------------------------------------------------------------------------------------------
// kvq_decode_attn_noalloc: kvq_decode_attn with its scratch in a file-scope device array, for
// callers that can hand the library only inputs and outputs (see include/kvq.h).  The array is a
// device symbol: its host-side name is not a device address, so the address is looked up once per
// device with cudaGetSymbolAddress while that device is current, and that address is what the
// kernels receive.
static __device__ __align__(256) uint8_t g_kvq_static_workspace[KVQ_STATIC_WORKSPACE_BYTES];

namespace {
void* g_static_ws_addr[kMaxDevices] = {nullptr};
std::mutex g_static_ws_mutex;
}  // namespace

extern "C" kvq_status kvq_decode_attn_noalloc(const kvq_cache* cache, const kvq_cache* prefix, int32_t prefix_len,
                                              const void* q, int32_t q_dtype, int32_t batch, int32_t num_q_heads,
                                              const int32_t* block_table, int32_t max_pages_per_seq,
                                              const int32_t* seq_lens, float sm_scale, const kvq_meter_params* mp,
                                              float* out, float* meter_state, int32_t* err_word, kvq_stream_t stream) {
  if (!cache || cache->num_kv_heads <= 0) return KVQ_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVQ_ERR_CUDA;
  void* ws = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_static_ws_mutex);
    if (!g_static_ws_addr[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_kvq_static_workspace) != cudaSuccess || !p) return KVQ_ERR_CUDA;
      g_static_ws_addr[dev] = p;
    }
    ws = g_static_ws_addr[dev];
  }
  if (batch > 0) {
    const size_t need = kvq_decode_workspace_size(batch, cache->num_kv_heads, num_q_heads);
    if (need == 0) return KVQ_ERR_INVALID_ARG;
    if (need > KVQ_STATIC_WORKSPACE_BYTES) return KVQ_ERR_WORKSPACE_TOO_SMALL;
  }
  return kvq_decode_attn(cache, prefix, prefix_len, q, q_dtype, batch, num_q_heads, block_table, max_pages_per_seq,
                         seq_lens, sm_scale, mp, out, meter_state, ws, KVQ_STATIC_WORKSPACE_BYTES, err_word, stream);
}

// ------------------------------------------------------------------------------------------------
// Test hook: the decode kernel's bounded mbarrier wait on a barrier that nothing completes.
namespace kvq {
namespace dec {
__global__ void wait_timeout_kernel(unsigned long long limit_ns, int32_t* err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncwarp();
  if (!__all_sync(kFull, mbar_wait(&bar, 0, limit_ns)) && threadIdx.x == 0) report(err, KVQ_ERR_TIMEOUT);
}
}  // namespace dec
}  // namespace kvq

extern "C" kvq_status kvq_debug_wait_timeout(uint64_t limit_ns, int32_t* err_word, kvq_stream_t stream) {
  if (!err_word || limit_ns > 2000000000ull) return KVQ_ERR_INVALID_ARG;
  kvq::dec::wait_timeout_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(limit_ns, err_word);
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}
