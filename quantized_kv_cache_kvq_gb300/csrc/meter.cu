// meter.cu -- meter finalisation and device telemetry (kvq_meter), status strings.
//
// WitCert (arXiv 2607.28699) Sec. 4.3: the sound meter is min(1, 1/2 (A^2 - 1)); above saturation
// the raw value is a risk score (certified gating at tau < 1, risk-ranked gating at tau >= 1).
// Sec. 6.2.4 ("Certificate telemetry in production"): reduce certificates on the GPU without a host
// synchronisation per layer, and count non-finite values separately from the finite statistics.
// Sec. 3: the output moves by at most 2 TV max_t ||v_t|| + sum_t p~_t rho^v_t; with the meter for TV
// that is the output-error bound 2 meter Vmax + R.  Sec. 4.3 Prop. 1: TV <= 1/2 (A/A^- - A^-/A), and
// neither this nor 1/2 (A^2 - 1) dominates, so the two-sided meter is the minimum; the det-tanh shape
// TV <= tanh(max |eps|) uses the largest radius.
#include <cmath>

#include "kvq_common.cuh"

namespace kvq {
namespace {

constexpr float kLn2 = 0.69314718055994531f;
constexpr int kMaxRankCells = 8192;

// meter = min(1, 1/2 (A-1)(A+1)) and raw = ln(1/2 (A^2 - 1)) from la = ln(A - 1)
__device__ __forceinline__ void finalize_one(float la, float& meter, float& raw) {
  if (isnan(la)) { meter = NAN; raw = NAN; return; }
  if (la == -INFINITY) { meter = 0.f; raw = -INFINITY; return; }
  // ln(A + 1) = ln(2 + e^la)
  const float lap1 = la < 0.f ? kLn2 + log1pf(0.5f * expf(la)) : la + log1pf(2.f * expf(-la));
  raw = la + lap1 - kLn2;
  if (la > 1.f) { meter = 1.f; return; }
  const float am1 = expf(la);
  meter = fminf(1.f, 0.5f * am1 * (am1 + 2.f));
}

__global__ void __launch_bounds__(256) finalize_kernel(const float* __restrict__ state, long long n, float tau,
                                                       float* __restrict__ meter_a, float* __restrict__ raw_a,
                                                       float* __restrict__ cert_b, float* __restrict__ out_bound,
                                                       float* __restrict__ two_sided, float* __restrict__ det_tanh,
                                                       int32_t* __restrict__ counts) {
  int cov_a = 0, cov_b = 0, nonfinite = 0, cells = 0;
  static_assert(KVQ_METER_STATE_FLOATS == 8, "two float4 per cell");
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const float4 s = reinterpret_cast<const float4*>(state)[2 * i];
    float m, r;
    finalize_one(s.x, m, r);
    meter_a[i] = m;
    raw_a[i] = r;
    if (out_bound || two_sided || det_tanh) {
      const float4 v = reinterpret_cast<const float4*>(state)[2 * i + 1];  // (R, Vmax, max c, 1 - A^-)
      if (out_bound) out_bound[i] = (isnan(v.x) || isnan(m)) ? NAN : __fmaf_rn(2.f * m, v.y, v.x);
      if (det_tanh) det_tanh[i] = isnan(v.z) ? NAN : tanhf(v.z);
      if (two_sided) {
        float t = NAN;
        if (!isnan(v.w) && !isnan(m)) {
          t = m;
          if (s.x != -INFINITY && s.x < 80.f && v.w < 1.f) {
            // 1/2 (A/A^- - A^-/A) with x = A - 1 = e^{la}, y = 1 - A^-, free of cancellation:
            // A/A^- - A^-/A = (A - A^-)(A + A^-) / (A A^-) = (x + y)(2 + x - y) / ((1 + x)(1 - y))
            const float x = expf(s.x), y = v.w;
            t = fminf(t, 0.5f * ((x + y) * (2.f + x - y)) / ((1.f + x) * (1.f - y)));
          }
        }
        two_sided[i] = t;
      }
    }
    cells += 1;
    if (isnan(s.x) || s.x == INFINITY) nonfinite += 1;
    else if (m < tau) cov_a += 1;
    if (cert_b) {
      float mb, rb;
      finalize_one(s.y, mb, rb);
      cert_b[i] = mb;
      if (!isnan(mb) && mb < tau) cov_b += 1;
    }
  }
  // block reduction, then one atomic per counter per block
  __shared__ int red[4][8];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int v[4] = {cov_a, cov_b, nonfinite, cells};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v[k] += __shfl_xor_sync(0xffffffffu, v[k], o);
    if (lane == 0) red[k][warp] = v[k];
  }
  __syncthreads();
  if (threadIdx.x < 4) {
    int t = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += red[threadIdx.x][w];
    if (t) atomicAdd(&counts[threadIdx.x], t);
  }
}

// Rank the L*H cells of one request by raw score (highest first, ties to the lower flat index).
__global__ void __launch_bounds__(512) rank_kernel(const float* __restrict__ raw_a, int n_layers, int batch, int hq,
                                                   int32_t* __restrict__ ranking) {
  __shared__ float key[kMaxRankCells];
  const int b = blockIdx.x;
  const int n = n_layers * hq;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int l = i / hq, h = i % hq;
    const float r = raw_a[(static_cast<size_t>(l) * batch + b) * hq + h];
    key[i] = isnan(r) ? INFINITY : r;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const float ki = key[i];
    int rank = 0;
    for (int j = 0; j < n; ++j) {
      const float kj = key[j];
      rank += (kj > ki) || (kj == ki && j < i);
    }
    ranking[static_cast<size_t>(b) * n + rank] = i;
  }
}

constexpr int kMaxGatePages = 16384;

// Float-float sums (an unevaluated pair hi + lo of binary32 numbers, Knuth's TwoSum): prefix sums of up to
// 16384 contributions to ~2^-44 relative with FP32 arithmetic only (double precision is slow on this part).
struct FF {
  float hi, lo;
};
__device__ __forceinline__ FF ff_add(FF a, FF b) {
  const float s = a.hi + b.hi;
  const float bb = s - a.hi;
  const float e = ((a.hi - (s - bb)) + (b.hi - bb)) + (a.lo + b.lo);
  const float h = s + e;
  return FF{h, e - (h - s)};
}

// Greedy block page-in (WitCert Sec. 6.3.5): one block per (sequence, query head) cell.  A cell whose
// meter is already within tau gets the empty plan at once.  The plan is the first k with
// (A - 1) - S_k <= target = sqrt(1 + 2 tau) - 1, S_k the sum of the k largest page contributions
// exp(lc - lse) (descending, ties to the lower page index; all P pages when no k reaches the target).
// Short plans (the usual case) take the largest remaining page up to kGateQuick times by a block arg-max
// and sum in float-float; longer ones (known as soon as the deficit exceeds the largest contribution
// left times the rounds left) sort all pages in shared memory (bitonic) and scan the prefix sums
// (per-thread chunks, then a block scan).
constexpr int kGateThreads = 512;
constexpr int kGateQuick = 16;
__global__ void __launch_bounds__(kGateThreads) gate_kernel(const float* __restrict__ lc, int stride,
                                                            const float* __restrict__ state, int hq,
                                                            const int32_t* __restrict__ seq_lens, int prefix_pages,
                                                            float target, int32_t* __restrict__ n_out,
                                                            int32_t* __restrict__ list, int max_list) {
  extern __shared__ __align__(16) float key[];
  __shared__ FF wsum[kGateThreads / 32];
  __shared__ float wv[kGateThreads / 32];
  __shared__ int wi[kGateThreads / 32], quick[kGateQuick];
  __shared__ int k_shared;
  const int cell = blockIdx.x, seq = cell / hq;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int len = max(seq_lens[seq], 0);
  const int P = min(min(prefix_pages + (len + 15) / 16, kMaxGatePages), stride);  // never past the row
  const float la = state[static_cast<size_t>(cell) * KVQ_METER_STATE_FLOATS];
  const float am1 = la == -INFINITY ? 0.f : expf(la);
  if (!(am1 > target) || P == 0) {  // already within tau (or nothing to page in): the empty plan
    if (threadIdx.x == 0) n_out[cell] = 0;
    if (list)
      for (int i = threadIdx.x; i < max_list; i += blockDim.x) list[static_cast<size_t>(cell) * max_list + i] = -1;
    return;
  }
  int n2 = 1;
  while (n2 < P) n2 <<= 1;
  int* idx = reinterpret_cast<int*>(key + n2);
  const float lse = state[static_cast<size_t>(cell) * KVQ_METER_STATE_FLOATS + 2];
  for (int i = threadIdx.x; i < n2; i += blockDim.x) {
    float k = -1.f;  // padding sorts last
    if (i < P) {
      const float v = lc[static_cast<size_t>(cell) * stride + i];
      k = v == -INFINITY ? 0.f : expf(v - lse);
      if (!(k >= 0.f)) k = 0.f;  // NaN (non-finite inputs, reported by the decode): no contribution
    }
    key[i] = k;
    idx[i] = i;
  }
  if (threadIdx.x == 0) k_shared = P;
  __syncthreads();
  {
    // short plans: repeated arg-max over the pages not yet taken (each thread reads only its own pages)
    FF S{0.f, 0.f};
    for (int k = 0; k < min(P, kGateQuick); ++k) {
      float bv = -1.f;
      int bi = 0x7fffffff;
      for (int i = threadIdx.x; i < P; i += blockDim.x) {
        const float v = key[i];
        if (v > bv) { bv = v; bi = i; }  // ascending i: ties keep the lower index
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
      }
      if (lane == 0) { wv[warp] = bv; wi[warp] = bi; }
      __syncthreads();
      bv = wv[0];
      bi = wi[0];
      for (int w = 1; w < static_cast<int>(blockDim.x >> 5); ++w)
        if (wv[w] > bv || (wv[w] == bv && wi[w] < bi)) { bv = wv[w]; bi = wi[w]; }
      __syncthreads();  // every warp has read wv / wi before the next round writes them
      if (bi >= P) break;  // no page left to take (cannot happen with finite keys): the sort path decides
      if (threadIdx.x == static_cast<unsigned>(bi) % blockDim.x) key[bi] = -1.f;  // taken (its owner's page)
      if (threadIdx.x == 0) quick[k] = bi;
      S = ff_add(S, FF{bv, 0.f});
      if ((am1 - S.hi) - S.lo <= target || k + 1 == P) {  // uniform: every thread holds the same S
        __syncthreads();
        const int n = k + 1;
        if (threadIdx.x == 0) n_out[cell] = n;
        if (list)
          for (int i = threadIdx.x; i < max_list; i += blockDim.x)
            list[static_cast<size_t>(cell) * max_list + i] = i < n ? quick[i] : -1;
        return;
      }
      // every page left contributes at most bv: when the deficit exceeds what the rounds left can remove,
      // the plan is longer than kGateQuick pages; sort at once (the sort computes the same plan)
      if ((am1 - S.hi) - S.lo - target > static_cast<float>(kGateQuick - k - 1) * bv) break;
    }
  }
  // a longer plan: start again from all pages and sort them
  for (int i = threadIdx.x; i < P; i += blockDim.x) {
    const float v = lc[static_cast<size_t>(cell) * stride + i];
    const float k = v == -INFINITY ? 0.f : expf(v - lse);
    key[i] = k >= 0.f ? k : 0.f;
  }
  __syncthreads();
  auto before = [&](int a, int b) { return key[a] > key[b] || (key[a] == key[b] && idx[a] < idx[b]); };
  for (int size = 2; size <= n2; size <<= 1) {
    for (int half = size >> 1; half > 0; half >>= 1) {
      for (int i = threadIdx.x; i < n2; i += blockDim.x) {
        const int j = i ^ half;
        if (j > i && ((i & size) == 0 ? before(j, i) : before(i, j))) {
          const float tk = key[i]; key[i] = key[j]; key[j] = tk;
          const int ti = idx[i]; idx[i] = idx[j]; idx[j] = ti;
        }
      }
      __syncthreads();
    }
  }
  // thread t owns sorted positions [b0, b1); its exclusive prefix comes from a block scan of chunk sums
  const int per = (P + blockDim.x - 1) / blockDim.x;
  const int b0 = min(P, static_cast<int>(threadIdx.x) * per), b1 = min(P, b0 + per);
  FF part{0.f, 0.f};
  for (int i = b0; i < b1; ++i) part = ff_add(part, FF{key[i], 0.f});
  FF incl = part;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const FF t{__shfl_up_sync(0xffffffffu, incl.hi, o), __shfl_up_sync(0xffffffffu, incl.lo, o)};
    if (lane >= o) incl = ff_add(t, incl);
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  FF S{__shfl_up_sync(0xffffffffu, incl.hi, 1), __shfl_up_sync(0xffffffffu, incl.lo, 1)};  // lanes before this one
  if (lane == 0) S = FF{0.f, 0.f};
  for (int w = 0; w < warp; ++w) S = ff_add(wsum[w], S);
  for (int k = b0; k < b1; ++k) {  // the first k (pages 0..k-1 taken) that reaches the target
    if ((am1 - S.hi) - S.lo <= target) { atomicMin(&k_shared, k); break; }
    S = ff_add(S, FF{key[k], 0.f});
  }
  __syncthreads();
  const int k = k_shared;
  if (threadIdx.x == 0) n_out[cell] = k;
  if (list)
    for (int i = threadIdx.x; i < max_list; i += blockDim.x)
      list[static_cast<size_t>(cell) * max_list + i] = i < k ? idx[i] : -1;
}

}  // namespace
}  // namespace kvq

using namespace kvq;

extern "C" kvq_status kvq_gate(const float* lc, int32_t stride, const float* state, int32_t batch, int32_t hq,
                               const int32_t* seq_lens, int32_t prefix_len, float tau, int32_t* n_page_in,
                               int32_t* page_list, int32_t max_list, kvq_stream_t stream) {
  if (batch < 0 || hq <= 0 || prefix_len < 0 || stride <= 0 || !(tau >= 0.f) || max_list < 0) return KVQ_ERR_INVALID_ARG;
  if (batch == 0) return KVQ_OK;
  if (!lc || !state || !seq_lens || !n_page_in || (page_list && max_list == 0)) return KVQ_ERR_INVALID_ARG;
  static bool configured[kMaxDevices] = {};  // the limit is a setting of each device's context
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KVQ_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices || !configured[dev]) {
    if (cudaFuncSetAttribute(gate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxGatePages * 8) !=
        cudaSuccess)
      return KVQ_ERR_CUDA;
    if (dev >= 0 && dev < kMaxDevices) configured[dev] = true;
  }
  // keys and indices of the largest row a cell can have (a row holds at most `stride` pages)
  int n2 = 1;
  while (n2 < stride && n2 < kMaxGatePages) n2 <<= 1;
  const int smem = n2 * 8;
  const int prefix_pages = (prefix_len + 15) / 16;
  const float target = static_cast<float>(std::sqrt(1.0 + 2.0 * static_cast<double>(tau)) - 1.0);  // meter <= tau
  gate_kernel<<<static_cast<unsigned>(static_cast<long long>(batch) * hq), kGateThreads, smem,
                reinterpret_cast<cudaStream_t>(stream)>>>(lc, stride, state, hq, seq_lens, prefix_pages, target, n_page_in,
                                                           page_list, max_list);
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

extern "C" kvq_status kvq_meter(const float* state, int32_t n_layers, int32_t batch, int32_t hq,
                                const kvq_meter_params* mp, float* meter_a, float* raw_a, float* cert_b,
                                float* out_bound, float* two_sided, float* det_tanh, int32_t* counts, int32_t* ranking,
                                kvq_stream_t stream) {
  if (!mp || n_layers < 0 || batch < 0 || hq <= 0) return KVQ_ERR_INVALID_ARG;
  if (!state || !meter_a || !raw_a || !counts) return KVQ_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(state) & 15u) != 0) return KVQ_ERR_INVALID_ARG;
  if (ranking && static_cast<long long>(n_layers) * hq > kMaxRankCells) return KVQ_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(counts, 0, 4 * sizeof(int32_t), s) != cudaSuccess) return KVQ_ERR_CUDA;
  const long long n = static_cast<long long>(n_layers) * batch * hq;
  if (n == 0) return KVQ_OK;
  long long blocks = (n + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  finalize_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(state, n, mp->tau, meter_a, raw_a, cert_b, out_bound,
                                                                two_sided, det_tanh, counts);
  if (cudaGetLastError() != cudaSuccess) return KVQ_ERR_CUDA;
  if (ranking) {
    rank_kernel<<<batch, 512, 0, s>>>(raw_a, n_layers, batch, hq, ranking);
    if (cudaGetLastError() != cudaSuccess) return KVQ_ERR_CUDA;
  }
  return KVQ_OK;
}

extern "C" const char* kvq_status_string(int32_t status) {
  switch (status) {
    case KVQ_OK: return "KVQ_OK";
    case KVQ_ERR_INVALID_ARG: return "KVQ_ERR_INVALID_ARG";
    case KVQ_ERR_UNSUPPORTED_LAYOUT: return "KVQ_ERR_UNSUPPORTED_LAYOUT";
    case KVQ_ERR_WORKSPACE_TOO_SMALL: return "KVQ_ERR_WORKSPACE_TOO_SMALL";
    case KVQ_ERR_CUDA: return "KVQ_ERR_CUDA";
    case KVQ_ERR_DEVICE_BOUNDS: return "KVQ_ERR_DEVICE_BOUNDS";
    case KVQ_ERR_NONFINITE_INPUT: return "KVQ_ERR_NONFINITE_INPUT";
    case KVQ_ERR_RANGE: return "KVQ_ERR_RANGE";
    case KVQ_ERR_TIMEOUT: return "KVQ_ERR_TIMEOUT";
  }
  return "KVQ_ERR_UNKNOWN";
}

extern "C" int32_t kvq_version(void) { return KVQ_VERSION; }
