// Test helper (not part of libkvq): the first four outputs of cuRAND's Philox4x32-10 device generator
// for (seed, subsequence, offset 0), used to pin the oracle's Philox to an implementation outside this
// repository.
#include <cuda_runtime.h>
#include <curand_kernel.h>

__global__ void philox_first4(unsigned long long seed, const unsigned long long* subseq, unsigned* out, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  curandStatePhilox4_32_10_t st;
  curand_init(seed, subseq[i], 0ull, &st);
  const uint4 r = curand4(&st);
  out[4 * i + 0] = r.x;
  out[4 * i + 1] = r.y;
  out[4 * i + 2] = r.z;
  out[4 * i + 3] = r.w;
}

extern "C" int curand_philox_first4(unsigned long long seed, const unsigned long long* subseq_host, int n,
                                    unsigned* out_host) {
  unsigned long long* d_s = nullptr;
  unsigned* d_o = nullptr;
  if (cudaMalloc(&d_s, sizeof(unsigned long long) * n) != cudaSuccess) return 1;
  if (cudaMalloc(&d_o, sizeof(unsigned) * 4 * n) != cudaSuccess) return 1;
  cudaMemcpy(d_s, subseq_host, sizeof(unsigned long long) * n, cudaMemcpyHostToDevice);
  philox_first4<<<(n + 127) / 128, 128>>>(seed, d_s, d_o, n);
  const cudaError_t e = cudaMemcpy(out_host, d_o, sizeof(unsigned) * 4 * n, cudaMemcpyDeviceToHost);
  cudaFree(d_s);
  cudaFree(d_o);
  return e == cudaSuccess ? 0 : 2;
}
