// GPU check of the SyncBN statistics' division by the pooled count,
// gar::div_count, against the IEEE division __ddiv_rn.  Built by
// tests/test_gpu_syncbn_arith.py against the library's own device header;
// the cases come from a counter-based hash.
#include <cstdint>
#include <cuda_runtime.h>

#include "gar_device.cuh"

namespace {

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z += 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ bool same_bits(double a, double b) {
  return __double_as_longlong(a) == __double_as_longlong(b) || (a != a && b != b);
}

// A double with a random sign, 52 random fraction bits and an unbiased
// exponent in [lo, hi].
__device__ __forceinline__ double random_double(uint64_t h, uint64_t g, int lo, int hi) {
  const int e = lo + int(g % uint64_t(hi - lo + 1));
  const uint64_t bits = (h & 0x800FFFFFFFFFFFFFull) | (uint64_t(e + 1023) << 52);
  return __longlong_as_double(static_cast<long long>(bits));
}

// mode 0: s a random double in the range of the sums, n a count with a
// random bit length of 1 to 53.  mode 1: s chosen so that s / n lies next
// to the midpoint between two neighbouring doubles (the hard cases of
// rounding), then moved by up to two units either way.
__global__ void k_div_count(uint64_t seed, uint64_t cases, int mode, unsigned long long* bad,
                            unsigned long long* first) {
  const uint64_t stride = uint64_t(gridDim.x) * blockDim.x;
  unsigned long long local = 0;
  for (uint64_t i = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < cases; i += stride) {
    const uint64_t h0 = mix64(seed ^ (4 * i)), h1 = mix64(seed ^ (4 * i + 1));
    const uint64_t h2 = mix64(seed ^ (4 * i + 2)), h3 = mix64(seed ^ (4 * i + 3));
    const int nb = 1 + int(h0 % 53);
    const uint64_t nv = (h1 >> (64 - nb)) | (uint64_t(1) << (nb - 1));
    const double n = double(nv);
    double s;
    if (mode == 0) {
      s = random_double(h2, h3, -149, 132);
    } else {
      const double q = fabs(random_double(h2, h3, -149 + 53, 132 - 54));
      const double half = (__longlong_as_double(__double_as_longlong(q) + 1) - q) * 0.5;
      s = __fma_rn(q, n, half * n);
      const int k = int(h0 >> 60) % 5 - 2;
      s = __longlong_as_double(__double_as_longlong(s) + k);
      if (h1 & 1) s = -s;
    }
    const double y = __drcp_rn(n);
    if (!same_bits(gar::div_count(s, n, y), __ddiv_rn(s, n))) {
      ++local;
      atomicMin(first, static_cast<unsigned long long>(i));
    }
  }
  if (local) atomicAdd(bad, local);
}

int run(void (*launch)(unsigned long long*, unsigned long long*), unsigned long long* mismatches,
        unsigned long long* first_case) {
  unsigned long long *bad = nullptr, *first = nullptr;
  if (cudaMalloc(&bad, sizeof(*bad)) != cudaSuccess) return -1;
  if (cudaMalloc(&first, sizeof(*first)) != cudaSuccess) {
    cudaFree(bad);
    return -1;
  }
  int rc = 0;
  if (cudaMemset(bad, 0, sizeof(*bad)) != cudaSuccess ||
      cudaMemset(first, 0xff, sizeof(*first)) != cudaSuccess)
    rc = -1;
  if (rc == 0) {
    launch(bad, first);
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpy(mismatches, bad, sizeof(*bad), cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(first_case, first, sizeof(*first), cudaMemcpyDeviceToHost) != cudaSuccess)
      rc = -1;
  }
  cudaFree(bad);
  cudaFree(first);
  return rc;
}

uint64_t g_seed, g_cases;
int g_mode;

void launch_div(unsigned long long* bad, unsigned long long* first) {
  k_div_count<<<152 * 8, 256>>>(g_seed, g_cases, g_mode, bad, first);
}

}  // namespace

// 0 on success (mismatch count and first mismatching case in the outputs),
// -1 on a CUDA error.
extern "C" int div_count_check(unsigned long long seed, unsigned long long cases, int mode,
                               unsigned long long* mismatches, unsigned long long* first_case) {
  g_seed = seed;
  g_cases = cases;
  g_mode = mode;
  return run(launch_div, mismatches, first_case);
}
