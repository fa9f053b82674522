// Exhaustive check of the kernels' division by a small integer rank count
// against the IEEE division __fdiv_rn: every fp32 bit pattern x, for one
// divisor d per call.  Mode 0 checks gar::div_small (Markstein's
// correction) bit for bit; mode 1 checks that gar::div_small_bf16 rounds to
// the same bf16 as the IEEE quotient.  Built by tests/test_gpu_division.py
// against the library's own device header.
#include <cstdint>
#include <cuda_runtime.h>

#include "gar_device.cuh"

__global__ void k_div_check(float d, int mode, unsigned long long* bad, unsigned int* first) {
  const float r = __frcp_rn(d);
  const uint64_t stride = uint64_t(gridDim.x) * blockDim.x;
  unsigned long long local = 0;
  for (uint64_t i = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < (1ull << 32); i += stride) {
    const float x = __uint_as_float(uint32_t(i));
    const float b = __fdiv_rn(x, d);
    bool same;
    if (mode == 0) {
      const float a = gar::div_small(x, d, r);
      same = __float_as_uint(a) == __float_as_uint(b) || ((a != a) && (b != b));
    } else {
      const float a = gar::div_small_bf16(x, d, r);
      same = gar::bf16_rne(a) == gar::bf16_rne(b) || ((a != a) && (b != b));
    }
    if (!same) {
      ++local;
      atomicMin(first, uint32_t(i));
    }
  }
  if (local) atomicAdd(bad, local);
}

// Returns 0 on success (mismatch count and first mismatching x in the
// outputs), -1 on a CUDA error.
extern "C" int div_check(int d, int mode, unsigned long long* mismatches, unsigned int* first_x) {
  unsigned long long* bad = nullptr;
  unsigned int* first = nullptr;
  if (cudaMalloc(&bad, sizeof(*bad)) != cudaSuccess) return -1;
  if (cudaMalloc(&first, sizeof(*first)) != cudaSuccess) { cudaFree(bad); return -1; }
  int rc = 0;
  if (cudaMemset(bad, 0, sizeof(*bad)) != cudaSuccess ||
      cudaMemset(first, 0xff, sizeof(*first)) != cudaSuccess)
    rc = -1;
  if (rc == 0) {
    k_div_check<<<152 * 8, 256>>>(float(d), mode, bad, first);
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpy(mismatches, bad, sizeof(*bad), cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(first_x, first, sizeof(*first), cudaMemcpyDeviceToHost) != cudaSuccess)
      rc = -1;
  }
  cudaFree(bad);
  cudaFree(first);
  return rc;
}
