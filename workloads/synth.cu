// synth.cu -- device-side copy of the seeded input generators of
// workloads/__init__.py (SplitMix64 in counter form; U(-1,1); the
// Irwin-Hall(4) bell-shaped draw; bf16 by truncation).  It exists so that
// multi-gigabyte synthetic replicas can be made in HBM directly; the host
// generator produces the same bits for any element.  It holds none of the
// collective's arithmetic.
#include <cstdint>
#include <cuda_runtime.h>

namespace {

constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ull;

__device__ __forceinline__ uint64_t splitmix64(uint64_t seed, uint64_t i) {
  uint64_t z = seed + (i + 1) * kGolden;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// kind 0: U(-1,1) = (z >> 40) * 2^-23 - 1 (exact in fp32).
// kind 1: (sum of the four 16-bit fields of z - 131070) * scale, in fp64,
//         then rounded once to fp32.
__global__ void k_fill(void* out, uint64_t n, uint64_t seed, uint64_t start, int kind, int bf16,
                       double scale) {
  const uint64_t stride = uint64_t(gridDim.x) * blockDim.x;
  for (uint64_t i = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
    const uint64_t z = splitmix64(seed, start + i);
    float f;
    if (kind == 0) {
      f = float(double(z >> 40) * 0x1p-23 - 1.0);
    } else {
      const int64_t s = int64_t(z & 0xFFFF) + int64_t((z >> 16) & 0xFFFF) +
                        int64_t((z >> 32) & 0xFFFF) + int64_t(z >> 48) - 131070;
      f = __double2float_rn(__dmul_rn(double(s), scale));
    }
    if (bf16)
      static_cast<uint16_t*>(out)[i] = uint16_t(__float_as_uint(f) >> 16);
    else
      static_cast<float*>(out)[i] = f;
  }
}

}  // namespace

extern "C" int synth_fill(void* out, uint64_t n, uint64_t seed, uint64_t start, int kind, int bf16,
                          double scale, void* stream) {
  if (n == 0) return 0;
  if (out == nullptr || (kind != 0 && kind != 1)) return 1;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  uint64_t blocks = (n + 255) / 256;
  const uint64_t cap = uint64_t(sms > 0 ? sms : 1) * 8;
  if (blocks > cap) blocks = cap;
  k_fill<<<unsigned(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(out, n, seed, start, kind,
                                                                          bf16, scale);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}
