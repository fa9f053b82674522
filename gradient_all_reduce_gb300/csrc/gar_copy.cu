// k_copy instantiations and launch (all-gather, broadcast).
#include <algorithm>
#include <mutex>
#include <unordered_map>

#include "gar_launch.h"

namespace gar {

int resident_ctas(const void* func, int threads, size_t smem) {
  static std::mutex mu;
  static std::unordered_map<const void*, std::pair<size_t, int>> cache;
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(func);
  if (it != cache.end() && it->second.first >= smem) return it->second.second;
  if (smem > 0) cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, func, threads, smem) != cudaSuccess || n < 1) {
    cudaGetLastError();
    n = 1;
  }
  cache[func] = {smem, n};
  return n;
}

template <class Cap>
cudaError_t launch_copy(const LaunchCtx& ctx, const SegTable<Cap>& tab) {
  if (ctx.tma) {
    auto* k = &k_copy_tma<Cap>;
    const size_t smem = size_t(kCopyTmaStages) * kCopyTmaTile;
    const int per_sm = resident_ctas(reinterpret_cast<const void*>(k), 32, smem);
    const unsigned grid = grid_for(tab.ntiles, per_sm * ctx.num_sms);
    if (grid == 0) return cudaSuccess;
    return launch_ex(ctx, k, grid, 32, smem, tab);
  }
  // A large copy from one source (a broadcast) runs destination by
  // destination in windows: the destination count travels in ndst (the
  // bulk-store kernel reads each segment's own count instead).  Everything
  // else keeps ndst = 0: one CTA per tile, every destination.
  SegTable<Cap> t = tab;
  t.ndst = 0;
  uint64_t items = t.ntiles;
  if (t.nseg == 1 && t.ntiles >= kCopyWindowMin) {
    for (uint32_t s = 0; s < t.nseg; ++s) t.ndst = std::max(t.ndst, int(t.flags[s] >> 8));
    items = (uint64_t(t.ntiles) + kCopyWindow - 1) / kCopyWindow * kCopyWindow * uint64_t(t.ndst);
  }
  const unsigned grid = items < 0x7FFFFFFFull ? unsigned(items) : 0x7FFFFFFFu;
  if (grid == 0) return cudaSuccess;
  return launch_ex(ctx, &k_copy<Cap>, grid, kThreads, 0, t);
}

__global__ void k_wait_selftest(uint32_t* status, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const bool ok = mbar_wait_bounded(smem_u32(&bar), 0, &abort_flag, limit_ns);
  if (!__all_sync(0xFFFFFFFFu, ok) && threadIdx.x == 0) atomicExch(status, 1u);
}

cudaError_t launch_wait_selftest(cudaStream_t stream, uint32_t* status, uint64_t limit_ns) {
  k_wait_selftest<<<1, 32, 0, stream>>>(status, limit_ns);
  return cudaGetLastError();
}

// Synchronized batch-norm statistics: one thread per channel pools the
// ranks' per-channel sums in fp64 (rank order), forms mean, biased
// variance and invstd with IEEE-rounded fp64 operations, and writes both,
// rounded to fp32, for every rank.
// One warp per CTA: the fp64 divide and square root are long dependent
// chains, so the channels are spread over as many SMs as possible.
constexpr int kSyncBnThreads = 32;

__global__ void __launch_bounds__(kSyncBnThreads) k_syncbn_stats(const __grid_constant__ SyncBnArgs a) {
  griddep_launch_dependents();
  griddep_wait();
  const uint64_t stride = uint64_t(gridDim.x) * blockDim.x;
  for (uint64_t c = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x; c < a.channels; c += stride) {
    double s1 = double(a.sum[0][c]), s2 = double(a.sqsum[0][c]);
    for (int r = 1; r < a.np; ++r) {
      s1 = __dadd_rn(s1, double(a.sum[r][c]));
      s2 = __dadd_rn(s2, double(a.sqsum[r][c]));
    }
    const double m = __ddiv_rn(s1, a.n);
    const double var = __dsub_rn(__ddiv_rn(s2, a.n), __dmul_rn(m, m));
    const double is = __ddiv_rn(1.0, __dsqrt_rn(__dadd_rn(var, a.eps)));
    const float mf = __double2float_rn(m), isf = __double2float_rn(is);
    for (int r = 0; r < a.np; ++r) {
      a.mean[r][c] = mf;
      a.invstd[r][c] = isf;
    }
  }
}

cudaError_t launch_syncbn_stats(const LaunchCtx& ctx, const SyncBnArgs& args) {
  const uint64_t blocks = (args.channels + kSyncBnThreads - 1) / kSyncBnThreads;
  const uint64_t cap = uint64_t(ctx.num_sms) * 16;
  const unsigned grid = unsigned(blocks < cap ? blocks : cap);
  if (grid == 0) return cudaSuccess;
  return launch_ex(ctx, &k_syncbn_stats, grid, kSyncBnThreads, 0, args);
}

template cudaError_t launch_copy<CapSmall>(const LaunchCtx&, const SegTable<CapSmall>&);
template cudaError_t launch_copy<CapLarge>(const LaunchCtx&, const SegTable<CapLarge>&);

}  // namespace gar
