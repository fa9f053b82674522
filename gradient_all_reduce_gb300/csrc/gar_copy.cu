// k_copy instantiations and launch (all-gather, broadcast).
#include <algorithm>
#include <mutex>
#include <unordered_map>

#include "gar_launch.h"

namespace gar {

cudaError_t resident_ctas(const void* func, int threads, size_t smem, int* per_sm) {
  // The dynamic shared-memory opt-in is an attribute of the function in the
  // current device's context: it is set on every call (a host-side call
  // that allocates nothing), so a second device, or a context created anew
  // after cudaDeviceReset, gets it too.  Occupancy is cached per device.
  if (smem > 0) {
    const cudaError_t e =
        cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) {
      cudaGetLastError();
      return e;
    }
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return cudaErrorInvalidDevice;
  }
  struct Key {
    int dev;
    const void* func;
    int threads;
    size_t smem;
    bool operator==(const Key& o) const {
      return dev == o.dev && func == o.func && threads == o.threads && smem == o.smem;
    }
  };
  struct Hash {
    size_t operator()(const Key& k) const {
      return std::hash<const void*>()(k.func) ^ (size_t(k.dev) << 1) ^ (k.smem << 7) ^
             (size_t(k.threads) << 3);
    }
  };
  static std::mutex mu;
  static std::unordered_map<Key, int, Hash> cache;
  const Key key{dev, func, threads, smem};
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) {
      *per_sm = it->second;
      return cudaSuccess;
    }
  }
  int n = 0;
  const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, func, threads, smem);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return e;
  }
  if (n < 1) return cudaErrorInvalidConfiguration;  // the kernel cannot run with this much
  std::lock_guard<std::mutex> lock(mu);
  cache[key] = n;
  *per_sm = n;
  return cudaSuccess;
}

template <class Cap>
cudaError_t launch_copy(const LaunchCtx& ctx, const SegTable<Cap>& tab) {
  if (ctx.tma) {
    auto* k = &k_copy_tma<Cap>;
    const size_t smem = size_t(kCopyTmaStages) * kCopyTmaTile;
    int per_sm = 0;
    const cudaError_t e = resident_ctas(reinterpret_cast<const void*>(k), 32, smem, &per_sm);
    if (e != cudaSuccess) return e;
    const unsigned grid = grid_for(tab.ntiles, per_sm * ctx.num_sms);
    if (grid == 0) return cudaSuccess;
    return launch_ex(ctx, k, grid, 32, smem, tab);
  }
  // A copy of at least kCopyWindowBytes runs by destination groups in
  // windows (a.dgroup destinations per item, see k_copy): the most
  // destinations of any segment travels in ndst (the bulk-store kernel
  // reads each segment's own count instead).  a.dgroup = 0 keeps ndst = 0:
  // one CTA per tile, every destination.
  // tab.unroll = 1 or 2: a copy below kCopyWindowBytes, cut into tiles of
  // that many vectors per thread (copy_unroll_for) and always in the classic
  // order.
  if (tab.unroll == 1 || tab.unroll == 2) {
    SegTable<Cap> t = tab;
    t.ndst = 0;
    const unsigned grid = grid_per_tile(t.ntiles);
    if (grid == 0) return cudaSuccess;
    return tab.unroll == 1 ? launch_ex(ctx, &k_copy<Cap, 1>, grid, kThreads, 0, t)
                           : launch_ex(ctx, &k_copy<Cap, 2>, grid, kThreads, 0, t);
  }
  SegTable<Cap> t = tab;
  t.ndst = 0;
  uint64_t items = t.ntiles;
  if (t.dgroup > 0) {
    for (uint32_t s = 0; s < t.nseg; ++s) t.ndst = std::max(t.ndst, int(t.flags[s] >> 8));
    const uint64_t groups = (uint64_t(t.ndst) + t.dgroup - 1) / uint64_t(t.dgroup);
    items = (uint64_t(t.ntiles) + kCopyWindow - 1) / kCopyWindow * kCopyWindow * groups;
  }
  const unsigned grid = items < 0x7FFFFFFFull ? unsigned(items) : 0x7FFFFFFFu;
  if (grid == 0) return cudaSuccess;
  return launch_ex(ctx, &k_copy<Cap, kCopyUnroll>, grid, kThreads, 0, t);
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

// Synchronized batch-norm statistics: for each channel, the ranks' fp32
// sums and sums of squares pooled in fp64 in rank order, then mean, biased
// variance and invstd = 1 / sqrt(var + eps) with IEEE-rounded fp64
// operations, written rounded to fp32 to every rank.
//
// The call is latency-bound: a few KB of inputs, and per channel a chain of
// dependent fp64 operations.  On GB300 every fp64 warp instruction takes
// about 64 cycles whatever the number of active lanes, and an SM issues one
// every 19 cycles for all its warps, so the kernel keeps the fp64 work per
// channel short and spreads the channels thin:
// - one lane per channel, so a warp instruction serves 32 channels, and
//   one-warp CTAs, so the warps spread over the SMs (with a group of lanes
//   per channel running the same chain, the SMs' fp64 units were the
//   bottleneck);
// - the two divisions by the pooled count by Markstein's correction with
//   the host's RN(1/n) (div_count: five dependent fp64 operations against
//   the IEEE division's ~560 cycles).
// The rank-ordered adds, the square root and the reciprocal are the IEEE
// operations.  The kernel is specialised on the rank count NP.
constexpr int kSyncBnThreads = 32;

template <int NP>
__global__ void __launch_bounds__(kSyncBnThreads) k_syncbn_stats(const __grid_constant__ SyncBnArgs a) {
  griddep_launch_dependents();
  GAR_CHECK(a.np == NP, a.status);
  const uint64_t stride = uint64_t(gridDim.x) * blockDim.x;
  uint64_t c = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  griddep_wait();
  for (; c < a.channels; c += stride) {
    float x1[NP], x2[NP];
#pragma unroll
    for (int r = 0; r < NP; ++r) {
      x1[r] = __ldg(a.sum[r] + c);
      x2[r] = __ldg(a.sqsum[r] + c);
    }
    double s1 = double(x1[0]), s2 = double(x2[0]);
#pragma unroll
    for (int r = 1; r < NP; ++r) {
      s1 = __dadd_rn(s1, double(x1[r]));
      s2 = __dadd_rn(s2, double(x2[r]));
    }
    const double m = div_count(s1, a.n, a.rn);
    const double var = __dsub_rn(div_count(s2, a.n, a.rn), __dmul_rn(m, m));
    // 1 / sqrt(var + eps): the correctly rounded reciprocal is the IEEE
    // quotient 1 / x, by a shorter sequence than the general division.
    const double is = __drcp_rn(__dsqrt_rn(__dadd_rn(var, a.eps)));
    const float mf = __double2float_rn(m), isf = __double2float_rn(is);
#pragma unroll
    for (int r = 0; r < NP; ++r) {
      a.mean[r][c] = mf;
      a.invstd[r][c] = isf;
    }
  }
}

template <int NP>
static cudaError_t launch_syncbn_np(const LaunchCtx& ctx, const SyncBnArgs& args) {
  if (args.np != NP) return launch_syncbn_np<NP - 1>(ctx, args);
  const uint64_t blocks = (args.channels + kSyncBnThreads - 1) / kSyncBnThreads;
  const uint64_t cap = uint64_t(ctx.num_sms) * 16;
  const unsigned grid = unsigned(blocks < cap ? blocks : cap);
  if (grid == 0) return cudaSuccess;
  return launch_ex(ctx, &k_syncbn_stats<NP>, grid, kSyncBnThreads, 0, args);
}
template <>
cudaError_t launch_syncbn_np<0>(const LaunchCtx&, const SyncBnArgs&) {
  return cudaErrorInvalidValue;
}

cudaError_t launch_syncbn_stats(const LaunchCtx& ctx, const SyncBnArgs& args) {
  if (args.np < 1 || args.np > kMaxRanks) return cudaErrorInvalidValue;
  return launch_syncbn_np<kMaxRanks>(ctx, args);
}

template cudaError_t launch_copy<CapSmall>(const LaunchCtx&, const SegTable<CapSmall>&);
template cudaError_t launch_copy<CapLarge>(const LaunchCtx&, const SegTable<CapLarge>&);

}  // namespace gar
