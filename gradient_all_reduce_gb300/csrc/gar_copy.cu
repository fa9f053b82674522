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
//
// The call is latency-bound: a few KB of inputs, and per channel a chain of
// about 70 fp64 instructions (conversions, adds, three divisions, a square
// root) on GB300's narrow fp64 pipe.  So the kernel is specialised on the
// rank count NP: a thread issues the loads of all 2 NP inputs before the
// first add, and executes exactly NP - 1 adds per sum (a loop to the
// largest rank count under a guard issued the guarded-off fp64
// instructions too).  The channels are spread over every SM sub-partition:
// each warp takes `lanes` channels (lane < lanes), so that up to
// 4 x SMs warps share the fp64 work, four to a CTA.
constexpr int kSyncBnThreads = 128;

template <int NP>
__global__ void __launch_bounds__(kSyncBnThreads) k_syncbn_stats(const __grid_constant__ SyncBnArgs a) {
  griddep_launch_dependents();
  griddep_wait();
  const uint32_t lane = threadIdx.x & 31u;
  if (lane >= a.lanes) return;
  const uint64_t warp = (uint64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const uint64_t stride = (uint64_t(gridDim.x) * blockDim.x >> 5) * a.lanes;
  GAR_CHECK(a.np == NP && a.lanes >= 1 && a.lanes <= 32, a.status);
  for (uint64_t c = warp * a.lanes + lane; c < a.channels; c += stride) {
    GAR_CHECK(c < a.channels, a.status);
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
    const double m = __ddiv_rn(s1, a.n);
    const double var = __dsub_rn(__ddiv_rn(s2, a.n), __dmul_rn(m, m));
    const double is = __ddiv_rn(1.0, __dsqrt_rn(__dadd_rn(var, a.eps)));
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
  SyncBnArgs a = args;
  // Channels per warp: as few as spread the channels over 4 warps per SM.
  const uint64_t warps_max = uint64_t(ctx.num_sms) * (kSyncBnThreads / 32);
  const uint64_t lanes = (a.channels + warps_max - 1) / warps_max;
  a.lanes = uint32_t(lanes < 1 ? 1 : (lanes > 32 ? 32 : lanes));
  const uint64_t warps = (a.channels + a.lanes - 1) / a.lanes;
  const uint64_t blocks = (warps + kSyncBnThreads / 32 - 1) / (kSyncBnThreads / 32);
  const unsigned grid = unsigned(blocks < warps_max ? blocks : warps_max);
  if (grid == 0) return cudaSuccess;
  return launch_ex(ctx, &k_syncbn_stats<NP>, grid, kSyncBnThreads, 0, a);
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
