// k_copy instantiations and launch (all-gather, broadcast).
#include <mutex>
#include <unordered_map>

#include "gar_launch.h"

namespace gar {

int resident_ctas(const void* func) {
  static std::mutex mu;
  static std::unordered_map<const void*, int> cache;
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(func);
  if (it != cache.end()) return it->second;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, func, kThreads, 0) != cudaSuccess || n < 1)
    n = 1;
  cache.emplace(func, n);
  return n;
}

template <class Cap>
cudaError_t launch_copy(const LaunchCtx& ctx, const SegTable<Cap>& tab) {
  const void* f = reinterpret_cast<const void*>(&k_copy<Cap>);
  const unsigned grid = grid_for(tab.ntiles, resident_ctas(f) * ctx.num_sms);
  if (grid == 0) return cudaSuccess;
  k_copy<Cap><<<grid, kThreads, 0, ctx.stream>>>(tab);
  return cudaGetLastError();
}

template cudaError_t launch_copy<CapSmall>(const LaunchCtx&, const SegTable<CapSmall>&);
template cudaError_t launch_copy<CapLarge>(const LaunchCtx&, const SegTable<CapLarge>&);

}  // namespace gar
