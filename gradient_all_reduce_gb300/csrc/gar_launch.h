// gar_launch.h -- internal interface between the C ABI (gar_api.cu) and the
// kernel translation units (gar_reduce_*.cu, gar_copy.cu).
#pragma once

#include <type_traits>

#include <cuda_runtime.h>

#include "gar_tma.cuh"

namespace gar {

struct LaunchCtx {
  int device;
  int num_sms;
  cudaStream_t stream;
  bool tma;             // k_reduce_tma (bulk-copy pipeline) instead of k_reduce
  bool pdl;             // launch with programmatic stream serialization
};

// Launch `kernel<<<grid, block, smem, ctx.stream>>>(tab)`, opting in to
// programmatic dependent launch when ctx.pdl is set.
template <class Tab>
cudaError_t launch_ex(const LaunchCtx& ctx, void (*kernel)(Tab), unsigned grid, unsigned block,
                      size_t smem, const Tab& tab) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = ctx.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = ctx.pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, tab);
}

// Shared-memory budget of the bulk-copy kernel's stages.
constexpr uint32_t kTmaSmemBudget = 200 * 1024;

// Stages of k_reduce_tma for P ranks (0 when fewer than two stages fit).
inline int tma_stages(int P, bool sgd, int elem_bytes) {
  const uint32_t sb = tma_stage_bytes(P, sgd, 16 / elem_bytes);
  const uint32_t s = kTmaSmemBudget / sb;
  if (s < 2) return 0;
  return s > uint32_t(kTmaMaxStages) ? kTmaMaxStages : int(s);
}

// Launch k_reduce on the table for fp32 or bf16 replicas, without or with
// the fused SGD step, choosing the specialisation for P (rank_class).  A
// flat all-reduce's one-segment table (CapTiny) never carries the SGD step.
template <class Cap>
cudaError_t launch_reduce_plain_f32(const LaunchCtx& ctx, const SegTable<Cap>& tab);
template <class Cap>
cudaError_t launch_reduce_plain_bf16(const LaunchCtx& ctx, const SegTable<Cap>& tab);
template <class Cap>
cudaError_t launch_reduce_sgd_f32(const LaunchCtx& ctx, const SegTable<Cap>& tab);
template <class Cap>
cudaError_t launch_reduce_sgd_bf16(const LaunchCtx& ctx, const SegTable<Cap>& tab);

template <class Cap>
inline cudaError_t launch_reduce_f32(const LaunchCtx& ctx, bool sgd, const SegTable<Cap>& tab) {
  if constexpr (std::is_same<Cap, CapTiny>::value) {
    return sgd ? cudaErrorNotSupported : launch_reduce_plain_f32(ctx, tab);
  } else {
    return sgd ? launch_reduce_sgd_f32(ctx, tab) : launch_reduce_plain_f32(ctx, tab);
  }
}
template <class Cap>
inline cudaError_t launch_reduce_bf16(const LaunchCtx& ctx, bool sgd, const SegTable<Cap>& tab) {
  if constexpr (std::is_same<Cap, CapTiny>::value) {
    return sgd ? cudaErrorNotSupported : launch_reduce_plain_bf16(ctx, tab);
  } else {
    return sgd ? launch_reduce_sgd_bf16(ctx, tab) : launch_reduce_plain_bf16(ctx, tab);
  }
}

// The accumulation kernels (DDP's no_sync) for fp32 or bf16 gradients.
template <class Cap>
cudaError_t launch_accumulate_f32(const LaunchCtx& ctx, const SegTable<Cap>& tab);
template <class Cap>
cudaError_t launch_accumulate_bf16(const LaunchCtx& ctx, const SegTable<Cap>& tab);
template <class Cap>
cudaError_t launch_reduce_acc_f32(const LaunchCtx& ctx, bool sgd, const SegTable<Cap>& tab);
template <class Cap>
cudaError_t launch_reduce_acc_bf16(const LaunchCtx& ctx, bool sgd, const SegTable<Cap>& tab);

template <class Cap>
cudaError_t launch_copy(const LaunchCtx& ctx, const SegTable<Cap>& tab);

// Arguments of the synchronized batch-norm statistics kernel.
struct SyncBnArgs {
  const float* sum[kMaxRanks];    // rank r's per-channel sums of x
  const float* sqsum[kMaxRanks];  // ... and of x * x
  float* mean[kMaxRanks];         // outputs, every rank
  float* invstd[kMaxRanks];
  double n;                       // total values per channel over all ranks
  double rn;                      // RN(1 / n)
  double eps;
  uint64_t channels;
  int np;
  uint32_t* status;               // the comm's status word (debug-build checks)
};
cudaError_t launch_syncbn_stats(const LaunchCtx& ctx, const SyncBnArgs& args);

// One warp runs the bounded mbarrier wait on a barrier nothing arrives at.
cudaError_t launch_wait_selftest(cudaStream_t stream, uint32_t* status, uint64_t limit_ns);

// Tile size in elements of k_reduce (or k_reduce_tma when tma is set) for
// P ranks, the given element size, with or without the SGD step, and the
// table's unroll (0 = the kernel's own).
inline uint64_t reduce_tile(int P, int elem_bytes, bool tma = false, bool sgd = false,
                            int unroll = 0) {
  if (tma) return tma_tile_elems(16 / elem_bytes);
  const int PT = rank_class(P);
  const int U = unroll > 0 ? unroll : (sgd ? unroll_for_sgd(PT) : unroll_for(PT));
  return uint64_t(U) * kThreads * (16 / elem_bytes);
}

// The register-staged kernels launch one CTA per tile.  The block scheduler
// then hands the tiles out in order as CTAs retire, so the CTAs in flight
// always cover one compact window of every buffer, and no CTA is left with
// a tail of its own.  Measured on GB300 against a persistent grid of the
// same kernels (grid-stride over equal tile counts): flat all-reduce at
// >= 256 MiB per replica 0.92-0.95 -> 1.03-1.05 of the copy peak, broadcast
// 0.84-0.93 -> 0.95-1.04, the ViT-B/16 bucket step 0.92 -> 0.98 launched
// one bucket after another and 0.98 -> 1.02 through the reducer.
inline unsigned grid_per_tile(uint32_t ntiles) { return ntiles < 0x7FFFFFFFu ? ntiles : 0x7FFFFFFFu; }

// Persistent grid of the bulk-copy pipelines (each CTA keeps a ring of
// shared-memory stages busy): at most (resident CTAs per SM) x (SMs), and
// as few CTAs as keep the per-CTA tile count the same, so that all CTAs
// finish together.
inline unsigned grid_for(uint32_t ntiles, int max_ctas) {
  if (ntiles == 0) return 0;
  const uint32_t per_cta = (ntiles + max_ctas - 1) / max_ctas;
  return (ntiles + per_cta - 1) / per_cta;
}

// Resident CTAs per SM of a kernel on the current device (cached per device,
// function, block size and shared memory) into *per_sm; smem is the dynamic
// shared memory per CTA, which the function's attribute is raised to on
// every call.  Returns the CUDA error of either step.
cudaError_t resident_ctas(const void* func, int threads, size_t smem, int* per_sm);

}  // namespace gar
