// gar_launch.h -- internal interface between the C ABI (gar_api.cu) and the
// kernel translation units (gar_reduce_*.cu, gar_copy.cu).
#pragma once

#include <cuda_runtime.h>

#include "gar_kernels.cuh"

namespace gar {

struct LaunchCtx {
  int device;
  int num_sms;
  cudaStream_t stream;
};

// Launch k_reduce on the table for fp32 or bf16 replicas, choosing the
// specialisation for P (2, 4, 8, else the generic runtime-P kernel).
template <class Cap>
cudaError_t launch_reduce_f32(const LaunchCtx& ctx, bool sgd, const SegTable<Cap>& tab);
template <class Cap>
cudaError_t launch_reduce_bf16(const LaunchCtx& ctx, bool sgd, const SegTable<Cap>& tab);

template <class Cap>
cudaError_t launch_copy(const LaunchCtx& ctx, const SegTable<Cap>& tab);

// Tile size in elements of k_reduce for P ranks and the given element size.
inline uint64_t reduce_tile(int P, int elem_bytes) {
  const int PT = (P == 2 || P == 4 || P == 8) ? P : 0;
  return reduce_tile_elems(PT, 16 / elem_bytes);
}

// Persistent grid: at most (resident CTAs per SM) x (SMs), and as few CTAs
// as keep the per-CTA tile count the same, so that all CTAs finish
// together.
inline unsigned grid_for(uint32_t ntiles, int max_ctas) {
  if (ntiles == 0) return 0;
  const uint32_t per_cta = (ntiles + max_ctas - 1) / max_ctas;
  return (ntiles + per_cta - 1) / per_cta;
}

// Resident CTAs per SM for a kernel (cached per function).
int resident_ctas(const void* func);

}  // namespace gar
