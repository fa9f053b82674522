// gar_host.h -- host-side pieces shared by the C ABI translation units: the
// comm object, argument checks, segment-table construction and dispatch.
#pragma once

#include <algorithm>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>

#include "gar.h"
#include "gar_launch.h"

struct ar_comm_s {
  int nranks;
  int device;
  int num_sms;
  ar_op_t default_op;
  uint32_t* d_status;   // sticky device-side status word (0 = ok)
  bool check_pointers;  // validate every pointer against its allocation
  int kernel_mode;      // 0 = default (k_reduce), 1 = k_reduce, 2 = bulk-copy k_reduce_tma
  bool pdl;             // programmatic dependent launch between consecutive kernels
  bool copy_tma;        // all-gather / broadcast on the bulk-store k_copy_tma (GAR_COPY=tma)
  uint64_t small_bytes; // a flat all-reduce below this many bytes per replica: one vector per thread
  int copy_group;       // destinations per windowed copy item (-1 = ceil(D / 4), 0 = classic order)
};

namespace gar_host {

using gar::CapLarge;
using gar::CapSmall;
using gar::CapTiny;
using gar::SegTable;

// True when c is a comm returned by ar_init and not yet destroyed.
bool is_live(const ar_comm_s* c);

// The buffer rules of a bucket (defined in gar_api.cu).
ar_status_t check_bucket_buffers(const ar_comm_s* comm, const ar_bucket_t* bucket,
                                 const ar_sgd_t* sgd);

// Makes the comm's device current for the duration of a call and restores
// the caller's device afterwards.
class DeviceGuard {
 public:
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev_) != cudaSuccess) prev_ = -1;
    ok_ = prev_ == dev || cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev_ >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev_) cudaSetDevice(prev_);
  }
  bool ok() const { return ok_; }

 private:
  int prev_ = -1;
  bool ok_ = false;
};

inline size_t elem_bytes(ar_dtype_t dt) { return dt == AR_BF16 ? 2 : 4; }
inline bool valid_dtype(ar_dtype_t dt) { return dt == AR_F32 || dt == AR_BF16; }

inline bool resolve_op(const ar_comm_s* c, ar_op_t op, ar_op_t* out) {
  if (op == AR_OP_DEFAULT) op = c->default_op;
  if (op != AR_SUM && op != AR_MEAN) return false;
  *out = op;
  return true;
}

inline uintptr_t addr(const void* p) { return reinterpret_cast<uintptr_t>(p); }

inline bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  if (na == 0 || nb == 0) return false;
  return addr(a) < addr(b) + nb && addr(b) < addr(a) + na;
}

inline bool mul_ok(size_t a, size_t b, size_t* out) {
  if (a != 0 && b > SIZE_MAX / a) return false;
  *out = a * b;
  return true;
}

// The driver's cuMemGetAddressRange, fetched through the runtime so the
// library needs no link-time dependency on libcuda.
using MemGetAddressRangeFn = CUresult (*)(CUdeviceptr*, size_t*, CUdeviceptr);

inline MemGetAddressRangeFn address_range_fn() {
  static MemGetAddressRangeFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<MemGetAddressRangeFn>(p);
  }();
  return fn;
}

// A buffer the comm's device may read and write: device memory of this
// device (the whole range inside one allocation), managed memory, or
// registered host memory mapped at the same address.  Pageable host memory
// is refused.  For device memory whose allocation the driver reports,
// [*lo, *hi) receives that allocation's bounds; otherwise both stay 0.
inline bool pointer_check(const ar_comm_s* c, const void* p, size_t bytes, uintptr_t* lo,
                          uintptr_t* hi) {
  *lo = *hi = 0;
  if (p == nullptr) return false;
  if (!c->check_pointers || bytes == 0) return true;
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  switch (at.type) {
    case cudaMemoryTypeDevice: {
      if (at.device != c->device) return false;
      MemGetAddressRangeFn range = address_range_fn();
      if (range != nullptr) {
        CUdeviceptr base = 0;
        size_t size = 0;
        if (range(&base, &size, static_cast<CUdeviceptr>(addr(p))) != CUDA_SUCCESS) return false;
        if (addr(p) + bytes > static_cast<uintptr_t>(base) + size) return false;
        *lo = static_cast<uintptr_t>(base);
        *hi = static_cast<uintptr_t>(base) + size;
      }
      return true;
    }
    case cudaMemoryTypeManaged:
      return true;
    case cudaMemoryTypeHost:
      return at.devicePointer == p;
    default:
      return false;
  }
}

inline bool pointer_ok(const ar_comm_s* c, const void* p, size_t bytes) {
  uintptr_t lo, hi;
  return pointer_check(c, p, bytes, &lo, &hi);
}

// pointer_ok over the many buffers of one call.  The device allocations
// found valid so far in the call are remembered, and a buffer that starts
// inside one of them is checked against that allocation's end alone, with
// no driver query: a bucket's tensors are mostly views of a few large
// allocations, and two driver queries per pointer cost about 0.17 us each.
// One checker serves one call; memory handed to a call must not be
// released while the call validates it.
class PointerChecker {
 public:
  explicit PointerChecker(const ar_comm_s* c) : c_(c) {}

  bool operator()(const void* p, size_t bytes) {
    if (p == nullptr) return false;
    if (!c_->check_pointers || bytes == 0) return true;
    const uintptr_t a = addr(p);
    auto it = seen_.upper_bound(a);
    if (it != seen_.begin()) {
      --it;
      if (a < it->second) return bytes <= it->second - a;
    }
    uintptr_t lo, hi;
    if (!pointer_check(c_, p, bytes, &lo, &hi)) return false;
    if (hi != 0) seen_.emplace(lo, hi);
    return true;
  }

 private:
  const ar_comm_s* c_;
  std::map<uintptr_t, uintptr_t> seen_;  // allocation base -> end
};

inline bool aligned(const void* p, size_t a) { return addr(p) % a == 0; }

// Which reduce kernel a call uses (see ar_comm_s::kernel_mode).  By default
// the register-staged k_reduce: on GB300, back to back, it measured 0.98-1.04
// of the copy peak against 0.84-0.91 for the bulk-copy pipeline (as fast
// as each other only cold and isolated).  The bulk-copy pipeline needs at
// least two shared-memory stages.
inline bool choose_tma(const ar_comm_s* c, int P, bool sgd, size_t es) {
  if (c->kernel_mode == 1) return false;
  if (gar::tma_stages(P, sgd, int(es)) < 2) return false;
  return c->kernel_mode == 2;
}

template <class Cap>
void init_table(SegTable<Cap>& t, int np, int ndst, int stride, int dst_off, bool mean) {
  t.unroll = 0;
  t.dgroup = 0;
  t.stages = 0;
  t.stage_bytes = 0;
  t.status = nullptr;
  t.nseg = 0;
  t.ntiles = 0;
  t.np = np;
  t.ndst = ndst;
  t.stride = stride;
  t.dst_off = dst_off;
  t.mean = mean ? 1 : 0;
  t.write_back = 1;
  t.store_w = 0;
  t.scale = 1.f;
  t.first = 0;
  t.lr = 0.f;
  t.mu = 0.f;
  t.tile0[0] = 0;
}

// Appends one segment; ptrs holds `stride` pointers.  Returns false when a
// 32-bit tile count would overflow.
template <class Cap>
inline bool add_segment(SegTable<Cap>& t, void* const* ptrs, uint64_t numel, uint64_t tile,
                 uint32_t flags, float* master = nullptr, float* mom = nullptr) {
  const uint32_t s = t.nseg;
  const uint64_t tiles = (numel + tile - 1) / tile;
  if (uint64_t(t.ntiles) + tiles > 0xFFFFFFF0ull) return false;
  for (int k = 0; k < t.stride; ++k) t.ptr[s * t.stride + k] = ptrs[k];
  t.numel[s] = numel;
  t.flags[s] = flags;
  t.master[s] = master;
  t.mom[s] = mom;
  t.ntiles += static_cast<uint32_t>(tiles);
  t.tile0[s + 1] = t.ntiles;
  t.nseg = s + 1;
  return true;
}

// Configures the table for the bulk-copy kernel (stages, stage size, status).
template <class Cap>
void set_tma(SegTable<Cap>& t, const ar_comm_s* c, bool sgd, size_t es) {
  t.stages = gar::tma_stages(t.np, sgd, int(es));
  t.stage_bytes = gar::tma_stage_bytes(t.np, sgd, 16 / int(es));
  t.status = c->d_status;
}

// Destinations per windowed item of a copy with at most D destinations per
// segment: ceil(D / 4), about four groups per window (see k_copy), unless
// the comm fixes it (GAR_COPY_GROUP; 0 selects the classic order).
inline int copy_group(const ar_comm_s* c, int D) {
  if (c->copy_group >= 0) return c->copy_group;
  return D < 1 ? 1 : (D + 3) / 4;
}

// Tile (bytes) of the copy kernel a comm uses for a copy of `src_bytes` of
// source, and the table's unroll that selects the register-staged kernel's
// form: 1 or 2 vectors per thread below kCopyWindowBytes, 0 above (four
// vectors, the windowed order).
inline uint64_t copy_tile(const ar_comm_s* c, uint64_t src_bytes) {
  if (c->copy_tma) return uint64_t(gar::kCopyTmaTile);
  return gar::copy_tile_bytes(src_bytes);
}
inline int copy_unroll(const ar_comm_s* c, uint64_t src_bytes) {
  if (c->copy_tma) return 0;
  const int u = gar::copy_unroll_for(src_bytes);
  return u == gar::kCopyUnroll ? 0 : u;
}

inline uint32_t vec_flag(void* const* ptrs, int n, float* const* extra = nullptr, int nextra = 0) {
  for (int k = 0; k < n; ++k)
    if (!aligned(ptrs[k], 16)) return 0;
  for (int k = 0; k < nextra; ++k)
    if (!aligned(extra[k], 16)) return 0;
  return gar::kSegVec;
}

inline ar_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? AR_OK : AR_ERR_CUDA; }

// A debug build (GAR_DEBUG=1) hands every kernel the comm's status word,
// where its index checks report; a release build passes the table as is.
template <class Cap, class F>
inline cudaError_t with_status(const ar_comm_s* c, const SegTable<Cap>& t, F&& launch) {
#if GAR_DEBUG
  if (t.status == nullptr) {
    SegTable<Cap> d = t;
    d.status = c->d_status;
    return launch(d);
  }
#else
  (void)c;
#endif
  return launch(t);
}

template <class Cap>
inline ar_status_t run_reduce(const ar_comm_s* c, ar_dtype_t dt, bool sgd, const SegTable<Cap>& t,
                              cudaStream_t st) {
  if (t.ntiles == 0) return AR_OK;
  const gar::LaunchCtx ctx{c->device, c->num_sms, st, t.stages > 0, c->pdl};
  return from_cuda(with_status(c, t, [&](const SegTable<Cap>& x) {
    return dt == AR_F32 ? gar::launch_reduce_f32<Cap>(ctx, sgd, x)
                        : gar::launch_reduce_bf16<Cap>(ctx, sgd, x);
  }));
}

template <class Cap>
inline ar_status_t run_copy(const ar_comm_s* c, const SegTable<Cap>& t, cudaStream_t st) {
  if (t.ntiles == 0) return AR_OK;
  const gar::LaunchCtx ctx{c->device, c->num_sms, st, c->copy_tma, c->pdl};
  return from_cuda(with_status(c, t, [&](const SegTable<Cap>& x) {
    return gar::launch_copy<Cap>(ctx, x);
  }));
}

// Common checks of a collective call: live comm, dtype, pointer arrays.
inline ar_status_t check_call(const ar_comm_s* c, ar_dtype_t dt) {
  if (!is_live(c)) return AR_ERR_STATE;
  if (!valid_dtype(dt)) return AR_ERR_INVALID_ARG;
  return AR_OK;
}

}  // namespace gar_host
