// gar_api.cu -- the C ABI declared in include/gar.h: comm lifetime, host-side
// argument validation, segment tables, and dispatch to the kernels.
#include <algorithm>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <unordered_set>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>

#include "gar.h"
#include "gar_host.h"
#include "gar_launch.h"

namespace gar_host {

std::mutex g_live_mu;
std::unordered_set<const ar_comm_s*> g_live;

bool is_live(const ar_comm_s* c) {
  std::lock_guard<std::mutex> lock(g_live_mu);
  return c != nullptr && g_live.count(c) != 0;
}

// The buffer rules of a bucket: every replica (and, with SGD, every fp32
// master and momentum array) element-aligned, pairwise disjoint, and inside
// memory the comm's device may use.  Empty tensors are not inspected.
ar_status_t check_bucket_buffers(const ar_comm_s* comm, const ar_bucket_t* bucket,
                                 const ar_sgd_t* sgd) {
  const int T = bucket->ntensors, P = comm->nranks;
  const size_t es = elem_bytes(bucket->dtype);
  // Sort the ranges and compare neighbours.
  struct Range { uintptr_t lo, hi; };
  std::vector<Range> ranges;
  ranges.reserve(size_t(T) * (P + 2));
  for (int t = 0; t < T; ++t) {
    size_t bytes, fbytes;
    if (!mul_ok(bucket->numel[t], es, &bytes) || !mul_ok(bucket->numel[t], 4, &fbytes))
      return AR_ERR_INVALID_ARG;
    if (bytes == 0) continue;  // an empty tensor's pointers are not inspected
    for (int r = 0; r < P; ++r) {
      const void* p = bucket->dev_ptrs[size_t(t) * P + r];
      if (p == nullptr || !aligned(p, es)) return AR_ERR_INVALID_ARG;
      ranges.push_back({addr(p), addr(p) + bytes});
    }
    if (sgd != nullptr) {
      const float* w = sgd->master[t];
      const float* v = sgd->momentum_buf[t];
      if (w == nullptr || v == nullptr || !aligned(w, 4) || !aligned(v, 4))
        return AR_ERR_INVALID_ARG;
      if (fbytes) {
        ranges.push_back({addr(w), addr(w) + fbytes});
        ranges.push_back({addr(v), addr(v) + fbytes});
      }
    }
  }
  std::sort(ranges.begin(), ranges.end(),
            [](const Range& a, const Range& b) { return a.lo < b.lo; });
  for (size_t k = 1; k < ranges.size(); ++k)
    if (ranges[k].lo < ranges[k - 1].hi) return AR_ERR_INVALID_ARG;
  PointerChecker ok(comm);
  for (int t = 0; t < T; ++t) {
    const size_t n = bucket->numel[t];
    if (n == 0) continue;
    for (int r = 0; r < P; ++r)
      if (!ok(bucket->dev_ptrs[size_t(t) * P + r], n * es)) return AR_ERR_INVALID_ARG;
    if (sgd != nullptr &&
        (!ok(sgd->master[t], n * 4) || !ok(sgd->momentum_buf[t], n * 4)))
      return AR_ERR_INVALID_ARG;
  }

  return AR_OK;
}

}  // namespace gar_host

using namespace gar_host;
using gar::CapLarge;
using gar::CapSmall;
using gar::SegTable;

extern "C" {

const char* ar_status_string(ar_status_t s) {
  switch (s) {
    case AR_OK: return "AR_OK";
    case AR_ERR_INVALID_ARG: return "AR_ERR_INVALID_ARG: invalid argument";
    case AR_ERR_UNSUPPORTED: return "AR_ERR_UNSUPPORTED: unsupported device or feature";
    case AR_ERR_CUDA: return "AR_ERR_CUDA: CUDA call or kernel launch failed";
    case AR_ERR_TIMEOUT: return "AR_ERR_TIMEOUT: a device-side bounded wait gave up";
    case AR_ERR_STATE: return "AR_ERR_STATE: comm is not live";
    case AR_ERR_DEVICE_CHECK:
      return "AR_ERR_DEVICE_CHECK: a device-side index check of a debug build failed";
  }
  return "unknown ar_status_t";
}

// Bytes per replica below which a flat all-reduce takes one vector per thread.
constexpr uint64_t kSmallAllReduceBytes = 16ull << 20;

ar_status_t ar_init(ar_comm_t* comm, int nranks, int cuda_device, ar_op_t default_op) {
  if (comm == nullptr) return AR_ERR_INVALID_ARG;
  *comm = nullptr;
  if (nranks < 1 || nranks > AR_MAX_RANKS) return AR_ERR_INVALID_ARG;
  if (default_op != AR_SUM && default_op != AR_MEAN) return AR_ERR_INVALID_ARG;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess) {
    cudaGetLastError();
    return AR_ERR_CUDA;
  }
  if (cuda_device < 0 || cuda_device >= ndev) return AR_ERR_INVALID_ARG;
  DeviceGuard guard(cuda_device);
  if (!guard.ok()) return AR_ERR_CUDA;
  int major = 0, minor = 0, sms = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, cuda_device) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, cuda_device) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, cuda_device) != cudaSuccess)
    return AR_ERR_CUDA;
  if (major != 10 || minor != 3) return AR_ERR_UNSUPPORTED;  // built for sm_103a only
  ar_comm_s* c = new (std::nothrow) ar_comm_s();
  if (c == nullptr) return AR_ERR_CUDA;
  c->nranks = nranks;
  c->device = cuda_device;
  c->num_sms = sms;
  c->default_op = default_op;
  const char* env = std::getenv("GAR_POINTER_CHECKS");
  c->check_pointers = !(env != nullptr && std::strcmp(env, "0") == 0);
  env = std::getenv("GAR_KERNEL");
  c->kernel_mode = 0;
  if (env != nullptr && std::strcmp(env, "ldg") == 0) c->kernel_mode = 1;
  if (env != nullptr && std::strcmp(env, "tma") == 0) c->kernel_mode = 2;
  env = std::getenv("GAR_PDL");
  c->pdl = !(env != nullptr && std::strcmp(env, "0") == 0);
  // All-gather and broadcast run on the register-staged copy kernel (one
  // CTA per tile) unless GAR_COPY=tma asks for the bulk-store pipeline
  // (measured on GB300, broadcast back to back at 64 MiB - 1 GiB per
  // replica: 1.01-1.08 of the copy peak against 0.85-1.02).
  env = std::getenv("GAR_COPY");
  c->copy_tma = env != nullptr && std::strcmp(env, "tma") == 0;
  // A flat all-reduce of fewer bytes per replica than this runs one vector
  // per thread (four times the CTAs of the default unroll at P <= 4), so
  // that a message of a few MB still spreads over every SM.
  c->small_bytes = kSmallAllReduceBytes;
  env = std::getenv("GAR_SMALL_ALL_REDUCE_BYTES");
  if (env != nullptr) c->small_bytes = std::strtoull(env, nullptr, 10);
  // Destinations per windowed copy item (all-gather, broadcast): by default
  // ceil(D / 4) for D destinations (copy_group).
  c->copy_group = -1;
  env = std::getenv("GAR_COPY_GROUP");
  if (env != nullptr) c->copy_group = std::max(0, std::min(AR_MAX_RANKS, std::atoi(env)));
  if (cudaMalloc(&c->d_status, sizeof(uint32_t)) != cudaSuccess) {
    delete c;
    return AR_ERR_CUDA;
  }
  if (cudaMemset(c->d_status, 0, sizeof(uint32_t)) != cudaSuccess) {
    cudaFree(c->d_status);
    delete c;
    return AR_ERR_CUDA;
  }
  {
    std::lock_guard<std::mutex> lock(g_live_mu);
    g_live.insert(c);
  }
  *comm = c;
  return AR_OK;
}

ar_status_t ar_destroy(ar_comm_t comm) {
  {
    std::lock_guard<std::mutex> lock(g_live_mu);
    if (comm == nullptr || g_live.erase(comm) == 0) return AR_ERR_STATE;
  }
  ar_status_t st = AR_OK;
  {
    DeviceGuard guard(comm->device);
    if (cudaDeviceSynchronize() != cudaSuccess) st = AR_ERR_CUDA;
    if (cudaFree(comm->d_status) != cudaSuccess) st = AR_ERR_CUDA;
  }
  delete comm;
  return st;
}

ar_status_t ar_get_async_error(ar_comm_t comm) {
  if (!is_live(comm)) return AR_ERR_STATE;
  DeviceGuard guard(comm->device);
  uint32_t s = 0;
  if (cudaMemcpy(&s, comm->d_status, sizeof s, cudaMemcpyDeviceToHost) != cudaSuccess)
    return AR_ERR_CUDA;
  if (s & gar::kStatusBounds) return AR_ERR_DEVICE_CHECK;
  if (s != 0) return AR_ERR_TIMEOUT;
  return cudaPeekAtLastError() == cudaSuccess ? AR_OK : AR_ERR_CUDA;
}

ar_status_t ar_selftest_wait_timeout(ar_comm_t comm, unsigned timeout_ms, ar_stream_t stream) {
  if (!is_live(comm)) return AR_ERR_STATE;
  if (timeout_ms < 1 || timeout_ms > 2000) return AR_ERR_INVALID_ARG;
  DeviceGuard guard(comm->device);
  if (!guard.ok()) return AR_ERR_CUDA;
  return from_cuda(gar::launch_wait_selftest(static_cast<cudaStream_t>(stream), comm->d_status,
                                             uint64_t(timeout_ms) * 1000000ull));
}

ar_status_t ar_all_reduce(ar_comm_t comm, const void* const* send, void* const* recv, size_t count,
                          ar_dtype_t dtype, ar_op_t op, ar_stream_t stream) {
  ar_status_t st = check_call(comm, dtype);
  if (st != AR_OK) return st;
  ar_op_t rop;
  if (!resolve_op(comm, op, &rop) || send == nullptr || recv == nullptr) return AR_ERR_INVALID_ARG;
  const int P = comm->nranks;
  const size_t es = elem_bytes(dtype);
  size_t bytes;
  if (!mul_ok(count, es, &bytes)) return AR_ERR_INVALID_ARG;
  if (count == 0) return AR_OK;
  DeviceGuard guard(comm->device);
  if (!guard.ok()) return AR_ERR_CUDA;
  for (int r = 0; r < P; ++r) {
    if (send[r] == nullptr || recv[r] == nullptr) return AR_ERR_INVALID_ARG;
    if (!aligned(send[r], es) || !aligned(recv[r], es)) return AR_ERR_INVALID_ARG;
  }
  for (int r = 0; r < P; ++r)
    for (int q = 0; q < P; ++q) {
      if (q != r && overlap(recv[r], bytes, recv[q], bytes)) return AR_ERR_INVALID_ARG;
      const bool in_place = q == r && recv[r] == send[r];
      if (!in_place && overlap(recv[r], bytes, send[q], bytes)) return AR_ERR_INVALID_ARG;
    }
  PointerChecker ok(comm);
  for (int r = 0; r < P; ++r)
    if (!ok(send[r], bytes) || !ok(recv[r], bytes))
      return AR_ERR_INVALID_ARG;

  SegTable<CapTiny> t;
  init_table(t, P, P, 2 * P, P, rop == AR_MEAN);
  const bool tma = choose_tma(comm, P, false, es);
  if (tma) set_tma(t, comm, false, es);
  if (!tma && bytes < comm->small_bytes) t.unroll = 1;
  void* ptrs[2 * AR_MAX_RANKS];
  for (int r = 0; r < P; ++r) {
    ptrs[r] = const_cast<void*>(send[r]);
    ptrs[P + r] = recv[r];
  }
  if (!add_segment(t, ptrs, count, gar::reduce_tile(P, int(es), tma, false, t.unroll),
                   vec_flag(ptrs, 2 * P)))
    return AR_ERR_INVALID_ARG;
  return run_reduce(comm, dtype, false, t, static_cast<cudaStream_t>(stream));
}

ar_status_t ar_reduce_scatter(ar_comm_t comm, const void* const* send, void* const* recv,
                              size_t count, ar_dtype_t dtype, ar_op_t op, ar_stream_t stream) {
  ar_status_t st = check_call(comm, dtype);
  if (st != AR_OK) return st;
  ar_op_t rop;
  if (!resolve_op(comm, op, &rop) || send == nullptr || recv == nullptr) return AR_ERR_INVALID_ARG;
  const int P = comm->nranks;
  if (count % size_t(P) != 0) return AR_ERR_INVALID_ARG;
  const size_t es = elem_bytes(dtype), shard = count / size_t(P);
  size_t bytes;
  if (!mul_ok(count, es, &bytes)) return AR_ERR_INVALID_ARG;
  const size_t sbytes = shard * es;
  if (count == 0) return AR_OK;
  DeviceGuard guard(comm->device);
  if (!guard.ok()) return AR_ERR_CUDA;
  for (int r = 0; r < P; ++r) {
    if (send[r] == nullptr || recv[r] == nullptr) return AR_ERR_INVALID_ARG;
    if (!aligned(send[r], es) || !aligned(recv[r], es)) return AR_ERR_INVALID_ARG;
  }
  for (int r = 0; r < P; ++r)
    for (int q = 0; q < P; ++q) {
      if (q != r && overlap(recv[r], sbytes, recv[q], sbytes)) return AR_ERR_INVALID_ARG;
      const bool in_place =
          q == r && addr(recv[r]) == addr(send[r]) + size_t(r) * sbytes;
      if (!in_place && overlap(recv[r], sbytes, send[q], bytes)) return AR_ERR_INVALID_ARG;
    }
  PointerChecker ok(comm);
  for (int r = 0; r < P; ++r)
    if (!ok(send[r], bytes) || !ok(recv[r], sbytes))
      return AR_ERR_INVALID_ARG;

  SegTable<CapSmall> t;
  init_table(t, P, 1, P + 1, P, rop == AR_MEAN);
  const bool tma = choose_tma(comm, P, false, es);
  if (tma) set_tma(t, comm, false, es);
  const uint64_t tile = gar::reduce_tile(P, int(es), tma);
  for (int r = 0; r < P; ++r) {
    void* ptrs[AR_MAX_RANKS + 1];
    for (int q = 0; q < P; ++q)
      ptrs[q] = static_cast<char*>(const_cast<void*>(send[q])) + size_t(r) * sbytes;
    ptrs[P] = recv[r];
    if (!add_segment(t, ptrs, shard, tile, vec_flag(ptrs, P + 1))) return AR_ERR_INVALID_ARG;
  }
  return run_reduce(comm, dtype, false, t, static_cast<cudaStream_t>(stream));
}

ar_status_t ar_all_gather(ar_comm_t comm, const void* const* send, void* const* recv, size_t count,
                          ar_dtype_t dtype, ar_stream_t stream) {
  ar_status_t st = check_call(comm, dtype);
  if (st != AR_OK) return st;
  if (send == nullptr || recv == nullptr) return AR_ERR_INVALID_ARG;
  const int P = comm->nranks;
  if (count % size_t(P) != 0) return AR_ERR_INVALID_ARG;
  const size_t es = elem_bytes(dtype), shard = count / size_t(P);
  size_t bytes;
  if (!mul_ok(count, es, &bytes)) return AR_ERR_INVALID_ARG;
  const size_t sbytes = shard * es;
  if (count == 0) return AR_OK;
  DeviceGuard guard(comm->device);
  if (!guard.ok()) return AR_ERR_CUDA;
  for (int r = 0; r < P; ++r) {
    if (send[r] == nullptr || recv[r] == nullptr) return AR_ERR_INVALID_ARG;
    if (!aligned(send[r], es) || !aligned(recv[r], es)) return AR_ERR_INVALID_ARG;
  }
  for (int r = 0; r < P; ++r)
    for (int q = 0; q < P; ++q) {
      if (q != r && overlap(recv[r], bytes, recv[q], bytes)) return AR_ERR_INVALID_ARG;
      const bool in_place =
          q == r && addr(send[r]) == addr(recv[r]) + size_t(r) * sbytes;
      if (!in_place && overlap(recv[r], bytes, send[q], sbytes)) return AR_ERR_INVALID_ARG;
    }
  PointerChecker ok(comm);
  for (int r = 0; r < P; ++r)
    if (!ok(send[r], sbytes) || !ok(recv[r], bytes))
      return AR_ERR_INVALID_ARG;

  SegTable<CapSmall> t;
  init_table(t, 1, 0, P + 1, 1, false);
  t.status = comm->d_status;
  t.unroll = copy_unroll(comm, bytes);
  const uint64_t tile = copy_tile(comm, bytes);
  int max_nd = 0;
  for (int q = 0; q < P; ++q) {
    void* ptrs[AR_MAX_RANKS + 1];
    int nd = 0;
    ptrs[0] = const_cast<void*>(send[q]);
    for (int r = 0; r < P; ++r) {
      void* d = static_cast<char*>(recv[r]) + size_t(q) * sbytes;
      if (d != send[q]) ptrs[1 + nd++] = d;  // an in-place shard is already there
    }
    for (int k = 1 + nd; k < P + 1; ++k) ptrs[k] = ptrs[0];
    const uint32_t flags = vec_flag(ptrs, 1 + nd) | (uint32_t(nd) << 8);
    if (!add_segment(t, ptrs, sbytes, tile, flags)) return AR_ERR_INVALID_ARG;
    max_nd = std::max(max_nd, nd);
  }
  t.dgroup = copy_group(comm, max_nd);
  return run_copy(comm, t, static_cast<cudaStream_t>(stream));
}

ar_status_t ar_broadcast(ar_comm_t comm, void* const* buf, size_t count, ar_dtype_t dtype, int root,
                         ar_stream_t stream) {
  ar_status_t st = check_call(comm, dtype);
  if (st != AR_OK) return st;
  const int P = comm->nranks;
  if (buf == nullptr || root < 0 || root >= P) return AR_ERR_INVALID_ARG;
  const size_t es = elem_bytes(dtype);
  size_t bytes;
  if (!mul_ok(count, es, &bytes)) return AR_ERR_INVALID_ARG;
  if (count == 0) return AR_OK;
  DeviceGuard guard(comm->device);
  if (!guard.ok()) return AR_ERR_CUDA;
  for (int r = 0; r < P; ++r) {
    if (buf[r] == nullptr || !aligned(buf[r], es)) return AR_ERR_INVALID_ARG;
    for (int q = 0; q < r; ++q)
      if (overlap(buf[r], bytes, buf[q], bytes)) return AR_ERR_INVALID_ARG;
  }
  if (P == 1) return AR_OK;
  PointerChecker ok(comm);
  for (int r = 0; r < P; ++r)
    if (!ok(buf[r], bytes)) return AR_ERR_INVALID_ARG;

  SegTable<CapSmall> t;
  init_table(t, 1, 0, P, 1, false);
  t.status = comm->d_status;
  t.dgroup = copy_group(comm, P - 1);
  t.unroll = copy_unroll(comm, bytes);
  void* ptrs[AR_MAX_RANKS];
  int nd = 0;
  ptrs[0] = buf[root];
  for (int r = 0; r < P; ++r)
    if (r != root) ptrs[1 + nd++] = buf[r];
  const uint32_t flags = vec_flag(ptrs, P) | (uint32_t(nd) << 8);
  if (!add_segment(t, ptrs, bytes, copy_tile(comm, bytes), flags)) return AR_ERR_INVALID_ARG;
  return run_copy(comm, t, static_cast<cudaStream_t>(stream));
}

ar_status_t ar_bucket_all_reduce(ar_comm_t comm, const ar_bucket_t* bucket, ar_op_t op,
                                 const ar_sgd_t* sgd, ar_stream_t stream) {
  if (!is_live(comm)) return AR_ERR_STATE;
  ar_op_t rop;
  if (bucket == nullptr || !resolve_op(comm, op, &rop) || !valid_dtype(bucket->dtype) ||
      bucket->ntensors < 0)
    return AR_ERR_INVALID_ARG;
  const int T = bucket->ntensors, P = comm->nranks;
  if (T == 0) return AR_OK;
  if (bucket->dev_ptrs == nullptr || bucket->numel == nullptr) return AR_ERR_INVALID_ARG;
  if (sgd != nullptr && (sgd->master == nullptr || sgd->momentum_buf == nullptr))
    return AR_ERR_INVALID_ARG;
  const size_t es = elem_bytes(bucket->dtype);
  DeviceGuard guard(comm->device);
  if (!guard.ok()) return AR_ERR_CUDA;

  ar_status_t chk = check_bucket_buffers(comm, bucket, sgd);
  if (chk != AR_OK) return chk;

  const bool tma = choose_tma(comm, P, sgd != nullptr, es);
  const uint64_t tile = gar::reduce_tile(P, int(es), tma, sgd != nullptr);
  const cudaStream_t strm = static_cast<cudaStream_t>(stream);
  auto fill = [&](auto& tab, int t0, int t1) -> ar_status_t {
    init_table(tab, P, P, P, 0, rop == AR_MEAN);
    if (tma) set_tma(tab, comm, sgd != nullptr, es);
    if (sgd != nullptr) {
      tab.lr = sgd->lr;
      tab.mu = sgd->momentum;
      tab.write_back = sgd->write_back_grads ? 1 : 0;
    }
    for (int t = t0; t < t1; ++t) {
      void* const* ptrs = bucket->dev_ptrs + size_t(t) * P;
      float* w = sgd ? sgd->master[t] : nullptr;
      float* v = sgd ? sgd->momentum_buf[t] : nullptr;
      float* extra[2] = {w, v};
      const uint32_t flags = vec_flag(ptrs, P, extra, sgd ? 2 : 0);
      if (!add_segment(tab, ptrs, bucket->numel[t], tile, flags, w, v)) return AR_ERR_INVALID_ARG;
    }
    return AR_OK;
  };
  // One launch per group of tensors that fits a parameter block.
  if (T <= CapSmall::kSeg && T * P <= CapSmall::kPtr) {
    SegTable<CapSmall> tab;
    ar_status_t s = fill(tab, 0, T);
    return s != AR_OK ? s : run_reduce(comm, bucket->dtype, sgd != nullptr, tab, strm);
  }
  const int per_launch = std::min(CapLarge::kSeg, CapLarge::kPtr / P);
  std::vector<SegTable<CapLarge>> tabs(1);
  for (int t0 = 0; t0 < T; t0 += per_launch) {
    ar_status_t s = fill(tabs[0], t0, std::min(T, t0 + per_launch));
    if (s == AR_OK) s = run_reduce(comm, bucket->dtype, sgd != nullptr, tabs[0], strm);
    if (s != AR_OK) return s;
  }
  return AR_OK;
}

// Accumulator rules on top of the bucket's: every accumulator fp32, 4-byte
// aligned, inside memory the device may use, and disjoint from every
// gradient replica, master / momentum array and other accumulator.
static ar_status_t check_acc_buffers(const ar_comm_s* comm, const ar_bucket_t* b,
                                     const ar_sgd_t* sgd, const ar_accum_t* acc) {
  if (acc == nullptr || (b->ntensors > 0 && acc->acc == nullptr)) return AR_ERR_INVALID_ARG;
  const int T = b->ntensors, P = comm->nranks;
  const size_t es = elem_bytes(b->dtype);
  PointerChecker ok(comm);
  struct Range { uintptr_t lo, hi; };
  std::vector<Range> ranges;
  for (int t = 0; t < T; ++t) {
    const size_t n = b->numel[t];
    if (n == 0) continue;
    for (int r = 0; r < P; ++r) {
      const void* g = b->dev_ptrs[size_t(t) * P + r];
      const float* a = acc->acc[size_t(t) * P + r];
      if (a == nullptr || !aligned(a, 4)) return AR_ERR_INVALID_ARG;
      if (!ok(a, n * 4)) return AR_ERR_INVALID_ARG;
      ranges.push_back({addr(g), addr(g) + n * es});
      ranges.push_back({addr(a), addr(a) + n * 4});
    }
    if (sgd != nullptr) {
      ranges.push_back({addr(sgd->master[t]), addr(sgd->master[t]) + n * 4});
      ranges.push_back({addr(sgd->momentum_buf[t]), addr(sgd->momentum_buf[t]) + n * 4});
    }
  }
  std::sort(ranges.begin(), ranges.end(), [](const Range& x, const Range& y) { return x.lo < y.lo; });
  for (size_t k = 1; k < ranges.size(); ++k)
    if (ranges[k].lo < ranges[k - 1].hi) return AR_ERR_INVALID_ARG;
  return AR_OK;
}

ar_status_t ar_bucket_accumulate(ar_comm_t comm, const ar_bucket_t* grads, const ar_accum_t* acc,
                                 ar_stream_t stream) {
  if (!is_live(comm)) return AR_ERR_STATE;
  if (grads == nullptr || !valid_dtype(grads->dtype) || grads->ntensors < 0) return AR_ERR_INVALID_ARG;
  const int T = grads->ntensors, P = comm->nranks;
  if (T == 0) return AR_OK;
  if (grads->dev_ptrs == nullptr || grads->numel == nullptr) return AR_ERR_INVALID_ARG;
  DeviceGuard guard(comm->device);
  if (!guard.ok()) return AR_ERR_CUDA;
  ar_status_t st = check_bucket_buffers(comm, grads, nullptr);
  if (st == AR_OK) st = check_acc_buffers(comm, grads, nullptr, acc);
  if (st != AR_OK) return st;
  const size_t es = elem_bytes(grads->dtype);
  const uint64_t tile = gar::accumulate_tile_elems(16 / int(es));
  const cudaStream_t strm = static_cast<cudaStream_t>(stream);
  const gar::LaunchCtx ctx{comm->device, comm->num_sms, strm, false, comm->pdl};
  // One segment per (tensor, rank): ptr = {gradient, accumulator}.
  auto run = [&](auto& tab, int k0, int k1) -> ar_status_t {
    init_table(tab, 1, 1, 2, 1, false);
    tab.status = comm->d_status;
    tab.scale = acc->scale;
    tab.first = acc->first ? 1 : 0;
    for (int k = k0; k < k1; ++k) {
      void* ptrs[2] = {grads->dev_ptrs[k], acc->acc[k]};
      if (!add_segment(tab, ptrs, grads->numel[k / P], tile, vec_flag(ptrs, 2)))
        return AR_ERR_INVALID_ARG;
    }
    if (tab.ntiles == 0) return AR_OK;
    return from_cuda(grads->dtype == AR_F32 ? gar::launch_accumulate_f32(ctx, tab)
                                            : gar::launch_accumulate_bf16(ctx, tab));
  };
  const int segs = T * P;
  if (segs <= CapSmall::kSeg) {
    SegTable<CapSmall> tab;
    return run(tab, 0, segs);
  }
  std::vector<SegTable<CapLarge>> tabs(1);
  for (int k0 = 0; k0 < segs; k0 += CapLarge::kSeg) {
    ar_status_t s2 = run(tabs[0], k0, std::min(segs, k0 + CapLarge::kSeg));
    if (s2 != AR_OK) return s2;
  }
  return AR_OK;
}

ar_status_t ar_bucket_all_reduce_accumulated(ar_comm_t comm, const ar_bucket_t* grads,
                                             const ar_accum_t* acc, ar_op_t op,
                                             const ar_sgd_t* sgd, ar_stream_t stream) {
  if (!is_live(comm)) return AR_ERR_STATE;
  ar_op_t rop;
  if (grads == nullptr || !resolve_op(comm, op, &rop) || !valid_dtype(grads->dtype) ||
      grads->ntensors < 0)
    return AR_ERR_INVALID_ARG;
  const int T = grads->ntensors, P = comm->nranks;
  if (T == 0) return AR_OK;
  if (grads->dev_ptrs == nullptr || grads->numel == nullptr) return AR_ERR_INVALID_ARG;
  if (sgd != nullptr && (sgd->master == nullptr || sgd->momentum_buf == nullptr))
    return AR_ERR_INVALID_ARG;
  DeviceGuard guard(comm->device);
  if (!guard.ok()) return AR_ERR_CUDA;
  ar_status_t st = check_bucket_buffers(comm, grads, sgd);
  if (st == AR_OK) st = check_acc_buffers(comm, grads, sgd, acc);
  if (st != AR_OK) return st;
  const size_t es = elem_bytes(grads->dtype);
  const uint64_t tile = gar::reduce_acc_tile_elems(16 / int(es));
  const cudaStream_t strm = static_cast<cudaStream_t>(stream);
  const gar::LaunchCtx ctx{comm->device, comm->num_sms, strm, false, comm->pdl};
  // One segment per tensor: ptr = {P gradient replicas, P accumulators}.
  auto run = [&](auto& tab, int t0, int t1) -> ar_status_t {
    init_table(tab, P, P, 2 * P, 0, rop == AR_MEAN);
    tab.status = comm->d_status;
    tab.scale = acc->scale;
    tab.first = acc->first ? 1 : 0;
    if (sgd != nullptr) {
      tab.lr = sgd->lr;
      tab.mu = sgd->momentum;
      tab.write_back = sgd->write_back_grads ? 1 : 0;
    }
    for (int t = t0; t < t1; ++t) {
      void* ptrs[2 * AR_MAX_RANKS];
      for (int r = 0; r < P; ++r) {
        ptrs[r] = grads->dev_ptrs[size_t(t) * P + r];
        ptrs[P + r] = acc->acc[size_t(t) * P + r];
      }
      float* w = sgd ? sgd->master[t] : nullptr;
      float* v = sgd ? sgd->momentum_buf[t] : nullptr;
      float* extra[2] = {w, v};
      if (!add_segment(tab, ptrs, grads->numel[t], tile, vec_flag(ptrs, 2 * P, extra, sgd ? 2 : 0),
                       w, v))
        return AR_ERR_INVALID_ARG;
    }
    if (tab.ntiles == 0) return AR_OK;
    return from_cuda(grads->dtype == AR_F32 ? gar::launch_reduce_acc_f32(ctx, sgd != nullptr, tab)
                                            : gar::launch_reduce_acc_bf16(ctx, sgd != nullptr, tab));
  };
  if (T <= CapSmall::kSeg && 2 * T * P <= CapSmall::kPtr) {
    SegTable<CapSmall> tab;
    return run(tab, 0, T);
  }
  const int per = std::min(CapLarge::kSeg, CapLarge::kPtr / (2 * P));
  std::vector<SegTable<CapLarge>> tabs(1);
  for (int t0 = 0; t0 < T; t0 += per) {
    ar_status_t s2 = run(tabs[0], t0, std::min(T, t0 + per));
    if (s2 != AR_OK) return s2;
  }
  return AR_OK;
}

ar_status_t ar_sharded_sgd_step(ar_comm_t comm, const void* const* grads, void* const* params,
                                float* const* master_shards, float* const* momentum_shards,
                                size_t count, ar_dtype_t dtype, ar_op_t op, float lr,
                                float momentum, ar_stream_t stream) {
  ar_status_t st = check_call(comm, dtype);
  if (st != AR_OK) return st;
  ar_op_t rop;
  if (!resolve_op(comm, op, &rop) || grads == nullptr || params == nullptr ||
      master_shards == nullptr || momentum_shards == nullptr)
    return AR_ERR_INVALID_ARG;
  const int P = comm->nranks;
  if (count % size_t(P) != 0) return AR_ERR_INVALID_ARG;
  const size_t es = elem_bytes(dtype), shard = count / size_t(P);
  size_t bytes;
  if (!mul_ok(count, es, &bytes)) return AR_ERR_INVALID_ARG;
  if (count == 0) return AR_OK;
  const size_t sbytes = shard * 4;
  DeviceGuard guard(comm->device);
  if (!guard.ok()) return AR_ERR_CUDA;
  // grads / params: in place (params[r] == grads[r]) or disjoint; shards:
  // fp32, disjoint from everything.
  PointerChecker ok(comm);
  struct Range { uintptr_t lo, hi; };
  std::vector<Range> ranges;
  for (int r = 0; r < P; ++r) {
    const void* g = grads[r];
    void* p = params[r];
    const float* w = master_shards[r];
    const float* v = momentum_shards[r];
    if (g == nullptr || p == nullptr || w == nullptr || v == nullptr) return AR_ERR_INVALID_ARG;
    if (!aligned(g, es) || !aligned(p, es) || !aligned(w, 4) || !aligned(v, 4))
      return AR_ERR_INVALID_ARG;
    if (!ok(g, bytes) || !ok(p, bytes) ||
        !ok(w, sbytes) || !ok(v, sbytes))
      return AR_ERR_INVALID_ARG;
    ranges.push_back({addr(g), addr(g) + bytes});
    if (p != g) ranges.push_back({addr(p), addr(p) + bytes});
    if (sbytes) {
      ranges.push_back({addr(w), addr(w) + sbytes});
      ranges.push_back({addr(v), addr(v) + sbytes});
    }
  }
  std::sort(ranges.begin(), ranges.end(), [](const Range& x, const Range& y) { return x.lo < y.lo; });
  for (size_t k = 1; k < ranges.size(); ++k)
    if (ranges[k].lo < ranges[k - 1].hi) return AR_ERR_INVALID_ARG;

  // One segment per shard r: the P replicas' part r of the gradient in, the
  // P replicas' part r of the parameters out, shard r's w and v.
  SegTable<CapSmall> t;
  init_table(t, P, P, 2 * P, P, rop == AR_MEAN);
  t.lr = lr;
  t.mu = momentum;
  t.write_back = 1;
  t.store_w = 1;
  const uint64_t tile = gar::reduce_tile(P, int(es), false, true);
  for (int r = 0; r < P; ++r) {
    void* ptrs[2 * AR_MAX_RANKS];
    for (int q = 0; q < P; ++q) {
      ptrs[q] = static_cast<char*>(const_cast<void*>(grads[q])) + size_t(r) * shard * es;
      ptrs[P + q] = static_cast<char*>(params[q]) + size_t(r) * shard * es;
    }
    float* extra[2] = {master_shards[r], momentum_shards[r]};
    if (!add_segment(t, ptrs, shard, tile, vec_flag(ptrs, 2 * P, extra, 2), master_shards[r],
                     momentum_shards[r]))
      return AR_ERR_INVALID_ARG;
  }
  return run_reduce(comm, dtype, true, t, static_cast<cudaStream_t>(stream));
}

ar_status_t ar_syncbn_stats(ar_comm_t comm, const float* const* sum, const float* const* sqsum,
                            const uint64_t* count, float* const* mean, float* const* invstd,
                            size_t channels, float eps, ar_stream_t stream) {
  if (!is_live(comm)) return AR_ERR_STATE;
  if (sum == nullptr || sqsum == nullptr || count == nullptr || mean == nullptr ||
      invstd == nullptr)
    return AR_ERR_INVALID_ARG;
  const int P = comm->nranks;
  uint64_t n = 0;
  for (int r = 0; r < P; ++r) {
    if (count[r] > (uint64_t(1) << 53) - n) return AR_ERR_INVALID_ARG;  // n stays exact in fp64
    n += count[r];
  }
  if (n == 0) return AR_ERR_INVALID_ARG;
  if (channels == 0) return AR_OK;
  size_t bytes;
  if (!mul_ok(channels, 4, &bytes)) return AR_ERR_INVALID_ARG;
  DeviceGuard guard(comm->device);
  if (!guard.ok()) return AR_ERR_CUDA;
  PointerChecker ok(comm);
  struct Range { uintptr_t lo, hi; };
  std::vector<Range> outs;
  for (int r = 0; r < P; ++r) {
    const void* ps[4] = {sum[r], sqsum[r], mean[r], invstd[r]};
    for (const void* p : ps)
      if (p == nullptr || !aligned(p, 4) || !ok(p, bytes)) return AR_ERR_INVALID_ARG;
    outs.push_back({addr(mean[r]), addr(mean[r]) + bytes});
    outs.push_back({addr(invstd[r]), addr(invstd[r]) + bytes});
  }
  std::sort(outs.begin(), outs.end(), [](const Range& x, const Range& y) { return x.lo < y.lo; });
  for (size_t k = 1; k < outs.size(); ++k)
    if (outs[k].lo < outs[k - 1].hi) return AR_ERR_INVALID_ARG;
  for (const Range& o : outs)
    for (int r = 0; r < P; ++r)
      if (overlap(reinterpret_cast<const void*>(o.lo), bytes, sum[r], bytes) ||
          overlap(reinterpret_cast<const void*>(o.lo), bytes, sqsum[r], bytes))
        return AR_ERR_INVALID_ARG;
  gar::SyncBnArgs a{};
  for (int r = 0; r < P; ++r) {
    a.sum[r] = sum[r];
    a.sqsum[r] = sqsum[r];
    a.mean[r] = mean[r];
    a.invstd[r] = invstd[r];
  }
  a.n = double(n);  // exact: n <= 2^53
  a.rn = 1.0 / a.n;  // the IEEE quotient, rounded to nearest
  a.eps = double(eps);
  a.channels = channels;
  a.np = P;
  a.status = comm->d_status;
  const gar::LaunchCtx ctx{comm->device, comm->num_sms, static_cast<cudaStream_t>(stream), false,
                           comm->pdl};
  return from_cuda(gar::launch_syncbn_stats(ctx, a));
}

ar_status_t ar_bucket_plan(int ntensors, const size_t* nbytes, size_t cap_bytes, int* bucket_of,
                           int* nbuckets) {
  if (ntensors < 0 || cap_bytes == 0 || nbuckets == nullptr) return AR_ERR_INVALID_ARG;
  if (ntensors > 0 && (nbytes == nullptr || bucket_of == nullptr)) return AR_ERR_INVALID_ARG;
  int b = -1;
  size_t fill = 0;
  for (int t = ntensors - 1; t >= 0; --t) {
    const bool full = fill > 0 && (fill > cap_bytes || nbytes[t] > cap_bytes - fill);
    if (b < 0 || full) {
      ++b;
      fill = 0;
    }
    bucket_of[t] = b;
    fill = nbytes[t] > SIZE_MAX - fill ? SIZE_MAX : fill + nbytes[t];
  }
  *nbuckets = b + 1;
  return AR_OK;
}

}  // extern "C"
