// gar_noalloc.cu -- ar_all_reduce_noalloc, the all-reduce that allocates
// nothing: its static scratch array, the per-device set-up and the entry
// point (declared in include/gar.h beside the other calls).
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include <cuda_runtime.h>

#include "gar.h"
#include "gar_host.h"
#include "gar_launch.h"

using namespace gar_host;
using gar::CapSmall;
using gar::SegTable;

// ---------------------------------------------------------------------------
// All-reduce without any allocation.
//
// ar_init allocates a device status word with cudaMalloc, so code that may
// not allocate device memory itself cannot create a comm: plugins whose host
// framework owns every device allocation through its own pool, services that
// reserve all memory at start-up and forbid allocations (cudaMalloc can
// synchronise the device) while serving, or code running under a memory
// cap.  ar_all_reduce_noalloc serves them: it runs the bulk-copy pipelined
// all-reduce (k_reduce_tma) with the one piece of scratch that kernel needs
// -- the status word its bounded waits set when they give up -- placed in
// the file-scope array below instead of in memory from cudaMalloc.
// Scratch of ar_all_reduce_noalloc: 256 bytes on every GPU that loads the
// library, held until the process exits.  Word 0 is the status word of the
// pipeline's bounded waits (0 = no wait gave up, 1 = one did).  A call needs
// that one word whatever its arguments, so no call can need more than the
// array holds; the static_assert keeps it that way.
constexpr size_t kNoAllocScratchBytes = 256;
constexpr size_t kNoAllocCallScratchBytes = sizeof(uint32_t);
static_assert(kNoAllocCallScratchBytes <= kNoAllocScratchBytes,
              "ar_all_reduce_noalloc needs more scratch than its static array holds");
static __device__ __align__(256) uint32_t g_noalloc_scratch[kNoAllocScratchBytes / sizeof(uint32_t)];

namespace {

constexpr int kNoAllocMaxDevices = 64;

struct NoAllocDevice {
  bool ready = false;
  int num_sms = 0;
  uint32_t* scratch = nullptr;  // device address of g_noalloc_scratch on this device
};

std::mutex g_noalloc_mu;
NoAllocDevice g_noalloc_dev[kNoAllocMaxDevices];

// Set-up, once per device, with that device current: check the device and
// look up the device address of the scratch array (the host-side name of
// the array is only a stand-in, not an address a kernel can use).  The
// address is kept for the device's context; a context created anew after
// cudaDeviceReset is not served (the entry point's contract says so).
ar_status_t noalloc_setup(int dev, int* num_sms, uint32_t** scratch) {
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoAllocDevice& d = g_noalloc_dev[dev];
  if (!d.ready) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return AR_ERR_CUDA;
    if (major != 10 || minor != 3) return AR_ERR_UNSUPPORTED;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return AR_ERR_CUDA;
    }
    d.scratch = static_cast<uint32_t*>(p);
    d.num_sms = sms;
    d.ready = true;
  }
  *num_sms = d.num_sms;
  *scratch = d.scratch;
  return AR_OK;
}

}  // namespace

extern "C" ar_status_t ar_all_reduce_noalloc(int nranks, const void* const* send, void* const* recv,
                                             size_t count, ar_dtype_t dtype, ar_op_t op,
                                             ar_stream_t stream) {
  if (nranks < 1 || nranks > AR_MAX_RANKS || !valid_dtype(dtype) ||
      (op != AR_SUM && op != AR_MEAN) || send == nullptr || recv == nullptr)
    return AR_ERR_INVALID_ARG;
  const int P = nranks;
  const size_t es = elem_bytes(dtype);
  size_t bytes;
  if (!mul_ok(count, es, &bytes)) return AR_ERR_INVALID_ARG;
  if (count == 0) return AR_OK;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return AR_ERR_CUDA;
  }
  if (dev < 0 || dev >= kNoAllocMaxDevices) return AR_ERR_UNSUPPORTED;
  int num_sms = 0;
  uint32_t* scratch = nullptr;
  ar_status_t st = noalloc_setup(dev, &num_sms, &scratch);
  if (st != AR_OK) return st;

  // The same argument checks as ar_all_reduce, against the current device.
  ar_comm_s view{};
  view.nranks = P;
  view.device = dev;
  view.num_sms = num_sms;
  const char* env = std::getenv("GAR_POINTER_CHECKS");
  view.check_pointers = !(env != nullptr && std::strcmp(env, "0") == 0);
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
  for (int r = 0; r < P; ++r)
    if (!pointer_ok(&view, send[r], bytes) || !pointer_ok(&view, recv[r], bytes))
      return AR_ERR_INVALID_ARG;

  SegTable<CapSmall> t;
  init_table(t, P, P, 2 * P, P, op == AR_MEAN);
  t.stages = gar::tma_stages(P, false, int(es));
  t.stage_bytes = gar::tma_stage_bytes(P, false, 16 / int(es));
  t.status = scratch;
  if (t.stages < 2) return AR_ERR_UNSUPPORTED;
  void* ptrs[2 * AR_MAX_RANKS];
  for (int r = 0; r < P; ++r) {
    ptrs[r] = const_cast<void*>(send[r]);
    ptrs[P + r] = recv[r];
  }
  if (!add_segment(t, ptrs, count, gar::reduce_tile(P, int(es), true), vec_flag(ptrs, 2 * P)))
    return AR_ERR_INVALID_ARG;
  const cudaStream_t strm = static_cast<cudaStream_t>(stream);
  // The status word keeps the previous call's value: clear it first.
  if (cudaMemsetAsync(scratch, 0, kNoAllocCallScratchBytes, strm) != cudaSuccess) return AR_ERR_CUDA;
  const gar::LaunchCtx ctx{dev, num_sms, strm, true, true};
  return from_cuda(dtype == AR_F32 ? gar::launch_reduce_f32<CapSmall>(ctx, false, t)
                                   : gar::launch_reduce_bf16<CapSmall>(ctx, false, t));
}
