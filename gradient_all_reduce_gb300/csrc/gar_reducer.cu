// gar_reducer.cu -- the DDP gradient reducer: bucketing engine of the C ABI.
//
// DDP packs gradients into ~25 MB buckets in reverse parameter order and
// launches an asynchronous all-reduce on each bucket as soon as all of its
// gradients are ready, while the backward pass goes on producing the next
// ones; every rank reduces the buckets in the same order ("Distributed
// Training", computervisiononline.com, "Data parallelism and all-reduce").
// Here the P ranks are P replica buffers on one GPU, so a reducer holds the
// whole group's gradient set:
//   create:      plan the buckets, validate every buffer once, and build
//                each bucket's launch table(s) ahead of time;
//   mark_ready:  a tensor's gradient is final on the caller's stream; when
//                a bucket's last tensor is marked, the bucket's kernel is
//                launched on one of two high-priority communication
//                streams (alternating, so consecutive buckets overlap),
//                ordered after the marking streams' work by events;
//   finalize:    launch any bucket still waiting (its unmarked tensors are
//                taken as ready on the caller's stream), then make the
//                caller's stream wait for every launched bucket; the marks
//                reset for the next step.
// Buckets that one call completes together (mark_ready_many, finalize) go
// out as one launch over their combined segment table when it fits one
// parameter block: the same arithmetic per element, fewer launches and no
// ramp-up and drain between them.  When one call completes every bucket of
// the step and every tensor of the step was marked on one stream, nothing
// is left to overlap with: the buckets launch on that stream itself, so
// that consecutive steps' kernels follow each other on one stream, where
// programmatic dependent launch lets each start while the one before
// drains (a launch on a communication stream is joined by events on both
// sides, which no kernel can start ahead of).
#include <mutex>
#include <new>
#include <unordered_set>
#include <vector>

#include "gar_host.h"

using namespace gar_host;

struct ar_reducer_s {
  struct Bucket {
    std::vector<int> tensors;                  // in launch-table order
    std::vector<SegTable<CapSmall>> small;     // launch tables (one of the two lists is used)
    std::vector<SegTable<CapLarge>> large;
    int pending = 0;                           // tensors not yet marked this step
    bool launched = false;
    cudaEvent_t done = nullptr;                // recorded after the bucket's kernel
    std::vector<cudaStream_t> mark_streams;    // distinct streams that marked its tensors
    bool direct = false;                       // launched on its marking stream (below)
    cudaStream_t direct_stream = nullptr;
  };

  ar_comm_s* comm = nullptr;
  int P = 0;
  int ntensors = 0;
  ar_dtype_t dtype = AR_F32;
  bool sgd = false;
  std::vector<int> bucket_of;
  std::vector<char> marked;
  std::vector<Bucket> buckets;
  cudaStream_t streams[2] = {nullptr, nullptr};
  cudaEvent_t done[2] = {nullptr, nullptr};
  bool used[2] = {false, false};
  int next = 0;
  cudaEvent_t join = nullptr;
  bool direct = false;                         // this step's buckets went to direct_stream
  cudaStream_t direct_stream = nullptr;
  SegTable<CapLarge> group;                    // combined table of buckets launched together
  uint64_t launches = 0;                       // kernel launches issued so far
};

namespace {

std::mutex g_red_mu;
std::unordered_set<const ar_reducer_s*> g_reducers;

bool reducer_live(const ar_reducer_s* r) {
  std::lock_guard<std::mutex> lock(g_red_mu);
  return r != nullptr && g_reducers.count(r) != 0;
}

void release(ar_reducer_s* r) {
  for (auto& bk : r->buckets)
    if (bk.done) cudaEventDestroy(bk.done);
  for (int k = 0; k < 2; ++k) {
    if (r->done[k]) cudaEventDestroy(r->done[k]);
    if (r->streams[k]) cudaStreamDestroy(r->streams[k]);
  }
  if (r->join) cudaEventDestroy(r->join);
  delete r;
}

// Where the buckets one call completes are launched: the communication
// streams, or (direct) the one stream that marked every tensor of the step,
// when the call completes every bucket of the step.
struct Target {
  bool direct = false;
  cudaStream_t stream = nullptr;
};

Target pick_target(const ar_reducer_s* r, const std::vector<int>& ready) {
  Target tg;
  size_t nonempty = 0;
  for (const auto& bk : r->buckets) {
    if (bk.launched) return tg;
    if (!bk.tensors.empty()) ++nonempty;
  }
  if (ready.size() != nonempty || ready.empty()) return tg;
  const cudaStream_t s = r->buckets[ready.front()].mark_streams.empty()
                             ? nullptr
                             : r->buckets[ready.front()].mark_streams.front();
  for (int b : ready) {
    const auto& ms = r->buckets[b].mark_streams;
    if (ms.size() != 1 || ms.front() != s) return tg;
  }
  tg.direct = true;
  tg.stream = s;
  return tg;
}

// The stream of a launch: the next communication stream (index *k), after
// the work of every stream that marked a tensor of buckets bs; or, direct,
// the marking stream itself (*k = -1), which orders the launch already.
ar_status_t launch_stream(ar_reducer_s* r, const Target& tg, const std::vector<int>& bs, int* k,
                          cudaStream_t* s) {
  if (tg.direct) {
    *k = -1;
    *s = tg.stream;
    return AR_OK;
  }
  *k = r->next;
  r->next ^= 1;
  *s = r->streams[*k];
  std::vector<cudaStream_t> waited;
  for (int b : bs)
    for (cudaStream_t ms : r->buckets[b].mark_streams) {
      bool seen = false;
      for (cudaStream_t x : waited) seen = seen || x == ms;
      if (seen) continue;
      waited.push_back(ms);
      if (cudaEventRecord(r->join, ms) != cudaSuccess) return AR_ERR_CUDA;
      if (cudaStreamWaitEvent(*s, r->join, 0) != cudaSuccess) return AR_ERR_CUDA;
    }
  return AR_OK;
}

// Buckets bs were launched on stream s (communication stream k, or direct
// when k < 0).  On a communication stream their completion events are
// recorded now; a direct launch records a bucket's event only when
// ar_reducer_wait_bucket asks for it, so that nothing comes between
// consecutive steps' kernels on the stream.
ar_status_t note_launched(ar_reducer_s* r, const std::vector<int>& bs, int k, cudaStream_t s) {
  if (k >= 0) {
    if (cudaEventRecord(r->done[k], s) != cudaSuccess) return AR_ERR_CUDA;
    r->used[k] = true;
  } else {
    r->direct = true;
    r->direct_stream = s;
  }
  for (int b : bs) {
    auto& bk = r->buckets[b];
    if (k >= 0 && cudaEventRecord(bk.done, s) != cudaSuccess) return AR_ERR_CUDA;
    bk.direct = k < 0;
    bk.direct_stream = s;
    bk.launched = true;
  }
  return AR_OK;
}

// Launch bucket b alone (each of its launch tables).
ar_status_t launch_bucket(ar_reducer_s* r, int b, const Target& tg) {
  ar_reducer_s::Bucket& bk = r->buckets[b];
  int k = -1;
  cudaStream_t s = nullptr;
  ar_status_t st = launch_stream(r, tg, {b}, &k, &s);
  if (st != AR_OK) return st;
  for (const auto& t : bk.small) {
    st = run_reduce(r->comm, r->dtype, r->sgd, t, s);
    if (st != AR_OK) return st;
    if (t.ntiles > 0) ++r->launches;
  }
  for (const auto& t : bk.large) {
    st = run_reduce(r->comm, r->dtype, r->sgd, t, s);
    if (st != AR_OK) return st;
    if (t.ntiles > 0) ++r->launches;
  }
  return note_launched(r, {b}, k, s);
}

void note_stream(ar_reducer_s::Bucket& bk, cudaStream_t s) {
  for (cudaStream_t x : bk.mark_streams)
    if (x == s) return;
  bk.mark_streams.push_back(s);
}

// The bucket's only launch table, if it has exactly one.
template <class F>
bool with_single_table(const ar_reducer_s::Bucket& bk, F&& f) {
  if (bk.small.size() + bk.large.size() != 1) return false;
  if (!bk.small.empty()) return f(bk.small.front());
  return f(bk.large.front());
}

// Appends src's segments to the combined table g (whose header matches,
// every table of a reducer being built with the same parameters); false,
// leaving g unchanged, if they do not fit.
template <class Cap>
bool append_segments(SegTable<CapLarge>& g, const SegTable<Cap>& src) {
  if (g.nseg + src.nseg > uint32_t(CapLarge::kSeg) ||
      uint64_t(g.nseg + src.nseg) * uint64_t(g.stride) > uint64_t(CapLarge::kPtr) ||
      uint64_t(g.ntiles) + src.ntiles > 0xFFFFFFF0ull)
    return false;
  for (uint32_t k = 0; k < src.nseg; ++k) {
    const uint32_t d = g.nseg;
    for (int q = 0; q < g.stride; ++q) g.ptr[size_t(d) * g.stride + q] = src.ptr[size_t(k) * src.stride + q];
    g.numel[d] = src.numel[k];
    g.flags[d] = src.flags[k];
    g.master[d] = src.master[k];
    g.mom[d] = src.mom[k];
    g.ntiles += src.tile0[k + 1] - src.tile0[k];
    g.tile0[d + 1] = g.ntiles;
    g.nseg = d + 1;
  }
  return true;
}

// The header of a combined table: src's launch parameters, no segments.
template <class Cap>
void start_group(SegTable<CapLarge>& g, const SegTable<Cap>& src) {
  g.nseg = 0;
  g.ntiles = 0;
  g.np = src.np;
  g.ndst = src.ndst;
  g.stride = src.stride;
  g.dst_off = src.dst_off;
  g.mean = src.mean;
  g.write_back = src.write_back;
  g.store_w = src.store_w;
  g.lr = src.lr;
  g.mu = src.mu;
  g.scale = src.scale;
  g.first = src.first;
  g.unroll = src.unroll;
  g.dgroup = src.dgroup;
  g.stages = src.stages;
  g.stage_bytes = src.stage_bytes;
  g.status = src.status;
  g.tile0[0] = 0;
}

// One launch of the combined table of buckets bs.
ar_status_t launch_group(ar_reducer_s* r, const std::vector<int>& bs, const Target& tg) {
  int k = -1;
  cudaStream_t s = nullptr;
  ar_status_t st = launch_stream(r, tg, bs, &k, &s);
  if (st != AR_OK) return st;
  st = run_reduce(r->comm, r->dtype, r->sgd, r->group, s);
  if (st != AR_OK) return st;
  if (r->group.ntiles > 0) ++r->launches;
  return note_launched(r, bs, k, s);
}

// Launch the buckets that one call completed, in completion order:
// consecutive buckets with a single launch table each share one launch of
// their combined table while it fits; any other bucket launches alone.
ar_status_t launch_ready(ar_reducer_s* r, const std::vector<int>& ready) {
  const Target tg = pick_target(r, ready);
  if (ready.size() == 1) return launch_bucket(r, ready.front(), tg);
  std::vector<int> group;
  auto flush = [&]() -> ar_status_t {
    ar_status_t st = AR_OK;
    if (group.size() == 1) st = launch_bucket(r, group.front(), tg);
    else if (!group.empty()) st = launch_group(r, group, tg);
    group.clear();
    return st;
  };
  for (int b : ready) {
    const auto& bk = r->buckets[b];
    const bool single = bk.small.size() + bk.large.size() == 1;
    if (!single) {
      ar_status_t st = flush();
      if (st == AR_OK) st = launch_bucket(r, b, tg);
      if (st != AR_OK) return st;
      continue;
    }
    if (group.empty()) with_single_table(bk, [&](const auto& t) { start_group(r->group, t); return true; });
    bool fits = with_single_table(bk, [&](const auto& t) { return append_segments(r->group, t); });
    if (!fits) {
      ar_status_t st = flush();
      if (st != AR_OK) return st;
      with_single_table(bk, [&](const auto& t) { start_group(r->group, t); return true; });
      fits = with_single_table(bk, [&](const auto& t) { return append_segments(r->group, t); });
      if (!fits) return AR_ERR_INVALID_ARG;  // a single table always fits
    }
    group.push_back(b);
  }
  return flush();
}

}  // namespace

extern "C" {

ar_status_t ar_reducer_create(ar_reducer_t* out, ar_comm_t comm, const ar_bucket_t* grads,
                              size_t cap_bytes, ar_op_t op, const ar_sgd_t* sgd) {
  if (out == nullptr) return AR_ERR_INVALID_ARG;
  *out = nullptr;
  if (!is_live(comm)) return AR_ERR_STATE;
  ar_op_t rop;
  if (grads == nullptr || cap_bytes == 0 || !resolve_op(comm, op, &rop) ||
      !valid_dtype(grads->dtype) || grads->ntensors < 0)
    return AR_ERR_INVALID_ARG;
  const int T = grads->ntensors, P = comm->nranks;
  if (T > 0 && (grads->dev_ptrs == nullptr || grads->numel == nullptr)) return AR_ERR_INVALID_ARG;
  if (sgd != nullptr && T > 0 && (sgd->master == nullptr || sgd->momentum_buf == nullptr))
    return AR_ERR_INVALID_ARG;
  const size_t es = elem_bytes(grads->dtype);
  DeviceGuard guard(comm->device);
  if (!guard.ok()) return AR_ERR_CUDA;

  // Validate the whole gradient set once (the rules of ar_bucket_all_reduce).
  ar_status_t st = check_bucket_buffers(comm, grads, sgd);
  if (st != AR_OK) return st;

  ar_reducer_s* r = new (std::nothrow) ar_reducer_s();
  if (r == nullptr) return AR_ERR_CUDA;
  r->comm = comm;
  r->P = P;
  r->ntensors = T;
  r->dtype = grads->dtype;
  r->sgd = sgd != nullptr;
  r->bucket_of.assign(size_t(T), 0);
  r->marked.assign(size_t(T), 0);
  std::vector<size_t> nbytes(static_cast<size_t>(T));
  for (int t = 0; t < T; ++t) nbytes[t] = grads->numel[t] * es;
  int nb = 0;
  if (ar_bucket_plan(T, nbytes.data(), cap_bytes, r->bucket_of.data(), &nb) != AR_OK) {
    delete r;
    return AR_ERR_INVALID_ARG;
  }
  r->buckets.resize(size_t(nb));
  for (int t = T - 1; t >= 0; --t) r->buckets[r->bucket_of[t]].tensors.push_back(t);

  const bool tma = choose_tma(comm, P, r->sgd, es);
  const uint64_t tile = gar::reduce_tile(P, int(es), tma, r->sgd);
  auto fill = [&](auto& tab, const std::vector<int>& ts, size_t t0, size_t t1) -> bool {
    init_table(tab, P, P, P, 0, rop == AR_MEAN);
    if (tma) set_tma(tab, comm, r->sgd, es);
    if (sgd != nullptr) {
      tab.lr = sgd->lr;
      tab.mu = sgd->momentum;
      tab.write_back = sgd->write_back_grads ? 1 : 0;
    }
    for (size_t i = t0; i < t1; ++i) {
      const int t = ts[i];
      void* const* ptrs = grads->dev_ptrs + size_t(t) * P;
      float* w = sgd ? sgd->master[t] : nullptr;
      float* v = sgd ? sgd->momentum_buf[t] : nullptr;
      float* extra[2] = {w, v};
      if (!add_segment(tab, ptrs, grads->numel[t], tile, vec_flag(ptrs, P, extra, sgd ? 2 : 0), w, v))
        return false;
    }
    return true;
  };
  for (auto& bk : r->buckets) {
    const size_t n = bk.tensors.size();
    bool ok = true;
    if (n <= size_t(CapSmall::kSeg) && n * P <= size_t(CapSmall::kPtr)) {
      bk.small.emplace_back();
      ok = fill(bk.small.back(), bk.tensors, 0, n);
    } else {
      const size_t per = size_t(std::min(CapLarge::kSeg, CapLarge::kPtr / P));
      for (size_t t0 = 0; t0 < n && ok; t0 += per) {
        bk.large.emplace_back();
        ok = fill(bk.large.back(), bk.tensors, t0, std::min(n, t0 + per));
      }
    }
    if (!ok) {
      delete r;
      return AR_ERR_INVALID_ARG;
    }
    bk.pending = int(n);
  }

  int lo = 0, hi = 0;
  if (cudaDeviceGetStreamPriorityRange(&lo, &hi) != cudaSuccess) hi = 0;
  for (int k = 0; k < 2; ++k) {
    if (cudaStreamCreateWithPriority(&r->streams[k], cudaStreamNonBlocking, hi) != cudaSuccess ||
        cudaEventCreateWithFlags(&r->done[k], cudaEventDisableTiming) != cudaSuccess) {
      release(r);
      return AR_ERR_CUDA;
    }
  }
  if (cudaEventCreateWithFlags(&r->join, cudaEventDisableTiming) != cudaSuccess) {
    release(r);
    return AR_ERR_CUDA;
  }
  for (auto& bk : r->buckets)
    if (cudaEventCreateWithFlags(&bk.done, cudaEventDisableTiming) != cudaSuccess) {
      release(r);
      return AR_ERR_CUDA;
    }
  {
    std::lock_guard<std::mutex> lock(g_red_mu);
    g_reducers.insert(r);
  }
  *out = r;
  return AR_OK;
}

ar_status_t ar_reducer_mark_ready(ar_reducer_t r, int tensor, ar_stream_t stream) {
  if (!reducer_live(r) || !is_live(r->comm)) return AR_ERR_STATE;
  if (tensor < 0 || tensor >= r->ntensors) return AR_ERR_INVALID_ARG;
  if (r->marked[tensor]) return AR_ERR_STATE;  // a gradient is marked once per step
  DeviceGuard guard(r->comm->device);
  if (!guard.ok()) return AR_ERR_CUDA;
  r->marked[tensor] = 1;
  ar_reducer_s::Bucket& bk = r->buckets[r->bucket_of[tensor]];
  note_stream(bk, static_cast<cudaStream_t>(stream));
  if (--bk.pending == 0) return launch_ready(r, {r->bucket_of[tensor]});
  return AR_OK;
}

ar_status_t ar_reducer_mark_ready_many(ar_reducer_t r, const int* tensors, int n,
                                       ar_stream_t stream) {
  if (!reducer_live(r) || !is_live(r->comm)) return AR_ERR_STATE;
  if (n < 0 || (n > 0 && tensors == nullptr)) return AR_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i)
    if (tensors[i] < 0 || tensors[i] >= r->ntensors) return AR_ERR_INVALID_ARG;
  DeviceGuard guard(r->comm->device);
  if (!guard.ok()) return AR_ERR_CUDA;
  // Mark all or none: a tensor marked before, or listed twice, undoes this
  // call's marks and refuses it.
  for (int i = 0; i < n; ++i) {
    if (r->marked[tensors[i]]) {
      for (int j = 0; j < i; ++j) r->marked[tensors[j]] = 0;
      return AR_ERR_STATE;
    }
    r->marked[tensors[i]] = 1;
  }
  std::vector<int> ready;
  for (int i = 0; i < n; ++i) {
    const int b = r->bucket_of[tensors[i]];
    ar_reducer_s::Bucket& bk = r->buckets[b];
    note_stream(bk, static_cast<cudaStream_t>(stream));
    if (--bk.pending == 0) ready.push_back(b);
  }
  return ready.empty() ? AR_OK : launch_ready(r, ready);
}

ar_status_t ar_reducer_finalize(ar_reducer_t r, ar_stream_t stream) {
  if (!reducer_live(r) || !is_live(r->comm)) return AR_ERR_STATE;
  DeviceGuard guard(r->comm->device);
  if (!guard.ok()) return AR_ERR_CUDA;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  std::vector<int> rest;
  for (size_t b = 0; b < r->buckets.size(); ++b) {
    auto& bk = r->buckets[b];
    if (!bk.launched && !bk.tensors.empty()) {
      note_stream(bk, s);
      rest.push_back(int(b));
    }
  }
  ar_status_t st = rest.empty() ? AR_OK : launch_ready(r, rest);
  for (int k = 0; k < 2 && st == AR_OK; ++k)
    if (r->used[k] && cudaStreamWaitEvent(s, r->done[k], 0) != cudaSuccess) st = AR_ERR_CUDA;
  if (st == AR_OK && r->direct && r->direct_stream != s &&
      (cudaEventRecord(r->join, r->direct_stream) != cudaSuccess ||
       cudaStreamWaitEvent(s, r->join, 0) != cudaSuccess))
    st = AR_ERR_CUDA;
  for (auto& bk : r->buckets) {
    bk.pending = int(bk.tensors.size());
    bk.launched = false;
    bk.direct = false;
    bk.mark_streams.clear();
  }
  std::fill(r->marked.begin(), r->marked.end(), 0);
  r->used[0] = r->used[1] = false;
  r->direct = false;
  return st;
}

ar_status_t ar_reducer_wait_bucket(ar_reducer_t r, int bucket, ar_stream_t stream) {
  if (!reducer_live(r) || !is_live(r->comm)) return AR_ERR_STATE;
  if (bucket < 0 || bucket >= int(r->buckets.size())) return AR_ERR_INVALID_ARG;
  const ar_reducer_s::Bucket& bk = r->buckets[bucket];
  if (!bk.launched) return AR_ERR_STATE;
  DeviceGuard guard(r->comm->device);
  if (!guard.ok()) return AR_ERR_CUDA;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (bk.direct) {
    // Launched on its marking stream: already ordered for that stream; any
    // other stream waits for an event recorded there now.
    if (bk.direct_stream == s) return AR_OK;
    if (cudaEventRecord(bk.done, bk.direct_stream) != cudaSuccess) return AR_ERR_CUDA;
  }
  return cudaStreamWaitEvent(s, bk.done, 0) == cudaSuccess ? AR_OK : AR_ERR_CUDA;
}

ar_status_t ar_reducer_set_sgd(ar_reducer_t r, float lr, float momentum) {
  if (!reducer_live(r)) return AR_ERR_STATE;
  if (!r->sgd) return AR_ERR_INVALID_ARG;
  for (auto& bk : r->buckets) {
    for (auto& t : bk.small) {
      t.lr = lr;
      t.mu = momentum;
    }
    for (auto& t : bk.large) {
      t.lr = lr;
      t.mu = momentum;
    }
  }
  return AR_OK;
}

ar_status_t ar_reducer_info(ar_reducer_t r, int* nbuckets, int* bucket_of) {
  if (!reducer_live(r)) return AR_ERR_STATE;
  if (nbuckets == nullptr) return AR_ERR_INVALID_ARG;
  *nbuckets = int(r->buckets.size());
  if (bucket_of != nullptr)
    for (int t = 0; t < r->ntensors; ++t) bucket_of[t] = r->bucket_of[t];
  return AR_OK;
}

ar_status_t ar_reducer_launches(ar_reducer_t r, uint64_t* launches) {
  if (!reducer_live(r)) return AR_ERR_STATE;
  if (launches == nullptr) return AR_ERR_INVALID_ARG;
  *launches = r->launches;
  return AR_OK;
}

ar_status_t ar_reducer_destroy(ar_reducer_t r) {
  {
    std::lock_guard<std::mutex> lock(g_red_mu);
    if (r == nullptr || g_reducers.erase(r) == 0) return AR_ERR_STATE;
  }
  ar_status_t st = AR_OK;
  {
    DeviceGuard guard(r->comm->device);
    for (int k = 0; k < 2; ++k)
      if (r->streams[k] && cudaStreamSynchronize(r->streams[k]) != cudaSuccess) st = AR_ERR_CUDA;
    release(r);
  }
  return st;
}

}  // extern "C"
