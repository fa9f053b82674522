// gar_kernels.cuh -- the two kernel families of the library.
//
// k_reduce: the rank-ordered reduction over P replica pointers.  One launch
// covers a list of "segments" -- a flat all-reduce is one segment, a
// reduce-scatter is P segments (one per shard), a gradient bucket is one
// segment per tensor.  Each segment has P source pointers and ndst
// destination pointers (every replica for an all-reduce, the owning rank
// for a reduce-scatter) and optionally fp32 master-weight / momentum arrays
// for the fused SGD step.
//
// k_copy: one source, several destinations (all-gather: one segment per
// source shard; broadcast: one segment from the root).
//
// Work is cut into tiles of kThreads * U 16-byte vectors of one segment.
// The host launches one CTA per tile (grid_per_tile), so the block
// scheduler hands the tiles out in order; the loops still stride by the
// grid, which covers a table with more tiles than a grid may hold.  The
// segment table travels by value in the kernel's parameter space
// (__grid_constant__), so a launch needs no device-side table and no copy.
#pragma once

#include "gar_device.cuh"

namespace gar {

// The kernel specialisation that serves P ranks: P itself, for every P from
// 1 to kMaxRanks -- registers for exactly P ranks, loops of exactly P, and a
// Mean over a P that is not a power of two divides by a compile-time
// constant.  (The register-staged kernels no longer use the runtime-P form
// Ranks<0>; the bulk-copy pipeline keeps it for P outside 2, 4, 8.)
//
// Kernels sized for the largest P of a class of rank counts, with P read at
// run time, paid for registers they did not use: the last no_sync
// micro-batch at P = 5 took 149 registers in the 8-rank kernel, 17 % of the
// SM's warps active and 79 % of DRAM throughput on GB300 (0.94 of the copy
// peak; 1.03 with the kernel for exactly 5 ranks).
__host__ __device__ constexpr int rank_class(int P) { return P; }

// Vectors per thread per tile: enough 16-byte loads in flight per thread
// (P * U * 16 bytes) to cover HBM latency, bounded by registers: 4 for up
// to 4 ranks, 2 for up to 8, 1 above (at 12 ranks, U = 1 took 80 registers
// and 3 CTAs per SM against 101 and 2 with U = 2: 0.91 -> 1.03 of the copy
// peak on GB300 at 128 MiB per replica).
__host__ __device__ constexpr int unroll_for(int PT) {
  return (PT <= 0 || PT > 8) ? 1 : (PT <= 4 ? 4 : 2);
}
// With the fused SGD step each vector also carries its fp32 master weights
// and momentum (2 x E floats), all loaded up front: 2 vectors per thread for
// up to 8 ranks (measured on GB300 for P = 8 on the ViT-B/16 buckets: 0.982
// of the copy peak back to back against 0.978 with 1), 1 beyond, where 2
// would take one CTA per SM (168 registers at 12 ranks).
__host__ __device__ constexpr int unroll_for_sgd(int PT) {
  return (PT <= 0 || PT > 8) ? 1 : 2;  // 2 for up to 8 ranks, 1 above
}
// Copy vectors per thread: 4 (16 KB tiles) for large copies.  The windowed
// copies below are bound by the work each CTA does per item, which a
// larger tile spreads over twice the bytes: on GB300 at 256 MiB per
// replica, broadcast P = 8 1.09 of the copy peak against 0.97 with 2
// vectors (same items, one destination each), all-gather P = 4 1.05
// against 0.93.  Smaller copies take fewer vectors per thread, so that a
// few MB still spread over every SM (copy_unroll_for).
constexpr int kCopyUnroll = 4;

// Segment table capacities: a flat all-reduce (one segment) uses a 400-byte
// parameter block, small launches (<= 16 segments) about 5 KB, large ones
// (<= 256 segments) about 25 KB, inside the 32,764-byte kernel-parameter
// limit; the smaller the block, the cheaper the launch.
struct CapTiny { static constexpr int kSeg = 1, kPtr = 2 * kMaxRanks; };  // one flat all-reduce
struct CapSmall { static constexpr int kSeg = 16, kPtr = 512; };
struct CapLarge { static constexpr int kSeg = 256, kPtr = 2048; };

enum : uint32_t { kSegVec = 1u };  // all pointers of the segment 16-byte aligned

template <class Cap>
struct SegTable {
  uint32_t nseg;              // segments in this launch
  uint32_t ntiles;            // total tiles (= tile0[nseg])
  int np;                     // P: source pointers per segment (k_reduce)
  int ndst;                   // destination pointers per segment
  int stride;                 // pointers per segment in ptr[]
  int dst_off;                // index of the first destination within a segment
  int mean;                   // divide by P
  int write_back;             // SGD: also store the reduced gradient
  int store_w;                // SGD: store the updated weights (rounded) instead
  float lr, mu;               // SGD hyper-parameters
  float scale;                // accumulation: factor on each micro-batch gradient
  int first;                  // accumulation: 1 = overwrite the accumulators
  int unroll;                 // k_reduce: 0 = the kernel's own unroll, 1 = one vector per thread
  int dgroup;                 // k_copy: destinations per windowed item (0 = the classic order)
  int stages;                 // bulk-copy kernel: shared-memory stages
  uint32_t stage_bytes;       // bulk-copy kernel: bytes per stage
  uint32_t* status;           // the comm's device status word (bounded waits)
  uint32_t tile0[Cap::kSeg + 1];  // first tile of each segment; tile0[nseg] = ntiles
  uint64_t numel[Cap::kSeg];      // elements (k_reduce) or bytes (k_copy) per segment
  uint32_t flags[Cap::kSeg];
  float* master[Cap::kSeg];       // SGD fp32 weights (k_reduce with SGD)
  float* mom[Cap::kSeg];          // SGD fp32 momentum
  void* ptr[Cap::kPtr];           // segment s: ptr[s*stride + 0 .. stride)
};

// The segment that holds `tile`: the last s >= from with tile0[s] <= tile
// (tile0 is non-decreasing, tile0[nseg] = ntiles; an empty segment's
// successor starts at the same tile, so empty segments are never chosen).
// A CTA may start at any tile, so this is a binary search, not a walk.
template <class Cap>
__device__ __forceinline__ uint32_t seg_of(const SegTable<Cap>& a, uint32_t tile, uint32_t from) {
  uint32_t lo = from, hi = a.nseg;  // tile0[lo] <= tile < tile0[hi]
  while (hi - lo > 1) {
    const uint32_t mid = (lo + hi) >> 1;
    if (a.tile0[mid] <= tile) lo = mid;
    else hi = mid;
  }
  return lo;
}

// Debug-build checks of a tile's segment (see GAR_CHECK): s is a segment of
// the launch whose tile range holds `tile`, its pointers lie inside the
// table, and its tile count is exactly what its element count needs at
// `per_tile` elements (or bytes) per tile -- the host and the kernel agree
// on the tile size.
template <class Cap>
__device__ __forceinline__ void check_segment(const SegTable<Cap>& a, uint32_t s, uint32_t tile,
                                              uint64_t per_tile) {
#if GAR_DEBUG
  const bool ok = s < a.nseg && s < uint32_t(Cap::kSeg) && a.tile0[s] <= tile &&
                  tile < a.tile0[s + 1] && (uint64_t(s) + 1) * a.stride <= uint64_t(Cap::kPtr) &&
                  a.tile0[s + 1] - a.tile0[s] == (a.numel[s] + per_tile - 1) / per_tile;
  if (!ok && a.status != nullptr) atomicOr(a.status, kStatusBounds);
  if (!ok) asm volatile("exit;");
#else
  (void)a;
  (void)s;
  (void)tile;
  (void)per_tile;
#endif
}

// --------------------------------------------------------------- reduce

// SGD on one vector's E elements, w and v already loaded (E / 4 float4
// each); stores the updated w and v.
template <class D>
__device__ __forceinline__ void sgd_vec(const float (&g)[D::kElems], float4 (&w4)[D::kElems / 4],
                                        float4 (&v4)[D::kElems / 4], float* w, float* v,
                                        uint64_t e0, float lr, float mu) {
#pragma unroll
  for (int q = 0; q < D::kElems / 4; ++q) {
    float* wq = &w4[q].x;
    float* vq = &v4[q].x;
#pragma unroll
    for (int k = 0; k < 4; ++k) sgd_step(g[4 * q + k], lr, mu, wq[k], vq[k]);
    st_f4(v + e0 + 4 * q, v4[q]);
    st_f4(w + e0 + 4 * q, w4[q]);
  }
}

// UO > 0 overrides the unroll (the host's tile size follows the table's
// `unroll`, which selects the kernel).
template <class D, int PT, bool SGD, class Cap, int UO = 0>
__global__ void __launch_bounds__(kThreads)
    k_reduce(const __grid_constant__ SegTable<Cap> a) {
  constexpr int U = UO > 0 ? UO : (SGD ? unroll_for_sgd(PT) : unroll_for(PT));
  constexpr int E = D::kElems;
  constexpr int MAXP = Ranks<PT>::kMax;
  constexpr int WV = SGD ? E / 4 : 1;  // float4 groups of w (and of v) per vector
  constexpr uint64_t kTileVec = uint64_t(U) * kThreads;
  const int np = a.np;
  const bool mean = a.mean != 0;
  griddep_launch_dependents();
  uint32_t s = 0;
  for (uint32_t tile = blockIdx.x; tile < a.ntiles; tile += gridDim.x) {
    s = seg_of(a, tile, s);
    check_segment(a, s, tile, kTileVec * E);
    GAR_CHECK(np <= a.stride && a.dst_off + a.ndst <= a.stride, a.status);
    const uint64_t n = a.numel[s];
    void* const* seg = a.ptr + uint64_t(s) * a.stride;
    void* const* dst = seg + a.dst_off;
    const uint64_t lt = tile - a.tile0[s];
    const bool do_store = !SGD || a.write_back;
    float* w = SGD ? a.master[s] : nullptr;
    float* v = SGD ? a.mom[s] : nullptr;
    GAR_CHECK(!SGD || (w != nullptr && v != nullptr), a.status);
    const bool vec = (a.flags[s] & kSegVec) != 0;
    const void* src[MAXP];
#pragma unroll
    for (int r = 0; r < MAXP; ++r)
      if (Ranks<PT>::has(r, np)) src[r] = seg[r];
    // Everything above reads the launch's own table (kernel parameters),
    // nothing the previous kernel writes: under programmatic dependent
    // launch it runs while that kernel drains.  Memory is touched only after
    // the wait (which returns at once after its first call).
    griddep_wait();

    if (vec) {
      const uint64_t nvec = n / E;
      const uint64_t v0 = lt * kTileVec + threadIdx.x;
      // Every load of the tile (all replicas, and w, v with SGD) is issued
      // before any arithmetic or store.
      uint4 in[U][MAXP];
      float4 w4[U][WV], v4[U][WV];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint64_t vi = v0 + uint64_t(u) * kThreads;
        if (vi < nvec) {
          GAR_CHECK((vi + 1) * E <= n, a.status);
#pragma unroll
          for (int r = 0; r < MAXP; ++r)
            if (Ranks<PT>::has(r, np))
              in[u][r] = ld_stream(static_cast<const uint4*>(src[r]) + vi);
          if constexpr (SGD) {
#pragma unroll
            for (int q = 0; q < WV; ++q) {
              w4[u][q] = ld_f4(w + vi * E + 4 * q);
              v4[u][q] = ld_f4(v + vi * E + 4 * q);
            }
          }
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (v0 + uint64_t(u) * kThreads < nvec) {
#pragma unroll
          for (int r = 0; r < MAXP; ++r)
            if (Ranks<PT>::has(r, np)) reg_fence(in[u][r]);
          if constexpr (SGD) {
#pragma unroll
            for (int q = 0; q < WV; ++q) {
              reg_fence(w4[u][q]);
              reg_fence(v4[u][q]);
            }
          }
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint64_t vi = v0 + uint64_t(u) * kThreads;
        if (vi < nvec) {
          float g[E];
          reduce_vec<D, PT, !SGD>(in[u], np, mean, g);
          if constexpr (SGD) {
            sgd_vec<D>(g, w4[u], v4[u], w, v, vi * E, a.lr, a.mu);
            if (a.store_w) {  // the sharded step: every rank gets the new weights
#pragma unroll
              for (int q = 0; q < WV; ++q) {
                g[4 * q] = w4[u][q].x;
                g[4 * q + 1] = w4[u][q].y;
                g[4 * q + 2] = w4[u][q].z;
                g[4 * q + 3] = w4[u][q].w;
              }
            }
          }
          if (do_store) {
            const uint4 out = D::pack(g);
            for (int d = 0; d < a.ndst; ++d) st_stream(static_cast<uint4*>(dst[d]) + vi, out);
          }
        }
      }
      // The last tile of a segment also takes its ragged tail (< E elements).
      if (lt + 1 == a.tile0[s + 1] - a.tile0[s]) {
        const uint64_t i = nvec * E + threadIdx.x;
        if (i < n) {
          GAR_CHECK(i - nvec * E < uint64_t(E), a.status);
          float g = reduce_scalar<D, PT>(seg, i, np, mean);
          if constexpr (SGD) {
            sgd_step(g, a.lr, a.mu, w[i], v[i]);
            if (a.store_w) g = w[i];
          }
          if (do_store)
            for (int d = 0; d < a.ndst; ++d) D::store1(dst[d], i, g);
        }
      }
    } else {
      // Unaligned segment: the same tile of elements with scalar accesses.
      const uint64_t e0 = lt * kTileVec * E;
      for (uint64_t k = threadIdx.x; k < kTileVec * E; k += kThreads) {
        const uint64_t i = e0 + k;
        if (i >= n) break;
        GAR_CHECK(i < n, a.status);
        float g = reduce_scalar<D, PT>(seg, i, np, mean);
        if constexpr (SGD) {
          sgd_step(g, a.lr, a.mu, w[i], v[i]);
          if (a.store_w) g = w[i];
        }
        if (do_store)
          for (int d = 0; d < a.ndst; ++d) D::store1(dst[d], i, g);
      }
    }
  }
}

// ----------------------------------------------------------------- copy
// numel[s] is in bytes (always even: elements are 2 or 4 bytes); segment s
// has flags[s] >> 8 destinations (an in-place all-gather skips the shard
// that is already in place).
//
// Windowed copies (a.ndst = D > 0, the most destinations of any segment;
// the host picks them for copies of at least kCopyWindowBytes): one
// CTA copies one tile of a segment to a group of a.dgroup = G of its
// destinations, and the work items run group by group within windows of
// kCopyWindow tiles -- item b is tile (b / (W NG)) W + b % W for destination
// group (b / W) % NG, NG = ceil(D / G).  The CTAs in flight then write a
// few destinations at a time, while the window's source tiles, read from
// HBM for the first group, are read again from L2: the source is loaded
// with an L2 evict-last policy so that the L2's replacement keeps it
// (without the hint the reuse depended on what had run before), and the CTA
// of a tile's last group returns the tile's lines to normal priority.
//
// The host takes G = ceil(D / 4): about four groups per window.  Measured on
// GB300 at 256 MiB per replica, of the copy peak, back to back (4 vectors per
// thread): all-gather P = 8 (D = 7) G = 1 / 2 / 3 / 4: 1.07 / 1.09 / 1.07 /
// 1.04, every destination from one CTA (the classic order below) 0.99;
// all-gather P = 4 (D = 3) G = 1 / 2 / 3: 1.05 / 1.03 / 1.01, classic 1.01;
// broadcast P = 8, G = 1: 1.09.  ncu on the classic order: 15 % issue
// activity but 83 % DRAM throughput (seven write streams at once); on
// windowed items of one destination and 8 KB, 70 % issue activity, the
// per-item work (segment search, window arithmetic, priority reset) limiting
// the rate, and the same DRAM bytes and L2 hits as the broadcast.
//
// Other copies (a.ndst = 0): each CTA copies one tile to every destination
// of its segment (small copies, below kCopyWindowBytes: 0.92 against
// 0.87 for single broadcasts from a cold L2 at 16 MiB per replica in the
// windowed order, as fewer CTAs carry the same bytes).
constexpr uint64_t kCopyWindow = 1024;          // tiles per window: 16 MB of source
constexpr uint64_t kCopyWindowBytes = 32u << 20;  // copies of at least this much source

// 16-byte load that asks L2 to keep the line (policy from createpolicy).
__device__ __forceinline__ uint4 ld_keep(const uint4* p, uint64_t policy) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p), "l"(policy));
  return r;
}

template <class Cap, int U>
__global__ void __launch_bounds__(kThreads) k_copy(const __grid_constant__ SegTable<Cap> a) {
  constexpr uint64_t kTileVec = uint64_t(U) * kThreads;
  griddep_launch_dependents();
  if (a.ndst == 0) {  // small copies: one tile to every destination per CTA
    for (uint32_t tile = blockIdx.x; tile < a.ntiles; tile += gridDim.x) {
      const uint32_t s = seg_of(a, tile, 0);
      check_segment(a, s, tile, kTileVec * 16);
      const uint64_t nbytes = a.numel[s];
      void* const* seg = a.ptr + uint64_t(s) * a.stride;
      const void* src = seg[0];
      void* const* dst = seg + a.dst_off;
      const uint64_t lt = tile - a.tile0[s];
      const int nd = int(a.flags[s] >> 8);
      GAR_CHECK(a.dst_off + nd <= a.stride && nbytes % 2 == 0, a.status);
      griddep_wait();  // the table lookups above overlap the previous kernel's drain
      if (a.flags[s] & kSegVec) {
        const uint64_t nvec = nbytes / 16;
        const uint64_t v0 = lt * kTileVec + threadIdx.x;
        uint4 x[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const uint64_t vi = v0 + uint64_t(u) * kThreads;
          GAR_CHECK(vi >= nvec || (vi + 1) * 16 <= nbytes, a.status);
          if (vi < nvec) x[u] = ld_stream_ro(static_cast<const uint4*>(src) + vi);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const uint64_t vi = v0 + uint64_t(u) * kThreads;
          if (vi < nvec)
            for (int d = 0; d < nd; ++d) st_stream(static_cast<uint4*>(dst[d]) + vi, x[u]);
        }
        if (lt + 1 == a.tile0[s + 1] - a.tile0[s]) {
          const uint64_t h = (nvec * 16) / 2 + threadIdx.x;  // 2-byte units of the tail
          if (h < nbytes / 2) {
            GAR_CHECK(2 * h + 2 <= nbytes, a.status);
            const uint16_t x1 = static_cast<const uint16_t*>(src)[h];
            for (int d = 0; d < nd; ++d) static_cast<uint16_t*>(dst[d])[h] = x1;
          }
        }
      } else {
        const uint64_t h0 = lt * kTileVec * 8;  // 2-byte units per tile
        for (uint64_t k = threadIdx.x; k < kTileVec * 8; k += kThreads) {
          const uint64_t h = h0 + k;
          if (h >= nbytes / 2) break;
          GAR_CHECK(2 * h + 2 <= nbytes, a.status);
          const uint16_t x1 = static_cast<const uint16_t*>(src)[h];
          for (int d = 0; d < nd; ++d) static_cast<uint16_t*>(dst[d])[h] = x1;
        }
      }
    }
    return;
  }
  uint64_t keep;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(keep));
  const uint32_t D = uint32_t(a.ndst);
  const uint32_t G = a.dgroup > 0 ? uint32_t(a.dgroup) : 1u;  // destinations per item
  const uint32_t NG = (D + G - 1) / G;                        // destination groups
  const uint64_t items = (uint64_t(a.ntiles) + kCopyWindow - 1) / kCopyWindow * kCopyWindow * NG;
  for (uint64_t b = blockIdx.x; b < items; b += gridDim.x) {
    // (window, destination group) pair and tile: a shift and one 32-bit
    // division (pairs number below 2^32: tiles / kCopyWindow * NG).
    const uint32_t q = uint32_t(b / kCopyWindow);
    const uint32_t win = q / NG, g = q - win * NG;
    const uint64_t tile = uint64_t(win) * kCopyWindow + b % kCopyWindow;
    if (tile >= a.ntiles) continue;
    const uint32_t s = seg_of(a, uint32_t(tile), 0);
    check_segment(a, s, uint32_t(tile), kTileVec * 16);
    const uint32_t nd = a.flags[s] >> 8;
    const uint32_t d0 = g * G;
    if (d0 >= nd) continue;
    const uint32_t d1 = min(d0 + G, nd);
    GAR_CHECK(a.dst_off + int(d1) <= a.stride, a.status);
    const uint64_t nbytes = a.numel[s];
    void* const* seg = a.ptr + uint64_t(s) * a.stride;
    const void* src = seg[0];
    void* const* outs = seg + a.dst_off;
    const uint64_t lt = tile - a.tile0[s];
    griddep_wait();  // the table lookups above overlap the previous kernel's drain
    if (a.flags[s] & kSegVec) {
      const uint64_t nvec = nbytes / 16;
      const uint64_t v0 = lt * kTileVec + threadIdx.x;
      uint4 x[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint64_t vi = v0 + uint64_t(u) * kThreads;
        GAR_CHECK(vi >= nvec || (vi + 1) * 16 <= nbytes, a.status);
        if (vi < nvec) x[u] = ld_keep(static_cast<const uint4*>(src) + vi, keep);
      }
      for (uint32_t d = d0; d < d1; ++d) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const uint64_t vi = v0 + uint64_t(u) * kThreads;
          if (vi < nvec) st_stream(static_cast<uint4*>(outs[d]) + vi, x[u]);
        }
      }
      if (d1 == nd) {
        // The tile's last destination: its source lines go back to normal
        // eviction priority.  Lines are 128 bytes: each address is the
        // 128-byte boundary at or below a byte of the tile (so inside the
        // source's allocation); the instruction changes no data.
        const uint4* base = static_cast<const uint4*>(src);
        const uint64_t first = lt * kTileVec, last = min(first + kTileVec, nvec);
        const uintptr_t lo = reinterpret_cast<uintptr_t>(base + first) & ~uintptr_t(127);
        const uintptr_t hi = reinterpret_cast<uintptr_t>(base + last);
        for (uintptr_t p = lo + uintptr_t(threadIdx.x) * 128; p < hi; p += uintptr_t(kThreads) * 128)
          asm volatile("applypriority.global.L2::evict_normal [%0], 128;" ::"l"(p) : "memory");
      }
      if (lt + 1 == a.tile0[s + 1] - a.tile0[s]) {
        const uint64_t h = (nvec * 16) / 2 + threadIdx.x;  // 2-byte units of the tail
        GAR_CHECK(h >= nbytes / 2 || 2 * h + 2 <= nbytes, a.status);
        if (h < nbytes / 2) {
          const uint16_t x1 = static_cast<const uint16_t*>(src)[h];
          for (uint32_t d = d0; d < d1; ++d) static_cast<uint16_t*>(outs[d])[h] = x1;
        }
      }
    } else {
      const uint64_t h0 = lt * kTileVec * 8;  // 2-byte units per tile
      for (uint64_t k = threadIdx.x; k < kTileVec * 8; k += kThreads) {
        const uint64_t h = h0 + k;
        if (h >= nbytes / 2) break;
        GAR_CHECK(2 * h + 2 <= nbytes, a.status);
        const uint16_t x1 = static_cast<const uint16_t*>(src)[h];
        for (uint32_t d = d0; d < d1; ++d) static_cast<uint16_t*>(outs[d])[h] = x1;
      }
    }
  }
}

// ------------------------------------------------------- accumulation
// DDP's no_sync gradient accumulation.  k_accumulate (a micro-batch before
// the last, no communication): segment = one (tensor, rank) pair, ptr[0] =
// the gradient (D), ptr[1] = its fp32 accumulator; per element, with
// s = fl(scale * g):  acc = first ? s : fl(acc + s).  The first micro-batch
// (no accumulator to read) is a kernel of its own, FIRST = true: fewer
// registers, 8 CTAs per SM, and 0.92 of the copy peak on GB300 against 0.85
// as a runtime branch of one kernel (one 25 MiB bf16 bucket, P = 8).
//
// A thread works on quads (4 consecutive elements) kThreads apart, so every
// warp-wide access covers one contiguous span: 8 or 16 bytes of gradient
// and 16 bytes of accumulator per lane.  With a bf16 vector of 8 elements
// per thread instead, each fp32 access wrote or read half of every 32-byte
// sector it touched (16 bytes at a 32-byte stride), and the L1-to-L2 write
// path ran at 72-82 % of its peak under ncu.  Measured on GB300 (one 25 MiB
// bf16 bucket, of the copy peak, back to back / from a cold L2): the first
// micro-batch at P = 8 rose from 0.94 / 0.92 to 1.00 / 1.02, at P = 2 from
// 0.82 / 0.76 to 0.90 / 0.95; later micro-batches at P = 8 from 1.03 / 1.04
// to 1.03 / 1.06.  Vectors per thread: 2 measured best for both kernels in
// the vector form (later micro-batches 1.03 against 1.02 with 4 and 1.00
// with 8; the first 0.92 against 0.78 and 0.84).
constexpr int kAccUnroll = 2;

template <class D, class Cap, bool FIRST>
__global__ void __launch_bounds__(kThreads) k_accumulate(const __grid_constant__ SegTable<Cap> a) {
  constexpr int J = kAccUnroll * D::kElems / 4;  // quads per thread per tile
  constexpr uint64_t kTileQuads = uint64_t(J) * kThreads;
  griddep_launch_dependents();
  uint32_t s = 0;
  for (uint32_t tile = blockIdx.x; tile < a.ntiles; tile += gridDim.x) {
    s = seg_of(a, tile, s);
    check_segment(a, s, tile, kTileQuads * 4);
    GAR_CHECK(a.stride >= 2, a.status);
    const uint64_t n = a.numel[s];
    const void* g = a.ptr[uint64_t(s) * a.stride];
    float* acc = static_cast<float*>(a.ptr[uint64_t(s) * a.stride + 1]);
    const uint64_t lt = tile - a.tile0[s];
    griddep_wait();  // the table lookups above overlap the previous kernel's drain
    if (a.flags[s] & kSegVec) {
      const uint64_t nq = n / 4;
      const uint64_t q0 = lt * kTileQuads + threadIdx.x;
      typename D::Quad x[J];
      float4 a4[J];
#pragma unroll
      for (int j = 0; j < J; ++j) {
        const uint64_t qi = q0 + uint64_t(j) * kThreads;
        if (qi < nq) {
          GAR_CHECK(4 * qi + 4 <= n, a.status);
          x[j] = D::ld_quad(g, qi);
          a4[j] = FIRST ? make_float4(0.f, 0.f, 0.f, 0.f) : ld_f4(acc + 4 * qi);
        }
      }
#pragma unroll
      for (int j = 0; j < J; ++j) {
        if (q0 + uint64_t(j) * kThreads < nq) {
          reg_fence(x[j]);
          reg_fence(a4[j]);
        }
      }
#pragma unroll
      for (int j = 0; j < J; ++j) {
        const uint64_t qi = q0 + uint64_t(j) * kThreads;
        if (qi < nq) {
          float f[4];
          D::unpack_quad(x[j], f);
          float* av = &a4[j].x;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float sv = __fmul_rn(a.scale, f[k]);
            av[k] = FIRST ? sv : __fadd_rn(av[k], sv);
          }
          st_f4(acc + 4 * qi, a4[j]);
        }
      }
      if (lt + 1 == a.tile0[s + 1] - a.tile0[s]) {
        const uint64_t i = nq * 4 + threadIdx.x;
        if (i < n) {
          GAR_CHECK(i - nq * 4 < 4, a.status);
          const float sv = __fmul_rn(a.scale, D::load1(g, i));
          acc[i] = FIRST ? sv : __fadd_rn(acc[i], sv);
        }
      }
    } else {
      const uint64_t e0 = lt * kTileQuads * 4;
      for (uint64_t k = threadIdx.x; k < kTileQuads * 4; k += kThreads) {
        const uint64_t i = e0 + k;
        if (i >= n) break;
        GAR_CHECK(i < n, a.status);
        const float sv = __fmul_rn(a.scale, D::load1(g, i));
        acc[i] = FIRST ? sv : __fadd_rn(acc[i], sv);
      }
    }
  }
}

// k_reduce_accumulated (the last micro-batch): segment = one tensor, ptr[0
// .. P) = its gradient replicas (also the destinations), ptr[P .. 2P) = the
// replicas' fp32 accumulators.  Rank r's total is t_r = first ? s_r :
// fl(acc_r + s_r) with s_r = fl(scale * g_r); the totals are reduced in rank
// order exactly as k_reduce reduces gradients, then the optional SGD step
// and the stores follow as in k_reduce.  The accumulators are only read.
//
// A thread takes one vector at a time and issues every load of it (the
// gradients, the accumulators, and w and v with SGD) before any arithmetic.
// Loading w and v only after the reduction cost a second round trip to HBM
// per vector.  Above 8 ranks a kernel holds 162-252 registers, room for
// one 256-thread CTA per SM; those kernels run 128-thread CTAs that take the
// tile's vectors in two turns, so that an SM holds two CTAs whose phases
// overlap.  Measured on GB300, one 25 MiB bf16 bucket per replica, Mean +
// SGD, from a cold L2, as fractions of the copy peak:
//   P                        2     3     4     5     6     8     11    16
//   w, v after the reduction 0.62  0.62  0.69  -     0.77  1.01  0.86  0.94
//   w, v up front            1.01  0.92  1.03  -     0.80  1.05  0.94  0.98
//   kernels then sized for up to 4, 8, 12 or 16 ranks with P read at run
//   time, 128-thread CTAs    1.01  0.97  1.03  0.94  0.96  1.04  0.95  1.00
//   a kernel for every P     1.00  1.04  1.03  1.03  1.04  1.05  1.02  1.02
// (The runtime-P kernels with 256-thread CTAs measured 0.76 and 0.80 at
// P = 5 and 6.)  The quad layout of k_accumulate (fp32 accesses contiguous
// across a warp) was tried here too: from a cold L2 it gained at P = 2 and 4
// (1.01 -> 1.05, 1.03 -> 1.05) but back to back nothing, and the runtime-P
// kernels lost 0.02-0.04 to the 10-16 registers it added, so the vector
// layout stays.
__host__ __device__ constexpr int acc_threads(int PT) {
  return (PT <= 0 || PT > 8) ? kThreads / 2 : kThreads;
}

template <int PT>
__device__ __forceinline__ float total_of(float g, float acc, float scale, bool first) {
  const float sv = __fmul_rn(scale, g);
  return first ? sv : __fadd_rn(acc, sv);
}

template <class D, int PT, bool SGD>
__device__ __forceinline__ void reduce_accumulated_vec(void* const* seg, int np, uint64_t vi,
                                                       float* w, float* v, float scale, float lr,
                                                       float mu, bool mean, bool first, bool do_store) {
  constexpr int E = D::kElems;
  constexpr int MAXP = Ranks<PT>::kMax;
  constexpr int WV = SGD ? E / 4 : 1;
  uint4 in[MAXP];
  float4 ac[MAXP][E / 4];
  float4 w4[WV], v4[WV];
#pragma unroll
  for (int r = 0; r < MAXP; ++r)
    if (Ranks<PT>::has(r, np)) {
      in[r] = ld_stream(static_cast<const uint4*>(seg[r]) + vi);
      if (!first) {
#pragma unroll
        for (int q = 0; q < E / 4; ++q)
          ac[r][q] = ld_f4(static_cast<const float*>(seg[np + r]) + vi * E + 4 * q);
      }
    }
  if constexpr (SGD) {
#pragma unroll
    for (int q = 0; q < WV; ++q) {
      w4[q] = ld_f4(w + vi * E + 4 * q);
      v4[q] = ld_f4(v + vi * E + 4 * q);
    }
  }
#pragma unroll
  for (int r = 0; r < MAXP; ++r)
    if (Ranks<PT>::has(r, np)) {
      reg_fence(in[r]);
      if (!first) {
#pragma unroll
        for (int q = 0; q < E / 4; ++q) reg_fence(ac[r][q]);
      }
    }
  if constexpr (SGD) {
#pragma unroll
    for (int q = 0; q < WV; ++q) {
      reg_fence(w4[q]);
      reg_fence(v4[q]);
    }
  }
  float g[E];
#pragma unroll
  for (int r = 0; r < MAXP; ++r) {
    if (Ranks<PT>::has(r, np)) {
      float x[E];
      D::unpack(in[r], x);
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float t = total_of<PT>(x[e], first ? 0.f : (&ac[r][e / 4].x)[e % 4], scale, first);
        g[e] = r == 0 ? t : __fadd_rn(g[e], t);
      }
    }
  }
  if (mean) {
#pragma unroll
    for (int e = 0; e < E; ++e) g[e] = mean_of<PT, E == 8>(g[e], np);
  }
  if constexpr (SGD) sgd_vec<D>(g, w4, v4, w, v, vi * E, lr, mu);
  if (do_store) {
    const uint4 out = D::pack(g);
    for (int d = 0; d < np; ++d) st_stream(static_cast<uint4*>(seg[d]) + vi, out);
  }
}

template <class D, int PT, bool SGD, class Cap>
__global__ void __launch_bounds__(kThreads)
    k_reduce_accumulated(const __grid_constant__ SegTable<Cap> a) {
  constexpr int E = D::kElems;
  constexpr int MAXP = Ranks<PT>::kMax;
  constexpr int T = acc_threads(PT);
  const int np = a.np;
  const bool mean = a.mean != 0, first = a.first != 0;
  griddep_launch_dependents();
  uint32_t s = 0;
  for (uint32_t tile = blockIdx.x; tile < a.ntiles; tile += gridDim.x) {
    s = seg_of(a, tile, s);
    check_segment(a, s, tile, uint64_t(kThreads) * E);
    GAR_CHECK(2 * np <= a.stride, a.status);
    const uint64_t n = a.numel[s];
    void* const* seg = a.ptr + uint64_t(s) * a.stride;
    const uint64_t lt = tile - a.tile0[s];
    const bool do_store = !SGD || a.write_back;
    float* w = SGD ? a.master[s] : nullptr;
    float* v = SGD ? a.mom[s] : nullptr;
    GAR_CHECK(!SGD || (w != nullptr && v != nullptr), a.status);
    griddep_wait();  // the table lookups above overlap the previous kernel's drain
    if (a.flags[s] & kSegVec) {
      const uint64_t nvec = n / E;
#pragma unroll
      for (int turn = 0; turn < kThreads / T; ++turn) {
        const uint64_t vi = lt * kThreads + uint64_t(turn) * T + threadIdx.x;
        GAR_CHECK(vi >= nvec || (vi + 1) * E <= n, a.status);
        if (vi < nvec)
          reduce_accumulated_vec<D, PT, SGD>(seg, np, vi, w, v, a.scale, a.lr, a.mu, mean, first,
                                             do_store);
      }
      if (lt + 1 == a.tile0[s + 1] - a.tile0[s]) {
        const uint64_t i = nvec * E + threadIdx.x;
        if (i < n) {
          GAR_CHECK(i - nvec * E < uint64_t(E), a.status);
          float g = 0.f;
          for (int r = 0; r < MAXP; ++r)
            if (Ranks<PT>::has(r, np)) {
              const float t = total_of<PT>(D::load1(seg[r], i),
                                           first ? 0.f : static_cast<const float*>(seg[np + r])[i],
                                           a.scale, first);
              g = r == 0 ? t : __fadd_rn(g, t);
            }
          if (mean) g = mean_of<PT, E == 8>(g, np);
          if constexpr (SGD) sgd_step(g, a.lr, a.mu, w[i], v[i]);
          if (do_store)
            for (int d = 0; d < np; ++d) D::store1(seg[d], i, g);
        }
      }
    } else {
      const uint64_t e0 = lt * uint64_t(kThreads) * E;
      for (uint64_t k = threadIdx.x; k < uint64_t(kThreads) * E; k += T) {
        const uint64_t i = e0 + k;
        if (i >= n) break;
        GAR_CHECK(i < n, a.status);
        float g = 0.f;
        for (int r = 0; r < MAXP; ++r)
          if (Ranks<PT>::has(r, np)) {
            const float t = total_of<PT>(D::load1(seg[r], i),
                                         first ? 0.f : static_cast<const float*>(seg[np + r])[i],
                                         a.scale, first);
            g = r == 0 ? t : __fadd_rn(g, t);
          }
        if (mean) g = mean_of<PT, E == 8>(g, np);
        if constexpr (SGD) sgd_step(g, a.lr, a.mu, w[i], v[i]);
        if (do_store)
          for (int d = 0; d < np; ++d) D::store1(seg[d], i, g);
      }
    }
  }
}

// Tile sizes (elements) of the accumulation kernels.
__host__ __device__ constexpr uint64_t accumulate_tile_elems(int elems_per_vec) {
  return uint64_t(kAccUnroll) * kThreads * elems_per_vec;
}
__host__ __device__ constexpr uint64_t reduce_acc_tile_elems(int elems_per_vec) {
  return uint64_t(kThreads) * elems_per_vec;
}

// Vectors per thread of a copy of `src_bytes` of source: 1 below 8 MiB, 2
// below kCopyWindowBytes, kCopyUnroll (and the windowed order) above.
// Measured on GB300 (broadcast and all-gather, P = 2, 4, 8, of the copy
// peak, one vector / two): at 4 MiB per replica 0.69-0.86 / 0.52-0.63
// replayed from a CUDA graph and the same cold; at 16 MiB 0.91-1.13 /
// 0.93-1.17 graph-replayed, 0.48-0.88 / 0.51-0.95 cold.
__host__ __device__ constexpr int copy_unroll_for(uint64_t src_bytes) {
  return src_bytes < (8u << 20) ? 1 : (src_bytes < kCopyWindowBytes ? 2 : kCopyUnroll);
}

// Tile of the copy kernel, in bytes, for a copy of `src_bytes` of source.
__host__ __device__ constexpr uint64_t copy_tile_bytes(uint64_t src_bytes) {
  return uint64_t(copy_unroll_for(src_bytes)) * kThreads * 16;
}

}  // namespace gar
