// gar_tma.cuh -- the bulk-copy (TMA) pipelined variant of k_reduce.
//
// One CTA per SM, warp-specialised:
//   warp 0 (producer): one lane issues cp.async.bulk global->shared copies
//     of a tile of every replica (and, for the SGD step, of the fp32 master
//     weights and momentum) into a ring of S shared-memory stages; each
//     stage has a "full" mbarrier that completes when all its bytes landed
//     (expect_tx) and an "empty" mbarrier the consumers arrive on.
//   warps 1..8 (consumers): wait for a full stage, read their 16-byte
//     vectors of every replica from shared memory, reduce in fp32 in rank
//     order, release the stage, and store the results straight to global
//     memory (every destination replica, and w, v for SGD).
// While the consumers work on stage k, the copies of stages k+1 .. k+S-1
// are in flight, so the HBM pipe never drains between tiles.
//
// Every wait is bounded: after kWaitLimitNs of waiting the thread records
// AR_ERR_TIMEOUT-style status 1 in the comm's status word, raises a shared
// abort flag and leaves; the producer first waits (also bounded) for the
// copies it issued, so no copy lands in freed shared memory.
//
// Tiles, segments and the unaligned/tail paths are the same as k_reduce's;
// tiles of segments that are not 16-byte aligned are done by the consumers
// with scalar global accesses and use no stage.
#pragma once

#include "gar_kernels.cuh"

namespace gar {

constexpr int kTmaConsumerWarps = 8;
constexpr int kTmaThreads = 32 * (1 + kTmaConsumerWarps);
constexpr int kTmaTileVec = 32 * kTmaConsumerWarps;  // 16-byte vectors per replica per tile
constexpr int kTmaMaxStages = 8;
constexpr uint64_t kWaitLimitNs = 2000000000ull;     // 2 s

// ------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Bounded wait for phase `parity` of barrier `bar`.  Gives up (false) after
// limit_ns, or at once when another thread has raised *abort (abort may be
// null: then only the time limit applies).
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  volatile int* abort,
                                                  uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t k = 1;; ++k) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((k & 255u) == 0) {
      if (abort != nullptr && *abort) return false;
      if (global_timer_ns() - t0 > limit_ns) return false;
    }
  }
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ float4 lds128f(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr));
  return v;
}

// Bytes of one stage: P grad tiles, plus w and v tiles for SGD.
__host__ __device__ constexpr uint32_t tma_grad_tile_bytes() { return uint32_t(kTmaTileVec) * 16; }
__host__ __device__ inline uint32_t tma_stage_bytes(int np, bool sgd, int elems_per_vec) {
  return uint32_t(np) * tma_grad_tile_bytes() +
         (sgd ? 2u * uint32_t(kTmaTileVec) * uint32_t(elems_per_vec) * 4u : 0u);
}

template <class D, int PT, bool SGD, class Cap>
__global__ void __launch_bounds__(kTmaThreads, 1)
    k_reduce_tma(const __grid_constant__ SegTable<Cap> a) {
  constexpr int E = D::kElems;
  constexpr int MAXP = Ranks<PT>::kMax;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kTmaMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kTmaMaxStages];
  __shared__ int abort_flag;

  const int np = a.np;
  const bool mean = a.mean != 0;
  const int S = a.stages;  // 2 .. kTmaMaxStages, chosen on the host
  const uint32_t stage_bytes = a.stage_bytes;
  const uint32_t smem0 = smem_u32(smem_raw);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), kTmaConsumerWarps);
    }
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  griddep_launch_dependents();
  griddep_wait();

  volatile int* abort = &abort_flag;
  uint32_t stage = 0, phase = 0;
  uint32_t seg = 0;

  if (warp == 0) {
    // ----------------------------------------------------------- producer
    if (lane == 0) {
      uint32_t fills[kTmaMaxStages];
      for (int k = 0; k < kTmaMaxStages; ++k) fills[k] = 0;
      bool ok = true;
      for (uint32_t tile = blockIdx.x; tile < a.ntiles; tile += gridDim.x) {
        while (tile >= a.tile0[seg + 1]) ++seg;
        if (!(a.flags[seg] & kSegVec)) continue;
        const uint64_t nvec = a.numel[seg] / E;
        const uint64_t v0 = uint64_t(tile - a.tile0[seg]) * kTmaTileVec;
        if (v0 >= nvec) continue;  // a tile holding only the ragged tail
        const uint64_t nv = nvec - v0 < uint64_t(kTmaTileVec) ? nvec - v0 : uint64_t(kTmaTileVec);
        const uint32_t gbytes = uint32_t(nv) * 16;
        const uint32_t fbytes = SGD ? uint32_t(nv) * E * 4 : 0;
        const uint32_t full = smem_u32(&full_bar[stage]);
        // A fresh barrier counts its preceding phase (parity 1) as complete,
        // so the first S fills do not wait.
        if (!mbar_wait_bounded(smem_u32(&empty_bar[stage]), phase ^ 1, abort)) {
          ok = false;
          break;
        }
        mbar_expect_tx(full, uint32_t(Ranks<PT>::count(np)) * gbytes + 2 * fbytes);
        void* const* ptrs = a.ptr + uint64_t(seg) * a.stride;
        const uint32_t base = smem0 + stage * stage_bytes;
#pragma unroll
        for (int r = 0; r < MAXP; ++r)
          if (Ranks<PT>::has(r, np))
            bulk_g2s(base + r * tma_grad_tile_bytes(),
                     static_cast<const uint4*>(ptrs[r]) + v0, gbytes, full);
        if constexpr (SGD) {
          const uint32_t fb = base + Ranks<PT>::count(np) * tma_grad_tile_bytes();
          bulk_g2s(fb, a.master[seg] + v0 * E, fbytes, full);
          bulk_g2s(fb + kTmaTileVec * E * 4, a.mom[seg] + v0 * E, fbytes, full);
        }
        ++fills[stage];
        if (++stage == uint32_t(S)) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok || *abort) {
        // Giving up: record it, stop the consumers, and wait (bounded, no
        // early exit) until the last fill of every stage has landed, so no
        // bulk copy writes shared memory after the CTA has gone.
        atomicExch(a.status, 1u);
        *abort = 1;
        for (int k = 0; k < S; ++k)
          if (fills[k] > 0) mbar_wait_bounded(smem_u32(&full_bar[k]), (fills[k] - 1) & 1u, nullptr);
      }
    }
    return;
  }

  // ------------------------------------------------------------- consumers
  const int ct = threadIdx.x - 32;  // 0 .. 255
  for (uint32_t tile = blockIdx.x; tile < a.ntiles; tile += gridDim.x) {
    while (tile >= a.tile0[seg + 1]) ++seg;
    const uint64_t n = a.numel[seg];
    void* const* ptrs = a.ptr + uint64_t(seg) * a.stride;
    void* const* dst = ptrs + a.dst_off;
    const bool do_store = !SGD || a.write_back;
    float* w = SGD ? a.master[seg] : nullptr;
    float* v = SGD ? a.mom[seg] : nullptr;
    const uint64_t lt = tile - a.tile0[seg];
    const bool last = lt + 1 == a.tile0[seg + 1] - a.tile0[seg];

    if (a.flags[seg] & kSegVec) {
      const uint64_t nvec = n / E;
      const uint64_t v0 = lt * kTmaTileVec;
      if (v0 < nvec) {
        // Every lane waits; the warp leaves together if any lane gave up.
        const bool ok = mbar_wait_bounded(smem_u32(&full_bar[stage]), phase, abort);
        if (!__all_sync(0xFFFFFFFFu, ok)) {
          if (lane == 0) {
            atomicExch(a.status, 1u);
            *abort = 1;
          }
          return;
        }
        const uint64_t vi = v0 + ct;
        const uint32_t base = smem0 + stage * stage_bytes;
        uint4 in[MAXP];
        float g[E];
        float wf[E], vf[E];
        if (vi < nvec) {
#pragma unroll
          for (int r = 0; r < MAXP; ++r)
            if (Ranks<PT>::has(r, np)) in[r] = lds128(base + r * tma_grad_tile_bytes() + ct * 16);
          if constexpr (SGD) {
            const uint32_t fb = base + Ranks<PT>::count(np) * tma_grad_tile_bytes() + ct * E * 4;
#pragma unroll
            for (int q = 0; q < E / 4; ++q) {
              const float4 a4 = lds128f(fb + q * 16);
              const float4 b4 = lds128f(fb + kTmaTileVec * E * 4 + q * 16);
              wf[4 * q] = a4.x; wf[4 * q + 1] = a4.y; wf[4 * q + 2] = a4.z; wf[4 * q + 3] = a4.w;
              vf[4 * q] = b4.x; vf[4 * q + 1] = b4.y; vf[4 * q + 2] = b4.z; vf[4 * q + 3] = b4.w;
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty_bar[stage]));
        if (++stage == uint32_t(S)) {
          stage = 0;
          phase ^= 1;
        }
        if (vi < nvec) {
          reduce_vec<D, PT>(in, np, mean, g);
          if constexpr (SGD) {
#pragma unroll
            for (int e = 0; e < E; ++e) sgd_step(g[e], a.lr, a.mu, wf[e], vf[e]);
#pragma unroll
            for (int q = 0; q < E / 4; ++q) {
              st_f4(w + vi * E + 4 * q, make_float4(wf[4 * q], wf[4 * q + 1], wf[4 * q + 2], wf[4 * q + 3]));
              st_f4(v + vi * E + 4 * q, make_float4(vf[4 * q], vf[4 * q + 1], vf[4 * q + 2], vf[4 * q + 3]));
            }
          }
          if (do_store) {
            const uint4 out = D::pack(g);
            for (int d = 0; d < a.ndst; ++d) st_stream(static_cast<uint4*>(dst[d]) + vi, out);
          }
        }
      }
      if (last) {  // ragged tail (< E elements) from global memory
        const uint64_t i = nvec * E + ct;
        if (i < n) {
          float g = reduce_scalar<D, PT>(ptrs, i, np, mean);
          if constexpr (SGD) sgd_step(g, a.lr, a.mu, w[i], v[i]);
          if (do_store)
            for (int d = 0; d < a.ndst; ++d) D::store1(dst[d], i, g);
        }
      }
    } else {
      const uint64_t e0 = lt * uint64_t(kTmaTileVec) * E;
      for (uint64_t k = ct; k < uint64_t(kTmaTileVec) * E; k += 32 * kTmaConsumerWarps) {
        const uint64_t i = e0 + k;
        if (i >= n) break;
        float g = reduce_scalar<D, PT>(ptrs, i, np, mean);
        if constexpr (SGD) sgd_step(g, a.lr, a.mu, w[i], v[i]);
        if (do_store)
          for (int d = 0; d < a.ndst; ++d) D::store1(dst[d], i, g);
      }
    }
    if (__shfl_sync(0xFFFFFFFFu, *abort, 0)) return;  // warp-uniform
  }
}

// ------------------------------------------------------- bulk-store copy
// k_copy_tma: the copy collectives (all-gather, broadcast) on the bulk-copy
// engine.  Lane 0 of each CTA runs a pipeline over its tiles (kCopyTmaTile
// bytes of one segment): a bulk load of tile j into stage j % S, then, once it has
// landed, one bulk store of the stage to every destination of the segment
// (a bulk group per tile).  The load of tile j + S - 1 reuses the stage of
// tile j - 1 after that tile's stores have finished reading it, so S - 1
// loads stay in flight while the stores drain.  Tiles without a 16-byte
// part (a ragged tail only) or of unaligned segments still take their
// pipeline slot, with nothing to load; their bytes are copied with 2-byte
// accesses by the warp.  Every wait is bounded.
#ifndef GAR_COPY_STAGES
#define GAR_COPY_STAGES 4
#endif
#ifndef GAR_COPY_TILE_KB
#define GAR_COPY_TILE_KB 16
#endif
constexpr int kCopyTmaStages = GAR_COPY_STAGES;
constexpr uint32_t kCopyTmaTile = GAR_COPY_TILE_KB * 1024;

__device__ __forceinline__ void bulk_s2g(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

template <class Cap>
__global__ void __launch_bounds__(32, 1) k_copy_tma(const __grid_constant__ SegTable<Cap> a) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kCopyTmaStages];
  const uint32_t smem0 = smem_u32(smem_raw);
  const int lane = threadIdx.x;
  if (lane == 0) {
    for (int k = 0; k < kCopyTmaStages; ++k) mbar_init(smem_u32(&full_bar[k]), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();
  griddep_launch_dependents();
  griddep_wait();

  // My tiles: blockIdx.x, blockIdx.x + G, ...; mine = how many.
  const uint32_t G = gridDim.x;
  const uint32_t mine = a.ntiles > blockIdx.x ? (a.ntiles - blockIdx.x + G - 1) / G : 0;

  // Where tile `tile` lives: segment, byte offset, bytes of its 16-byte part.
  struct Tile { uint32_t seg; uint64_t off; uint32_t vbytes; };
  auto locate = [&](uint32_t tile, uint32_t& segc) {
    while (tile >= a.tile0[segc + 1]) ++segc;
    Tile t;
    t.seg = segc;
    t.off = uint64_t(tile - a.tile0[segc]) * kCopyTmaTile;
    const uint64_t vb = (a.flags[segc] & kSegVec) ? (a.numel[segc] / 16) * 16 : 0;
    t.vbytes = t.off < vb ? uint32_t(vb - t.off < kCopyTmaTile ? vb - t.off : kCopyTmaTile) : 0u;
    return t;
  };

  bool ok = true;
  uint32_t seg_load = 0, seg_store = 0;
  if (lane == 0) {
    // Prologue: loads of my tiles 0 .. S-2.
    for (uint32_t j = 0; j + 1 < kCopyTmaStages && j < mine; ++j) {
      const Tile t = locate(blockIdx.x + j * G, seg_load);
      const uint32_t full = smem_u32(&full_bar[j % kCopyTmaStages]);
      mbar_expect_tx(full, t.vbytes);
      if (t.vbytes)
        bulk_g2s(smem0 + (j % kCopyTmaStages) * kCopyTmaTile,
                 static_cast<const char*>(a.ptr[uint64_t(t.seg) * a.stride]) + t.off, t.vbytes, full);
    }
  }
  for (uint32_t j = 0; j < mine; ++j) {
    const uint32_t tile = blockIdx.x + j * G;
    const uint32_t stage = j % kCopyTmaStages;
    uint32_t segc = seg_store;
    const Tile t = locate(tile, segc);
    seg_store = segc;
    void* const* seg = a.ptr + uint64_t(t.seg) * a.stride;
    const int nd = int(a.flags[t.seg] >> 8);
    if (lane == 0 && ok) {
      if (!mbar_wait_bounded(smem_u32(&full_bar[stage]), (j / kCopyTmaStages) & 1u, nullptr)) {
        atomicExch(a.status, 1u);
        ok = false;
      } else {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        if (t.vbytes)
          for (int d = 0; d < nd; ++d)
            bulk_s2g(static_cast<char*>(seg[a.dst_off + d]) + t.off,
                     smem0 + stage * kCopyTmaTile, t.vbytes);
        bulk_commit();
        // Load tile j + S - 1 into the stage of tile j - 1, once that
        // tile's stores have read it (all groups but the newest).
        const uint32_t jn = j + kCopyTmaStages - 1;
        if (jn < mine) {
          bulk_wait_read_1();
          const Tile tn = locate(blockIdx.x + jn * G, seg_load);
          const uint32_t full = smem_u32(&full_bar[jn % kCopyTmaStages]);
          mbar_expect_tx(full, tn.vbytes);
          if (tn.vbytes)
            bulk_g2s(smem0 + (jn % kCopyTmaStages) * kCopyTmaTile,
                     static_cast<const char*>(a.ptr[uint64_t(tn.seg) * a.stride]) + tn.off,
                     tn.vbytes, full);
        }
      }
    }
    // The bytes of the tile that the bulk copies do not cover (a ragged
    // tail, or the whole tile of an unaligned segment), 2 bytes at a time.
    const uint64_t nbytes = a.numel[t.seg];
    const uint64_t end = t.off + kCopyTmaTile < nbytes ? t.off + kCopyTmaTile : nbytes;
    const uint16_t* src = static_cast<const uint16_t*>(seg[0]);
    for (uint64_t h = (t.off + t.vbytes) / 2 + lane; h < end / 2; h += 32) {
      const uint16_t x = src[h];
      for (int d = 0; d < nd; ++d) static_cast<uint16_t*>(seg[a.dst_off + d])[h] = x;
    }
  }
  if (lane == 0) bulk_wait_all();
}

// Failure-detection self-test: one warp waits on an mbarrier that nothing
// ever arrives at, with the pipeline's bounded wait; when the wait gives up
// it records status 1, exactly as a stalled pipeline stage would.
__global__ void k_wait_selftest(uint32_t* status, uint64_t limit_ns);

// Tile size in elements of k_reduce_tma.
__host__ __device__ constexpr uint64_t tma_tile_elems(int elems_per_vec) {
  return uint64_t(kTmaTileVec) * elems_per_vec;
}

}  // namespace gar
