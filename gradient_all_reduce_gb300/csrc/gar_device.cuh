// gar_device.cuh -- device helpers shared by the GB300 collective kernels:
// 16-byte streaming loads/stores, bf16 <-> fp32 conversion, and the
// rank-ordered fp32 reduction of one 16-byte vector position.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace gar {

constexpr int kMaxRanks = 16;
constexpr int kThreads = 256;  // threads per CTA of every kernel

// Bits of a comm's device status word.
constexpr uint32_t kStatusTimeout = 1u;  // a bounded wait gave up
constexpr uint32_t kStatusBounds = 2u;   // a debug-build index check failed

// Device-side index checks of a debug build (compiled with GAR_DEBUG=1): a
// kernel checks, before an access, that the index it is about to use lies
// inside the segment, channel range or table that the launch describes.  A
// failed check sets kStatusBounds in the status word and the thread leaves
// the kernel without the access -- it never traps, so the context stays
// usable and the host reads the failure with ar_get_async_error.  Only the
// kernels without block-wide barriers carry checks (a thread that leaves
// early would strand a barrier).  A release build compiles every check
// away.
#ifndef GAR_DEBUG
#define GAR_DEBUG 0
#endif
#if GAR_DEBUG
__device__ __forceinline__ bool dcheck(bool ok, uint32_t* status) {
  if (!ok && status != nullptr) atomicOr(status, kStatusBounds);
  return ok;
}
#define GAR_CHECK(cond, status) \
  if (!::gar::dcheck((cond), (status))) return
#else
#define GAR_CHECK(cond, status) ((void)0)
#endif

// ------------------------------------------------------------ memory ops
// Every replica value is read exactly once and written at most once per
// call, so loads bypass L1 (no reuse) and stores are streaming.
//
// Replica loads (ld_stream) take the coherent path: an in-place call
// writes the very buffers it reads, and PTX allows the non-coherent (.nc)
// path only for data that no thread writes while the kernel runs.  (Each
// 16-byte position is read by one thread before that thread writes it, so
// .nc would never have returned a stale value either; on GB300 the two
// forms measured the same, 1.035 of the copy peak for an fp32 all-reduce at
// P = 8 and 0.977 for a 25 MiB fused-SGD bucket.)  Loads of buffers the
// kernel never writes -- a copy's source, a gradient being accumulated --
// keep the .nc path (ld_stream8, ld_keep, ld_stream_ro).

// Cache hints of the streaming accesses (tuning knobs, fixed at build time):
// GAR_LD_PREFETCH 1 adds an L2 256-byte prefetch hint to the loads;
// GAR_ST_STREAMING 1 marks the stores evict-first (.cs), 0 leaves them
// write-back with the default policy.
#ifndef GAR_LD_PREFETCH
#define GAR_LD_PREFETCH 0
#endif
#ifndef GAR_ST_STREAMING
#define GAR_ST_STREAMING 1
#endif

// GAR_LD_COHERENT 0 loads the replicas through the non-coherent path
// instead (only valid for calls that are not in place).
#ifndef GAR_LD_COHERENT
#define GAR_LD_COHERENT 1
#endif

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 r;
#if GAR_LD_COHERENT
  asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
#elif GAR_LD_PREFETCH
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
#else
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
#endif
  return r;
}

// 16-byte load of a buffer that no thread of the kernel writes.
__device__ __forceinline__ uint4 ld_stream_ro(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ void st_stream(void* p, const uint4& v) {
#if GAR_ST_STREAMING
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
#else
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
#endif
}

// 8-byte form of ld_stream (four bf16 elements).
__device__ __forceinline__ uint2 ld_stream8(const void* p) {
  uint2 r;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
  return r;
}

// fp32 master-weight / momentum arrays are read and written by the same
// thread (read-modify-write), so they use the coherent path.
__device__ __forceinline__ float4 ld_f4(const float* p) {
  float4 r;
  asm volatile("ld.global.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ void st_f4(float* p, const float4& v) {
  asm volatile("st.global.cs.v4.f32 [%0], {%1,%2,%3,%4};" ::"l"(p), "f"(v.x), "f"(v.y),
               "f"(v.z), "f"(v.w)
               : "memory");
}

// Register fences: an empty volatile asm that "modifies" a loaded value.  It
// keeps the arithmetic on that value after every earlier volatile load, so
// a thread issues all of its loads before it waits on any of them.
__device__ __forceinline__ void reg_fence(uint4& v) {
  asm volatile("" : "+r"(v.x), "+r"(v.y), "+r"(v.z), "+r"(v.w));
}
__device__ __forceinline__ void reg_fence(uint2& v) { asm volatile("" : "+r"(v.x), "+r"(v.y)); }
__device__ __forceinline__ void reg_fence(float4& v) {
  asm volatile("" : "+f"(v.x), "+f"(v.y), "+f"(v.z), "+f"(v.w));
}

// Programmatic dependent launch: let the next kernel of the stream start
// its launch now, and wait until the previous kernel has finished and its
// writes are visible (both are no-ops when the launch did not opt in).  A
// kernel calls the wait before its first global-memory access and after
// its reads of its own parameter table, which need nothing from the
// previous kernel; the wait returns at once when called again.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------- dtypes
// bf16 is the upper half of an fp32 bit pattern: widening is a shift.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// fp32 -> bf16, IEEE round to nearest, ties to even, by the hardware
// conversion (cvt.rn without .ftz: subnormals are kept, a value that rounds
// past the largest finite bf16 becomes infinity, a NaN stays a NaN).  The
// packed form takes two values; its first source operand fills the upper
// half.
__device__ __forceinline__ uint32_t bf16x2_rne(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}
__device__ __forceinline__ uint16_t bf16_rne(float f) {
  uint16_t h;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h) : "f"(f));
  return h;
}

struct F32 {
  static constexpr int kElems = 4;  // elements per 16-byte vector
  static constexpr int kBytes = 4;
  __device__ static __forceinline__ void unpack(const uint4& v, float (&f)[4]) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
  }
  __device__ static __forceinline__ uint4 pack(const float (&f)[4]) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
  }
  // A quad is 4 consecutive elements (16 bytes): quad q holds elements 4q .. 4q + 3.
  using Quad = uint4;
  __device__ static __forceinline__ Quad ld_quad(const void* p, uint64_t q) {
    return ld_stream_ro(static_cast<const uint4*>(p) + q);
  }
  __device__ static __forceinline__ void unpack_quad(const Quad& v, float (&f)[4]) { unpack(v, f); }
  __device__ static __forceinline__ float load1(const void* p, uint64_t i) {
    return static_cast<const float*>(p)[i];
  }
  __device__ static __forceinline__ void store1(void* p, uint64_t i, float f) {
    static_cast<float*>(p)[i] = f;
  }
};

struct BF16 {
  static constexpr int kElems = 8;
  static constexpr int kBytes = 2;
  // Element 2k of a 32-bit word is its low half (little-endian order).
  __device__ static __forceinline__ void unpack(const uint4& v, float (&f)[8]) {
    f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
    f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
    f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
  }
  __device__ static __forceinline__ uint4 pack(const float (&f)[8]) {
    return make_uint4(bf16x2_rne(f[0], f[1]), bf16x2_rne(f[2], f[3]), bf16x2_rne(f[4], f[5]),
                      bf16x2_rne(f[6], f[7]));
  }
  // A quad is 4 consecutive elements (8 bytes): quad q holds elements 4q .. 4q + 3.
  using Quad = uint2;
  __device__ static __forceinline__ Quad ld_quad(const void* p, uint64_t q) {
    return ld_stream8(static_cast<const uint2*>(p) + q);
  }
  __device__ static __forceinline__ void unpack_quad(const Quad& v, float (&f)[4]) {
    f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
    f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
  }
  __device__ static __forceinline__ float load1(const void* p, uint64_t i) {
    return __uint_as_float(uint32_t(static_cast<const uint16_t*>(p)[i]) << 16);
  }
  __device__ static __forceinline__ void store1(void* p, uint64_t i, float f) {
    static_cast<uint16_t*>(p)[i] = bf16_rne(f);
  }
};

// ---------------------------------------------------------- reduction
// PT > 0: P is the compile-time constant PT (every register-staged kernel).
// PT < 0: P is the runtime value np, at most -PT; PT == 0: at most
// kMaxRanks (the bulk-copy pipeline's kernel for P outside 2, 4, 8).
// Bounded loops run to the maximum under a guard so the operands stay in
// registers.
template <int PT>
struct Ranks {
  static constexpr int kMax = PT > 0 ? PT : (PT < 0 ? -PT : kMaxRanks);
  __device__ static __forceinline__ bool has(int r, int np) { return PT > 0 ? r < PT : r < np; }
  __device__ static __forceinline__ int count(int np) { return PT > 0 ? PT : np; }
};

// x / d rounded to nearest even, for d a small integer that is not a power
// of two and r = RN(1/d), by Markstein's correction (P. W. Markstein,
// "Computation of elementary functions on the IBM RISC System/6000
// processor", IBM J. Res. Develop. 34(1), 1990): y = RN(x r) is within an ulp
// of x/d, one fused multiply-add gives the residual x - y d exactly, and
// RN(y + r (x - y d)) is the correctly rounded quotient.  Zeros, infinities,
// NaNs and |x| < 2^-100 (where the residual could underflow) take the IEEE
// division.  Checked equal to __fdiv_rn for every fp32 x and d = 3..15 by
// an exhaustive GPU test.
__device__ __forceinline__ float div_small(float x, float d, float r) {
  const float ax = fabsf(x);
  if (!(ax >= 0x1p-100f) || ax == __int_as_float(0x7f800000)) return __fdiv_rn(x, d);
  const float y = __fmul_rn(x, r);
  const float e = __fmaf_rn(-y, d, x);
  return __fmaf_rn(e, r, y);
}

// x / d for a quotient that is only ever stored as bf16 (round to nearest
// even of the correctly rounded fp32 quotient q).  With r = RN(1/d) and
// y = RN(x r), y = (x/d)(1 + e1)(1 + e2) with |e1|, |e2| <= 2^-24, so y lies
// within three units in the last place of q (as bit patterns).  Two fp32
// values that close round to the same bf16 unless a rounding boundary lies
// between them, and the boundaries sit next to a low half of 0x8000 (the
// tie).  So y serves unless its low half lies in 0x7FFC .. 0x8003, where
// div_small gives q itself.  Zeros and infinities pass through y unchanged
// and a NaN stays a NaN.  Checked on the GPU for every fp32 x and d = 3..15:
// the bf16 rounding equals that of __fdiv_rn.
__device__ __forceinline__ float div_small_bf16(float x, float d, float r) {
  const float y = __fmul_rn(x, r);
  return ((__float_as_uint(y) - 0x7FFCu) & 0xFFFFu) < 8u ? div_small(x, d, r) : y;
}

// Mean: one correctly rounded fp32 division by P.  For P a power of two
// the product with the exact reciprocal is the same correctly rounded
// quotient, so powers of two multiply instead (decided at compile time for
// a fixed P, per call for a runtime P).  Other P divide by Markstein's
// correction: always for a compile-time P (divisor and reciprocal are
// constants), and for a runtime P when FAST (the bulk-copy pipeline's bf16
// kernel: 8 divisions per vector); its fp32 kernel takes the IEEE division.
// BF16_OUT: the mean is only stored as bf16, so a quotient with the same
// bf16 rounding serves (div_small_bf16).
template <int PT, bool FAST = false, bool BF16_OUT = false>
__device__ __forceinline__ float mean_of(float sum, int np) {
  if constexpr (PT > 0 && (PT & (PT - 1)) == 0) {
    return __fmul_rn(sum, 1.0f / float(PT));
  } else if constexpr (PT > 0) {
    constexpr float d = float(PT), r = 1.0f / float(PT);  // r = RN(1/d), folded at compile time
    if constexpr (BF16_OUT) {
      return div_small_bf16(sum, d, r);
    } else {
      return div_small(sum, d, r);
    }
  } else {
    const float d = float(np), r = __frcp_rn(d);
    if constexpr (FAST && BF16_OUT) {
      return (np & (np - 1)) == 0 ? __fmul_rn(sum, r) : div_small_bf16(sum, d, r);
    } else if constexpr (FAST) {
      return (np & (np - 1)) == 0 ? __fmul_rn(sum, r) : div_small(sum, d, r);
    } else {
      return (np & (np - 1)) == 0 ? __fmul_rn(sum, r) : __fdiv_rn(sum, d);
    }
  }
}

// acc[e] = in[0][e] + in[1][e] + ... + in[P-1][e], left to right in fp32,
// seeded with rank 0's value; then divided by P when mean is set.  STORE_ONLY:
// the caller only stores the result in the replicas' element type.
template <class D, int PT, bool STORE_ONLY = false>
__device__ __forceinline__ void reduce_vec(const uint4 (&in)[Ranks<PT>::kMax], int np, bool mean,
                                           float (&acc)[D::kElems]) {
  D::unpack(in[0], acc);
#pragma unroll
  for (int r = 1; r < Ranks<PT>::kMax; ++r) {
    if (Ranks<PT>::has(r, np)) {
      float x[D::kElems];
      D::unpack(in[r], x);
#pragma unroll
      for (int e = 0; e < D::kElems; ++e) acc[e] = __fadd_rn(acc[e], x[e]);
    }
  }
  if (mean) {
#pragma unroll
    for (int e = 0; e < D::kElems; ++e)
      acc[e] = mean_of<PT, D::kElems == 8, STORE_ONLY && D::kElems == 8>(acc[e], np);
  }
}

// The same for one element read with scalar loads (ragged tails and
// buffers that are not 16-byte aligned).
template <class D, int PT>
__device__ __forceinline__ float reduce_scalar(const void* const* src, uint64_t i, int np,
                                               bool mean) {
  float acc = D::load1(src[0], i);
#pragma unroll
  for (int r = 1; r < Ranks<PT>::kMax; ++r)
    if (Ranks<PT>::has(r, np)) acc = __fadd_rn(acc, D::load1(src[r], i));
  return mean ? mean_of<PT, D::kElems == 8>(acc, np) : acc;
}

// SGD with momentum on one element: v = fl(fl(mu*v) + g); w = fl(w - fl(lr*v)).
__device__ __forceinline__ void sgd_step(float g, float lr, float mu, float& w, float& v) {
  v = __fadd_rn(__fmul_rn(mu, v), g);
  w = __fsub_rn(w, __fmul_rn(lr, v));
}

// ---------------------------------------------------------------------------
// The SyncBN statistics' division by the pooled count.  On GB300 a dependent
// fp64 warp instruction takes about 64 cycles and the IEEE division about
// 560.

// s / n rounded to nearest even, for n an integer count (1 <= n <= 2^53)
// and y = RN(1/n), by Markstein's correction applied twice (P. W.
// Markstein, IBM J. Res. Develop. 34(1), 1990).  q0 = RN(s y) lies within
// two ulps of s/n; one correction, q1 = RN(q0 + y RN(s - q0 n)), lands
// within half an ulp plus 2^-51 ulp, so q1 is one of the two fp64 numbers
// around s/n.  For such a q1 the residual s - q1 n is exact (one FMA), and
// with y within half an ulp of 1/n, RN(q1 + y (s - q1 n)) is RN(s/n).  No
// step underflows or overflows for the sums this serves (|s| >= 2^-149
// unless zero, |s| < 2^133).  Zero (whose sign the correction would lose),
// infinity and NaN take the IEEE division.
__device__ __forceinline__ double div_count(double s, double n, double y) {
  if (s == 0.0 || !(fabs(s) < __longlong_as_double(0x7FF0000000000000ll))) return __ddiv_rn(s, n);
  double q = __dmul_rn(s, y);
  double r = __fma_rn(-q, n, s);
  q = __fma_rn(r, y, q);
  r = __fma_rn(-q, n, s);
  return __fma_rn(r, y, q);
}

}  // namespace gar
