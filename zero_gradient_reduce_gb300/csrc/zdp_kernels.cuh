// zdp_kernels.cuh -- device code of the ZeRO step: ring-order gradient sum,
// AdamW, bf16 cast and replica stores.
//
// The step is a pure streaming computation: per element it reads P gradient
// values and 12 bytes of fp32 state and writes 12 bytes of state and P
// replica values, (4P + 24) bytes per parameter with bf16 gradients, at well
// under one flop per byte.  HBM bandwidth bounds it, so the kernels are laid
// out for memory-level parallelism, not arithmetic:
//  * one thread handles a vector of 8 consecutive elements: one 16-byte load
//    per rank gradient, two per fp32 state array, one 16-byte store per
//    replica; a warp touches 512 contiguous bytes of every stream;
//  * every load of a vector is issued before the first add consumes one (for
//    P > 8, group by group of 8 ranks);
//  * persistent grid-stride grids with a measured number of resident blocks
//    per SM (see zdp_internal.h);
//  * streaming cache hints (evict-first, ld/st.global.cs) on every access:
//    nothing is reused within a step.
// Numerics: the ring sum adds in a fixed order with __fadd_rn and the AdamW
// update uses only *_rn intrinsics, so no multiply-add is ever contracted and
// every result is the IEEE fp32 result of the stated formula.
//
// Rank-count templates: PT in 1..8 is exactly P = PT; PT = 8*G (G = 2..8)
// is exactly P = PT, or (not EXACT) any P in (PT-8, PT) as G groups of 8
// ranks whose last group is partial.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "zdp_internal.h"

namespace zdp {

// ---------------------------------------------------------------------------
// Number formats
// ---------------------------------------------------------------------------

// Two gradient values packed in a 32-bit word (element 2k in the low half).
template <int GT>
__device__ __forceinline__ float2 widen2(uint32_t u) {
  if constexpr (GT == ZDP_BF16) {
    // bf16 is the upper half of an fp32: widening is a shift, exact.
    return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
  } else {
    __half2 h = *reinterpret_cast<__half2*>(&u);
    return __half22float2(h);  // exact
  }
}

template <int GT>
__device__ __forceinline__ float widen1(uint16_t u) {
  if constexpr (GT == ZDP_BF16) {
    return __uint_as_float(static_cast<uint32_t>(u) << 16);
  } else {
    return __half2float(__ushort_as_half(u));
  }
}

// Round two fp32 values to bf16 (nearest, ties to even); `lo` lands in the
// low half, so the word is two consecutive elements in memory order.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

__device__ __forceinline__ uint16_t to_bf16(float x) {
  return static_cast<uint16_t>(pack_bf16x2(x, 0.0f) & 0xffffu);
}

__device__ __forceinline__ bool non_finite(float x) {
  return (__float_as_uint(x) & 0x7f800000u) == 0x7f800000u;
}

// ---------------------------------------------------------------------------
// Owner of a global element: r = i / S, without a 64-bit division.  The fp32
// estimate i * (1/S) has relative error below 2^-22, i.e. absolute error
// below 64 * 2^-22 < 1 since i / S < P <= 64, so one correction step lands on
// the exact floor.
// ---------------------------------------------------------------------------
// fp32 value of a non-negative 64-bit index, from two 32-bit conversions
// and one fma (relative error below 2^-23; measured 0.2% faster on the fused
// step than the 64-bit conversion).  owner_calc corrects the estimate by one.
__device__ __forceinline__ float index_to_float(int64_t i) {
  const float hi = __uint2float_rn(static_cast<uint32_t>(static_cast<uint64_t>(i) >> 32));
  const float lo = __uint2float_rn(static_cast<uint32_t>(i));
  return __fmaf_rn(hi, 4294967296.0f, lo);
}

__device__ __forceinline__ int owner_calc(int64_t i, int64_t S, float inv_s, int P) {
  int r = static_cast<int>(index_to_float(i) * inv_s);
  r = r > P - 1 ? P - 1 : r;
  if (static_cast<int64_t>(r) * S > i) {
    --r;
  } else if (static_cast<int64_t>(r + 1) * S <= i) {
    ++r;
  }
  // i < n <= P*S keeps r in [0, P-1]; the clamp makes that hold for any input.
  return r < 0 ? 0 : (r > P - 1 ? P - 1 : r);
}

__device__ __forceinline__ int owner_of(int64_t i, const KParams& p, int P) {
  return owner_calc(i, p.S, p.inv_s, P);
}

// ---------------------------------------------------------------------------
// Memory access with streaming (evict-first) hints.  Measured on GB300: the
// .cs stores matter (plain stores cost ~13% of throughput); the load hint
// does not.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 ld16(const void* ptr) {
  return __ldcs(reinterpret_cast<const uint4*>(ptr));
}
__device__ __forceinline__ void st16(void* ptr, uint4 x) {
  __stcs(reinterpret_cast<uint4*>(ptr), x);
}

template <int GT>
__device__ __forceinline__ const uint4* grad_vec(const KParams& p, int q, int64_t i0) {
  return reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.g[q]) + (i0 - p.goff));
}

template <int GT>
__device__ __forceinline__ uint16_t grad_elem(const KParams& p, int q, int64_t i) {
  return __ldcs(static_cast<const uint16_t*>(p.g[q]) + (i - p.goff));
}

// ---------------------------------------------------------------------------
// Ring-order sum.  Element i owned by rank r: acc = G_{(r+1)%P}[i], then
// acc += G_{(r+2)%P}[i], ..., acc += G_r[i], each add rounded to fp32.
// ---------------------------------------------------------------------------

template <int GT>
__device__ __forceinline__ void vec_set(float (&acc)[kVec], const uint4& d) {
  const uint32_t w[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 f = widen2<GT>(w[k]);
    acc[2 * k] = f.x;
    acc[2 * k + 1] = f.y;
  }
}

template <int GT>
__device__ __forceinline__ void vec_add(float (&acc)[kVec], const uint4& d) {
  const uint32_t w[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 f = widen2<GT>(w[k]);
    acc[2 * k] = __fadd_rn(acc[2 * k], f.x);
    acc[2 * k + 1] = __fadd_rn(acc[2 * k + 1], f.y);
  }
}

__device__ __forceinline__ int ring_next(int q, int P) { return q + 1 == P ? 0 : q + 1; }

// Rank-count templates: PT <= 8 is exactly P = PT.  PT = 8*G with EXACT
// is exactly P = PT; without EXACT it serves any P in (PT-8, PT), whose
// last group of 8 is partial.
template <int PT, bool EXACT>
__device__ __forceinline__ int ranks(const KParams& p) {
  return (PT <= 8 || EXACT) ? PT : p.P;
}

// Loads the next `full ? 8 : cnt` ranks of the ring into d[] and advances q.
template <int GT>
__device__ __forceinline__ void load8(const KParams& p, int P, int& q, bool full, int cnt,
                                      int64_t i0, uint4 (&d)[8]) {
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    if (full || k < cnt) {
      d[k] = ld16(grad_vec<GT>(p, q, i0));
      q = ring_next(q, P);
    }
  }
}

template <int GT>
__device__ __forceinline__ void add8(bool full, int cnt, bool first, const uint4 (&d)[8],
                                     float (&acc)[kVec]) {
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    if (full || k < cnt) {
      if (first && k == 0) {
        vec_set<GT>(acc, d[0]);
      } else {
        vec_add<GT>(acc, d[k]);
      }
    }
  }
}

// The 8 elements starting at i0 (a multiple of 8), all owned by rank r.
template <int PT, bool EXACT, int GT>
__device__ __forceinline__ void ring_sum_vec(const KParams& p, int P, int r, int64_t i0,
                                             float (&acc)[kVec]) {
  int q = ring_next(r, P);
  if constexpr (PT <= 8) {
    uint4 d[PT];
#pragma unroll
    for (int k = 0; k < PT; ++k) {
      d[k] = ld16(grad_vec<GT>(p, q, i0));
      q = ring_next(q, PT);
    }
    vec_set<GT>(acc, d[0]);
#pragma unroll
    for (int k = 1; k < PT; ++k) vec_add<GT>(acc, d[k]);
  } else {
    // Groups of 8 ranks through two register buffers: the loads of group
    // gi+1 are issued before the adds of group gi.  Only the last group can
    // be partial (when !EXACT); every `full` below is a compile-time
    // constant once the loop is unrolled.
    constexpr int G = PT / 8;
    const int last = EXACT ? 8 : P - 8 * (G - 1);
    uint4 buf[2][8];
    load8<GT>(p, P, q, EXACT || G > 1, last, i0, buf[0]);
#pragma unroll
    for (int gi = 0; gi < G; ++gi) {
      if (gi + 1 < G) load8<GT>(p, P, q, EXACT || gi + 1 < G - 1, last, i0, buf[(gi + 1) & 1]);
      add8<GT>(EXACT || gi < G - 1, last, gi == 0, buf[gi & 1], acc);
    }
  }
}

template <int GT>
__device__ __forceinline__ float ring_sum_elem(const KParams& p, int P, int r, int64_t i) {
  int q = ring_next(r, P);
  float acc = widen1<GT>(grad_elem<GT>(p, q, i));
  for (int k = 1; k < P; ++k) {
    q = ring_next(q, P);
    acc = __fadd_rn(acc, widen1<GT>(grad_elem<GT>(p, q, i)));
  }
  return acc;
}

// ---------------------------------------------------------------------------
// AdamW on one element, every operation rounded on its own.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void adamw(float& w, float& m, float& v, float g, const AdamK& a) {
  const float m_new = __fadd_rn(__fmul_rn(a.b1, m), __fmul_rn(a.one_minus_b1, g));
  const float g_sq = __fmul_rn(g, g);
  const float v_new = __fadd_rn(__fmul_rn(a.b2, v), __fmul_rn(a.one_minus_b2, g_sq));
  const float m_hat = __fdiv_rn(m_new, a.bc1);
  const float v_hat = __fdiv_rn(v_new, a.bc2);
  const float denom = __fadd_rn(__fsqrt_rn(v_hat), a.eps);
  const float u = __fdiv_rn(m_hat, denom);
  const float w_decayed = __fsub_rn(w, __fmul_rn(a.lr_wd, w));
  w = __fsub_rn(w_decayed, __fmul_rn(a.lr, u));
  m = m_new;
  v = v_new;
}

// ---------------------------------------------------------------------------
// fp32 vectors of 8 (two 16-byte accesses)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ld_f8(const float* ptr, float (&x)[kVec]) {
  const uint4 a = ld16(ptr);
  const uint4 b = ld16(ptr + 4);
  x[0] = __uint_as_float(a.x); x[1] = __uint_as_float(a.y);
  x[2] = __uint_as_float(a.z); x[3] = __uint_as_float(a.w);
  x[4] = __uint_as_float(b.x); x[5] = __uint_as_float(b.y);
  x[6] = __uint_as_float(b.z); x[7] = __uint_as_float(b.w);
}

__device__ __forceinline__ void st_f8(float* ptr, const float (&x)[kVec]) {
  st16(ptr, make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]),
                       __float_as_uint(x[3])));
  st16(ptr + 4, make_uint4(__float_as_uint(x[4]), __float_as_uint(x[5]), __float_as_uint(x[6]),
                           __float_as_uint(x[7])));
}

__device__ __forceinline__ uint4 pack_bf16x8(const float (&x)[kVec]) {
  return make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]), pack_bf16x2(x[4], x[5]),
                    pack_bf16x2(x[6], x[7]));
}

// ---------------------------------------------------------------------------
// AdamW moments stored as fp32 or bf16 (p.mt is uniform over the grid).  bf16
// moments are widened exactly and stored rounded to nearest even.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ld_moments8(const void* pm, const void* pv, int mt, int64_t i0,
                                            float (&m)[kVec], float (&v)[kVec]) {
  if (mt == ZDP_MOMENTS_F32) {
    ld_f8(static_cast<const float*>(pm) + i0, m);
    ld_f8(static_cast<const float*>(pv) + i0, v);
  } else {
    vec_set<ZDP_BF16>(m, ld16(static_cast<const uint16_t*>(pm) + i0));
    vec_set<ZDP_BF16>(v, ld16(static_cast<const uint16_t*>(pv) + i0));
  }
}

__device__ __forceinline__ void st_moments8(void* pm, void* pv, int mt, int64_t i0,
                                            const float (&m)[kVec], const float (&v)[kVec]) {
  if (mt == ZDP_MOMENTS_F32) {
    st_f8(static_cast<float*>(pm) + i0, m);
    st_f8(static_cast<float*>(pv) + i0, v);
  } else {
    st16(static_cast<uint16_t*>(pm) + i0, pack_bf16x8(m));
    st16(static_cast<uint16_t*>(pv) + i0, pack_bf16x8(v));
  }
}

__device__ __forceinline__ float ld_moment(const void* base, int64_t i, int mt) {
  return mt == ZDP_MOMENTS_F32 ? static_cast<const float*>(base)[i]
                               : widen1<ZDP_BF16>(static_cast<const uint16_t*>(base)[i]);
}

__device__ __forceinline__ void st_moment(void* base, int64_t i, int mt, float x) {
  if (mt == ZDP_MOMENTS_F32) {
    static_cast<float*>(base)[i] = x;
  } else {
    static_cast<uint16_t*>(base)[i] = to_bf16(x);
  }
}

// ---------------------------------------------------------------------------
// Flag and sum-of-squares accounting, one atomic per block at most.
//
// GB300 executes fp64 at a small fraction of its fp32 rate, so the sum of
// squares is accumulated in fp32 without losing accuracy: g*g is split
// exactly into p + e (p = fl(g*g), e = fma(g, g, -p)), p is added to the
// running sum `hi` with TwoSum (the rounding error is captured exactly),
// and the small parts collect in `lo`.  Every 32 vectors (<= 256 terms) the
// pair is flushed into an fp64 total, which bounds the error of the fp32
// `lo` far below the 1e-9 relative tolerance of the result.  Values whose
// square could leave the range where this split is exact in fp32
// (|g| outside [2^-40, 2^50), and inf/NaN) go straight to the fp64 total,
// so an infinite or NaN gradient gives the same inf/NaN as an fp64 sum.
// ---------------------------------------------------------------------------
struct SumSq {
  float hi = 0.0f, lo = 0.0f;
  double total = 0.0;
  int pending = 0;

  __device__ __forceinline__ void add(float g) {
    const float a = fabsf(g);
    if (!(a >= 0x1p-40f && a < 0x1p50f)) {  // also taken by NaN
      const double d = static_cast<double>(g);
      total = __fma_rn(d, d, total);
      return;
    }
    const float p = __fmul_rn(g, g);
    const float e = __fmaf_rn(g, g, -p);
    const float s = __fadd_rn(hi, p);
    const float bp = __fsub_rn(s, hi);
    const float err = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bp)), __fsub_rn(p, bp));
    hi = s;
    lo = __fadd_rn(lo, __fadd_rn(err, e));
  }
  __device__ __forceinline__ void flush() {
    total += static_cast<double>(hi);
    total += static_cast<double>(lo);
    hi = 0.0f;
    lo = 0.0f;
    pending = 0;
  }
  // The squares of one vector.  When all 8 lie in the compensated range (the
  // usual case) one branch per vector skips the per-element range tests and
  // their fp64 fallbacks; the operations on each square are those of add(),
  // in the same order, so the sum is the same.
  __device__ __forceinline__ void add_vec(const float (&g)[kVec]) {
    bool odd = false;
#pragma unroll
    for (int k = 0; k < kVec; ++k) {
      const float a = fabsf(g[k]);
      odd |= !(a >= 0x1p-40f && a < 0x1p50f);
    }
    if (odd) {
#pragma unroll
      for (int k = 0; k < kVec; ++k) add(g[k]);
      return;
    }
#pragma unroll
    for (int k = 0; k < kVec; ++k) {
      const float p = __fmul_rn(g[k], g[k]);
      const float e = __fmaf_rn(g[k], g[k], -p);
      const float s = __fadd_rn(hi, p);
      const float bp = __fsub_rn(s, hi);
      const float err = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bp)), __fsub_rn(p, bp));
      hi = s;
      lo = __fadd_rn(lo, __fadd_rn(err, e));
    }
  }
  // Called once per processed vector.
  __device__ __forceinline__ void tick() {
    if (++pending == 32) flush();
  }
  __device__ __forceinline__ double value() {
    flush();
    return total;
  }
};

// `sq` is uniform over the grid: whether the caller asked for the sum of squares.
// SQV: test the squares' range once per vector (SumSq::add_vec) instead of once
// per element; the same sum, faster or slower depending on the kernel.
template <bool SQV = false>
__device__ __forceinline__ void account(const float (&g)[kVec], bool sq, bool& bad, SumSq& ss) {
#pragma unroll
  for (int k = 0; k < kVec; ++k) bad |= non_finite(g[k]);
  if (sq) {
    if constexpr (SQV) {
      ss.add_vec(g);
    } else {
#pragma unroll
      for (int k = 0; k < kVec; ++k) ss.add(g[k]);
    }
    ss.tick();
  }
}

__device__ __forceinline__ void account1(float g, bool sq, bool& bad, SumSq& ss) {
  bad |= non_finite(g);
  if (sq) {
    ss.add(g);
    ss.tick();
  }
}

// Block-level OR of the flag and sum of the squares into the caller's words.
__device__ __forceinline__ void publish_to(int32_t* flag, double* sumsq, bool bad, SumSq& acc) {
  // Every thread of the block reaches this point exactly once.
  const int any_bad = __syncthreads_or(bad ? 1 : 0);
  if (threadIdx.x == 0 && any_bad && flag) atomicOr(flag, 1);
  if (sumsq) {
    double ss = acc.value();
    __shared__ double part[kThreads / 32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_down_sync(0xffffffffu, ss, o);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x == 0) {
      double t = 0.0;
#pragma unroll
      for (int k = 0; k < kThreads / 32; ++k) t += part[k];
      atomicAdd(sumsq, t);
    }
  }
}

__device__ __forceinline__ void publish(const KParams& p, bool bad, SumSq& acc) {
  publish_to(p.flag, p.sumsq, bad, acc);
}

// ---------------------------------------------------------------------------
// Kernels.  All are persistent grid-stride loops over the global range
// [p.lo, p.hi).  VEC kernels walk 8-element vectors aligned to global
// multiples of 8; a vector that is cut by the range ends or by a shard
// boundary falls back to per-element work.  Non-VEC kernels (some buffer is
// not 16-byte aligned) work element by element throughout.
// ---------------------------------------------------------------------------

// Per-element body of the fused step.
template <int GT>
__device__ __forceinline__ void fused_elem(const KParams& p, int P, int64_t i, bool sq, bool& bad,
                                           SumSq& ss) {
  const int r = owner_of(i, p, P);
  const float g = __fmul_rn(ring_sum_elem<GT>(p, P, r, i), p.scale);
  account1(g, sq, bad, ss);
  float w = p.w[i], m = ld_moment(p.m, i, p.mt), v = ld_moment(p.v, i, p.mt);
  adamw(w, m, v, g, p.ad);
  p.w[i] = w;
  st_moment(p.m, i, p.mt, m);
  st_moment(p.v, i, p.mt, v);
  const uint16_t b = to_bf16(w);
  for (int q = 0; q < P; ++q) p.rep[q][i] = b;
}

#ifndef ZDP_PDL
#define ZDP_PDL 1
#endif

// Programmatic dependent launch between consecutive k_fused launches of one
// call (disjoint bucket ranges): every block lets the next launch begin as
// soon as it starts, and waits for the previous launch to complete before it
// exits, so a launch completes only after all earlier ones.  Both are no-ops
// for a launch made without programmatic stream serialization.
__device__ __forceinline__ void allow_next_launch() {
#if ZDP_PDL
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#endif
}
__device__ __forceinline__ void wait_previous_launch() {
#if ZDP_PDL
  asm volatile("griddepcontrol.wait;" ::: "memory");
#endif
}

// Reduce-scatter + AdamW + cast + all-gather in one pass.  SQV: see account().
template <int PT, bool EXACT, int GT, bool VEC, bool SQV = false>
__global__ void __launch_bounds__(kThreads) k_fused(const __grid_constant__ KParams p) {
  allow_next_launch();
  const int P = ranks<PT, EXACT>(p);
  const bool sq = p.sumsq != nullptr;
  bool bad = false;
  SumSq ss;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  if constexpr (VEC) {
    const int64_t vlo = p.lo / kVec, vhi = (p.hi + kVec - 1) / kVec;
    for (int64_t vi = vlo + tid; vi < vhi; vi += stride) {
      const int64_t i0 = vi * kVec;
      const int r = owner_of(i0, p, P);
      if (i0 >= p.lo && i0 + kVec <= p.hi && i0 + kVec <= static_cast<int64_t>(r + 1) * p.S) {
        float w[kVec], m[kVec], v[kVec], g[kVec];
        ld_f8(p.w + i0, w);
        ld_moments8(p.m, p.v, p.mt, i0, m, v);
        ring_sum_vec<PT, EXACT, GT>(p, P, r, i0, g);
#pragma unroll
        for (int k = 0; k < kVec; ++k) g[k] = __fmul_rn(g[k], p.scale);
        account<SQV>(g, sq, bad, ss);
#pragma unroll
        for (int k = 0; k < kVec; ++k) adamw(w[k], m[k], v[k], g[k], p.ad);
        st_f8(p.w + i0, w);
        st_moments8(p.m, p.v, p.mt, i0, m, v);
        const uint4 b = pack_bf16x8(w);
#pragma unroll 8
        for (int q = 0; q < P; ++q) st16(p.rep[q] + i0, b);
      } else {
        for (int k = 0; k < kVec; ++k) {
          const int64_t i = i0 + k;
          if (i >= p.lo && i < p.hi) fused_elem<GT>(p, P, i, sq, bad, ss);
        }
      }
    }
  } else {
    for (int64_t i = p.lo + tid; i < p.hi; i += stride) fused_elem<GT>(p, P, i, sq, bad, ss);
  }
  publish(p, bad, ss);
  wait_previous_launch();
}

// The fused step for exactly P <= 8 ranks with the moment type MT fixed at
// compile time, and MINB resident blocks per SM asked of the register
// allocator (__launch_bounds__).  The operations and their order are those
// of k_fused, which carries the code of both moment types.  It runs where it
// measured faster (pick_fused_mt in kernels_grad.inc), most of all for bf16
// moments at P = 1 and 2: there k_fused is bound by instruction issue and
// latency (0.78 and 0.84 of the copy ceiling on GB300) and this kernel at 8
// blocks per SM runs 0.93 and 0.94.
template <int P, int GT, int MT, bool SQV, int MINB>
__global__ void __launch_bounds__(kThreads, MINB) k_fused_mt(const __grid_constant__ KParams p) {
  allow_next_launch();
  const bool sq = p.sumsq != nullptr;
  bool bad = false;
  SumSq ss;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  const int64_t vlo = p.lo / kVec, vhi = (p.hi + kVec - 1) / kVec;
  for (int64_t vi = vlo + tid; vi < vhi; vi += stride) {
    const int64_t i0 = vi * kVec;
    const int r = owner_of(i0, p, P);
    if (i0 >= p.lo && i0 + kVec <= p.hi && i0 + kVec <= static_cast<int64_t>(r + 1) * p.S) {
      float w[kVec], m[kVec], v[kVec], g[kVec];
      ld_f8(p.w + i0, w);
      ld_moments8(p.m, p.v, MT, i0, m, v);
      ring_sum_vec<P, true, GT>(p, P, r, i0, g);
#pragma unroll
      for (int k = 0; k < kVec; ++k) g[k] = __fmul_rn(g[k], p.scale);
      account<SQV>(g, sq, bad, ss);
#pragma unroll
      for (int k = 0; k < kVec; ++k) adamw(w[k], m[k], v[k], g[k], p.ad);
      st_f8(p.w + i0, w);
      st_moments8(p.m, p.v, MT, i0, m, v);
      const uint4 b = pack_bf16x8(w);
#pragma unroll
      for (int q = 0; q < P; ++q) st16(p.rep[q] + i0, b);
    } else {
      for (int k = 0; k < kVec; ++k) {
        const int64_t i = i0 + k;
        if (i >= p.lo && i < p.hi) fused_elem<GT>(p, P, i, sq, bad, ss);
      }
    }
  }
  publish(p, bad, ss);
  wait_previous_launch();
}

// Reduce-scatter only: reduced gradients to gout.
template <int PT, bool EXACT, int GT, bool VEC>
__global__ void __launch_bounds__(kThreads) k_reduce(const __grid_constant__ KParams p) {
  allow_next_launch();
  const int P = ranks<PT, EXACT>(p);
  const bool sq = p.sumsq != nullptr;
  bool bad = false;
  SumSq ss;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  if constexpr (VEC) {
    const int64_t vlo = p.lo / kVec, vhi = (p.hi + kVec - 1) / kVec;
    for (int64_t vi = vlo + tid; vi < vhi; vi += stride) {
      const int64_t i0 = vi * kVec;
      const int r = owner_of(i0, p, P);
      if (i0 >= p.lo && i0 + kVec <= p.hi && i0 + kVec <= static_cast<int64_t>(r + 1) * p.S) {
        float g[kVec];
        ring_sum_vec<PT, EXACT, GT>(p, P, r, i0, g);
#pragma unroll
        for (int k = 0; k < kVec; ++k) g[k] = __fmul_rn(g[k], p.scale);
        account(g, sq, bad, ss);
        st_f8(p.gout + (i0 - p.gout_base), g);
      } else {
        for (int k = 0; k < kVec; ++k) {
          const int64_t i = i0 + k;
          if (i >= p.lo && i < p.hi) {
            const float g = __fmul_rn(ring_sum_elem<GT>(p, P, owner_of(i, p, P), i), p.scale);
            account1(g, sq, bad, ss);
            p.gout[i - p.gout_base] = g;
          }
        }
      }
    }
  } else {
    for (int64_t i = p.lo + tid; i < p.hi; i += stride) {
      const float g = __fmul_rn(ring_sum_elem<GT>(p, P, owner_of(i, p, P), i), p.scale);
      account1(g, sq, bad, ss);
      p.gout[i - p.gout_base] = g;
    }
  }
  publish(p, bad, ss);
  wait_previous_launch();
}

// AdamW from reduced gradients gin, then cast + all-gather into nrep
// replicas.  With a gate, nothing is written when *gate != 0.
template <bool VEC>
__global__ void __launch_bounds__(kThreads) k_adam_gather(const __grid_constant__ KParams p) {
  allow_next_launch();
  if (p.gate && *p.gate) {  // uniform over the grid: the whole launch writes nothing
    if (blockIdx.x == 0 && threadIdx.x == 0 && p.flag) atomicOr(p.flag, 1);
    wait_previous_launch();
    return;
  }
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  if constexpr (VEC) {
    const int64_t vlo = p.lo / kVec, vhi = (p.hi + kVec - 1) / kVec;
    for (int64_t vi = vlo + tid; vi < vhi; vi += stride) {
      const int64_t i0 = vi * kVec;
      if (i0 >= p.lo && i0 + kVec <= p.hi) {
        float w[kVec], m[kVec], v[kVec], g[kVec];
        ld_f8(p.w + i0, w);
        ld_moments8(p.m, p.v, p.mt, i0, m, v);
        ld_f8(p.gin + (i0 - p.gin_base), g);
#pragma unroll
        for (int k = 0; k < kVec; ++k) adamw(w[k], m[k], v[k], g[k], p.ad);
        st_f8(p.w + i0, w);
        st_moments8(p.m, p.v, p.mt, i0, m, v);
        if (p.nrep > 0) {
          const uint4 b = pack_bf16x8(w);
          for (int q = 0; q < p.nrep; ++q) st16(p.rep[q] + i0, b);
        }
      } else {
        for (int k = 0; k < kVec; ++k) {
          const int64_t i = i0 + k;
          if (i >= p.lo && i < p.hi) {
            float w = p.w[i], m = ld_moment(p.m, i, p.mt), v = ld_moment(p.v, i, p.mt);
            adamw(w, m, v, p.gin[i - p.gin_base], p.ad);
            p.w[i] = w;
            st_moment(p.m, i, p.mt, m);
            st_moment(p.v, i, p.mt, v);
            const uint16_t b = to_bf16(w);
            for (int q = 0; q < p.nrep; ++q) p.rep[q][i] = b;
          }
        }
      }
    }
  } else {
    for (int64_t i = p.lo + tid; i < p.hi; i += stride) {
      float w = p.w[i], m = ld_moment(p.m, i, p.mt), v = ld_moment(p.v, i, p.mt);
      adamw(w, m, v, p.gin[i - p.gin_base], p.ad);
      p.w[i] = w;
      st_moment(p.m, i, p.mt, m);
      st_moment(p.v, i, p.mt, v);
      const uint16_t b = to_bf16(w);
      for (int q = 0; q < p.nrep; ++q) p.rep[q][i] = b;
    }
  }
  wait_previous_launch();
}

// k_adam_gather's vector path with the replica count and the moment type
// fixed at compile time (the same operations in the same order).  Measured
// on GB300 against k_adam_gather: the checked two-pass 1.3B step at P = 8
// with fp32 moments 13.12 -> 12.88 ms; slower for bf16 moments (11.31 ->
// 11.62), for AdamW without replicas and for the checked step at P = 2 and 4
// (1-3 %), so only 8 replicas with fp32 moments run it (launch_adam_gather).
// (__launch_bounds__ names its minimum of one block explicitly: that is the
// register allocation that was measured.)
template <int NREP, int MT>
__global__ void __launch_bounds__(kThreads, 1) k_adam_gather_mt(const __grid_constant__ KParams p) {
  allow_next_launch();
  if (p.gate && *p.gate) {
    if (blockIdx.x == 0 && threadIdx.x == 0 && p.flag) atomicOr(p.flag, 1);
    wait_previous_launch();
    return;
  }
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  const int64_t vlo = p.lo / kVec, vhi = (p.hi + kVec - 1) / kVec;
  for (int64_t vi = vlo + tid; vi < vhi; vi += stride) {
    const int64_t i0 = vi * kVec;
    if (i0 >= p.lo && i0 + kVec <= p.hi) {
      float w[kVec], m[kVec], v[kVec], g[kVec];
      ld_f8(p.w + i0, w);
      ld_moments8(p.m, p.v, MT, i0, m, v);
      ld_f8(p.gin + (i0 - p.gin_base), g);
#pragma unroll
      for (int k = 0; k < kVec; ++k) adamw(w[k], m[k], v[k], g[k], p.ad);
      st_f8(p.w + i0, w);
      st_moments8(p.m, p.v, MT, i0, m, v);
      if constexpr (NREP > 0) {
        const uint4 b = pack_bf16x8(w);
#pragma unroll
        for (int q = 0; q < NREP; ++q) st16(p.rep[q] + i0, b);
      }
    } else {
      for (int k = 0; k < kVec; ++k) {
        const int64_t i = i0 + k;
        if (i >= p.lo && i < p.hi) {
          float w = p.w[i], m = ld_moment(p.m, i, MT), v = ld_moment(p.v, i, MT);
          adamw(w, m, v, p.gin[i - p.gin_base], p.ad);
          p.w[i] = w;
          st_moment(p.m, i, MT, m);
          st_moment(p.v, i, MT, v);
          const uint16_t b = to_bf16(w);
          for (int q = 0; q < NREP; ++q) p.rep[q][i] = b;
        }
      }
    }
  }
  wait_previous_launch();
}

// Cast + all-gather: rep[q][i] = bf16(w[i]).
template <bool VEC>
__global__ void __launch_bounds__(kThreads) k_gather(const __grid_constant__ KParams p) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  if constexpr (VEC) {
    const int64_t vlo = p.lo / kVec, vhi = (p.hi + kVec - 1) / kVec;
    for (int64_t vi = vlo + tid; vi < vhi; vi += stride) {
      const int64_t i0 = vi * kVec;
      if (i0 >= p.lo && i0 + kVec <= p.hi) {
        float w[kVec];
        ld_f8(p.w + i0, w);
        const uint4 b = pack_bf16x8(w);
        for (int q = 0; q < p.nrep; ++q) st16(p.rep[q] + i0, b);
      } else {
        for (int k = 0; k < kVec; ++k) {
          const int64_t i = i0 + k;
          if (i >= p.lo && i < p.hi) {
            const uint16_t b = to_bf16(p.w[i]);
            for (int q = 0; q < p.nrep; ++q) p.rep[q][i] = b;
          }
        }
      }
    }
  } else {
    for (int64_t i = p.lo + tid; i < p.hi; i += stride) {
      const uint16_t b = to_bf16(p.w[i]);
      for (int q = 0; q < p.nrep; ++q) p.rep[q][i] = b;
    }
  }
}

}  // namespace zdp
