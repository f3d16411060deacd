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
//  * every load of a vector is issued before the first add consumes one, so
//    a thread keeps (2P + 24) * 8 bytes in flight; with P > 8 the ranks are
//    loaded in groups of 8 with the next group's loads issued before the
//    current group's adds;
//  * persistent grid-stride grids sized to resident blocks x SMs;
//  * streaming cache hints (evict-first) on every access: nothing is reused.
// Numerics: the ring sum adds in a fixed order with __fadd_rn and the AdamW
// update uses only *_rn intrinsics, so no multiply-add is ever contracted and
// every result is the IEEE fp32 result of the stated formula.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "zdp_internal.h"

#ifndef ZDP_CONTIG
#define ZDP_CONTIG 0  // 1: block-contiguous spans instead of a grid-wide stride (fused kernel)
#endif

#ifndef ZDP_SQ_FP64
#define ZDP_SQ_FP64 0  // 1: accumulate the sum of squares with one fp64 fma per element
#endif

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
__device__ __forceinline__ int owner_of(int64_t i, const KParams& p, int P) {
  int r = static_cast<int>(static_cast<float>(i) * p.inv_s);
  r = r > P - 1 ? P - 1 : r;
  if (static_cast<int64_t>(r) * p.S > i) {
    --r;
  } else if (static_cast<int64_t>(r + 1) * p.S <= i) {
    ++r;
  }
  // i < n <= P*S keeps r in [0, P-1]; the clamp makes that hold for any input.
  return r < 0 ? 0 : (r > P - 1 ? P - 1 : r);
}

// ---------------------------------------------------------------------------
// Memory access with streaming (evict-first) hints.
// ---------------------------------------------------------------------------
#ifndef ZDP_LD_HINT
#define ZDP_LD_HINT 0  // 0 ld.global.cs, 1 ld.global.nc.L1::no_allocate, 2 ld.global
#endif
#ifndef ZDP_ST_HINT
#define ZDP_ST_HINT 0  // 0 st.global.cs, 1 st.global
#endif
__device__ __forceinline__ uint4 ld16(const void* ptr) {
#if ZDP_LD_HINT == 0
  return __ldcs(reinterpret_cast<const uint4*>(ptr));
#elif ZDP_LD_HINT == 1
  uint4 x;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(x.x), "=r"(x.y), "=r"(x.z), "=r"(x.w)
               : "l"(ptr));
  return x;
#else
  return *reinterpret_cast<const uint4*>(ptr);
#endif
}
__device__ __forceinline__ void st16(void* ptr, uint4 x) {
#if ZDP_ST_HINT == 0
  __stcs(reinterpret_cast<uint4*>(ptr), x);
#else
  *reinterpret_cast<uint4*>(ptr) = x;
#endif
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

// Loads ranks q, q+1, ... (mod P) into d[0..cnt) and advances q.
template <int GT>
__device__ __forceinline__ void load_group(const KParams& p, int P, int& q, int cnt,
                                           int64_t i0, uint4 (&d)[8]) {
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    if (k < cnt) {
      d[k] = ld16(grad_vec<GT>(p, q, i0));
      q = ring_next(q, P);
    }
  }
}

template <int GT>
__device__ __forceinline__ void add_group(int cnt, bool first, const uint4 (&d)[8],
                                          float (&acc)[kVec]) {
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    if (k < cnt) {
      if (first && k == 0) {
        vec_set<GT>(acc, d[0]);
      } else {
        vec_add<GT>(acc, d[k]);
      }
    }
  }
}

// Vector of 8 elements starting at i0 (a multiple of 8), all owned by r.
// PT > 0: P known at compile time.
template <int PT, int GT>
__device__ __forceinline__ void ring_sum_vec(const KParams& p, int P, int r, int64_t i0,
                                             float (&acc)[kVec]) {
  int q = ring_next(r, P);
  if constexpr (PT >= 1 && PT <= 8) {
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
    // Groups of 8 ranks, two buffers: the loads of group k+1 are issued
    // before the adds of group k.
    uint4 a[8], b[8];
    int left = P;
    int ca = left < 8 ? left : 8;
    load_group<GT>(p, P, q, ca, i0, a);
    left -= ca;
    bool first = true;
    while (true) {
      const int cb = left < 8 ? left : 8;
      load_group<GT>(p, P, q, cb, i0, b);
      left -= cb;
      add_group<GT>(ca, first, a, acc);
      first = false;
      if (cb == 0) break;
      ca = left < 8 ? left : 8;
      load_group<GT>(p, P, q, ca, i0, a);
      left -= ca;
      add_group<GT>(cb, false, b, acc);
      if (ca == 0) break;
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
#if ZDP_SQ_FP64
    const double d = static_cast<double>(g);
    total = __fma_rn(d, d, total);
#else
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
#endif
  }
  __device__ __forceinline__ void flush() {
    total += static_cast<double>(hi);
    total += static_cast<double>(lo);
    hi = 0.0f;
    lo = 0.0f;
    pending = 0;
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

template <bool SQ>
__device__ __forceinline__ void account(const float (&g)[kVec], bool& bad, SumSq& ss) {
#pragma unroll
  for (int k = 0; k < kVec; ++k) {
    bad |= non_finite(g[k]);
    if constexpr (SQ) ss.add(g[k]);
  }
  if constexpr (SQ) ss.tick();
}

template <bool SQ>
__device__ __forceinline__ void account1(float g, bool& bad, SumSq& ss) {
  bad |= non_finite(g);
  if constexpr (SQ) {
    ss.add(g);
    ss.tick();
  }
}

template <bool SQ, int NT>
__device__ __forceinline__ void publish_n(const KParams& p, bool bad, SumSq& acc) {
  // Every thread of the block reaches this point exactly once.
  const int any_bad = __syncthreads_or(bad ? 1 : 0);
  if (threadIdx.x == 0 && any_bad && p.flag) atomicOr(p.flag, 1);
  if constexpr (SQ) {
    double ss = acc.value();
    __shared__ double part[NT / 32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_down_sync(0xffffffffu, ss, o);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x == 0 && p.sumsq) {
      double t = 0.0;
#pragma unroll
      for (int k = 0; k < NT / 32; ++k) t += part[k];
      atomicAdd(p.sumsq, t);
    }
  }
}

template <bool SQ>
__device__ __forceinline__ void publish(const KParams& p, bool bad, SumSq& acc) {
  publish_n<SQ, kThreads>(p, bad, acc);
}

// ---------------------------------------------------------------------------
// Kernels.  All are persistent grid-stride loops over the global range
// [p.lo, p.hi).  VEC kernels walk 8-element vectors aligned to global
// multiples of 8; a vector that is cut by the range ends or by a shard
// boundary falls back to per-element work.
// ---------------------------------------------------------------------------

// Per-element body of the fused step.
template <int GT, bool SQ>
__device__ __forceinline__ void fused_elem(const KParams& p, int P, int64_t i, bool& bad,
                                           SumSq& ss) {
  const int r = owner_of(i, p, P);
  const float g = __fmul_rn(ring_sum_elem<GT>(p, P, r, i), p.scale);
  account1<SQ>(g, bad, ss);
  float w = p.w[i], m = p.m[i], v = p.v[i];
  adamw(w, m, v, g, p.ad);
  p.w[i] = w;
  p.m[i] = m;
  p.v[i] = v;
  const uint16_t b = to_bf16(w);
  for (int q = 0; q < P; ++q) p.rep[q][i] = b;
}

// Reduce-scatter + AdamW + cast + all-gather in one pass.
template <int PT, int GT, bool SQ, bool VEC>
__global__ void __launch_bounds__(kThreads) k_fused(const __grid_constant__ KParams p) {
  const int P = PT > 0 ? PT : p.P;
  bool bad = false;
  SumSq ss;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  if constexpr (VEC) {
#if ZDP_CONTIG
    // each block walks its own contiguous span of vectors
    const int64_t nv = (p.hi + kVec - 1) / kVec - p.lo / kVec;
    const int64_t span = (nv + gridDim.x - 1) / gridDim.x;
    const int64_t vlo = p.lo / kVec + static_cast<int64_t>(blockIdx.x) * span;
    const int64_t vend = (p.hi + kVec - 1) / kVec;
    const int64_t vhi = vlo + span < vend ? vlo + span : vend;
    for (int64_t vi = vlo + threadIdx.x; vi < vhi; vi += kThreads) {
#else
    const int64_t vlo = p.lo / kVec, vhi = (p.hi + kVec - 1) / kVec;
    for (int64_t vi = vlo + tid; vi < vhi; vi += stride) {
#endif
      const int64_t i0 = vi * kVec;
      const int r = owner_of(i0, p, P);
      if (i0 >= p.lo && i0 + kVec <= p.hi && i0 + kVec <= static_cast<int64_t>(r + 1) * p.S) {
        float w[kVec], m[kVec], v[kVec], g[kVec];
        ld_f8(p.w + i0, w);
        ld_f8(p.m + i0, m);
        ld_f8(p.v + i0, v);
        ring_sum_vec<PT, GT>(p, P, r, i0, g);
#pragma unroll
        for (int k = 0; k < kVec; ++k) g[k] = __fmul_rn(g[k], p.scale);
        account<SQ>(g, bad, ss);
#pragma unroll
        for (int k = 0; k < kVec; ++k) adamw(w[k], m[k], v[k], g[k], p.ad);
        st_f8(p.w + i0, w);
        st_f8(p.m + i0, m);
        st_f8(p.v + i0, v);
        const uint4 b = pack_bf16x8(w);
#pragma unroll 8
        for (int q = 0; q < P; ++q) st16(p.rep[q] + i0, b);
      } else {
        for (int k = 0; k < kVec; ++k) {
          const int64_t i = i0 + k;
          if (i >= p.lo && i < p.hi) fused_elem<GT, SQ>(p, P, i, bad, ss);
        }
      }
    }
  } else {
    for (int64_t i = p.lo + tid; i < p.hi; i += stride) fused_elem<GT, SQ>(p, P, i, bad, ss);
  }
  publish<SQ>(p, bad, ss);
}

// ---------------------------------------------------------------------------
// TMA-staged fused step.
//
// One CTA per SM.  Warp 0 lane 0 is the producer: for every tile of kTileE
// elements it issues 1-D bulk copies (cp.async.bulk, the TMA engine) of the
// P gradient slices and the master/m/v slices into one stage of a ring of
// shared-memory buffers, completion counted on that stage's "full" mbarrier.
// Warps 1..kConsumerWarps compute: each thread takes one 8-element vector of
// the tile from shared memory, runs the ring sum and AdamW in registers and
// stores state and replicas straight to HBM; each warp then arrives on the
// stage's "empty" mbarrier so the producer can refill it.  Memory latency is
// hidden by the stages in flight, independently of how long the AdamW chain
// of a tile takes.
//
// Every wait is bounded: after kWaitLimitNs of %globaltimer a waiting thread
// raises ZDP_STATUS_TIMEOUT in the status word and the CTA stops; the
// producer then waits (bounded again) until every copy it issued has landed,
// so no bulk copy is still writing shared memory when the CTA exits.
// ---------------------------------------------------------------------------
constexpr int kConsumerWarps = 8;
constexpr int kTileE = kConsumerWarps * 32 * kVec;   // 2048 elements per tile
constexpr int kTmaThreads = 32 * (1 + kConsumerWarps);
constexpr uint64_t kWaitLimitNs = 2000000000ull;      // 2 s
constexpr int kMaxStages = 8;
constexpr int kTmaSmemBudget = 200 * 1024;

__host__ __device__ constexpr int tma_stage_bytes(int P) {
  return P * kTileE * 2 + 3 * kTileE * 4;
}
__host__ __device__ constexpr int tma_stages(int P) {
  return kTmaSmemBudget / tma_stage_bytes(P) < kMaxStages ? kTmaSmemBudget / tma_stage_bytes(P)
                                                          : kMaxStages;
}
__host__ __device__ constexpr int tma_smem_bytes(int P) {
  return tma_stages(P) * tma_stage_bytes(P) + 2 * kMaxStages * 8 + 128;
}

__device__ __forceinline__ uint32_t smem_addr(const void* ptr) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(ptr));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Waits for the phase with the given parity to complete; false after the
// time limit or once another thread of the CTA has aborted.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          volatile int* abort_flag) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (true) {
#pragma unroll 1
    for (int k = 0; k < 32; ++k)
      if (mbar_test(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_ns() - t0 > kWaitLimitNs) return false;
  }
}
__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(pol)
      : "memory");
}

template <int GT>
__device__ __forceinline__ uint4 lds16(const void* ptr) {
  uint4 x;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(x.x), "=r"(x.y), "=r"(x.z), "=r"(x.w)
               : "r"(smem_addr(ptr)));
  return x;
}

__device__ __forceinline__ void lds_f8(const float* ptr, float (&x)[kVec]) {
  const uint4 a = lds16<0>(ptr);
  const uint4 b = lds16<0>(ptr + 4);
  x[0] = __uint_as_float(a.x); x[1] = __uint_as_float(a.y);
  x[2] = __uint_as_float(a.z); x[3] = __uint_as_float(a.w);
  x[4] = __uint_as_float(b.x); x[5] = __uint_as_float(b.y);
  x[6] = __uint_as_float(b.z); x[7] = __uint_as_float(b.w);
}

// Requires: every buffer's element 0 16-byte aligned (the VEC condition).
// Processes [p.lo, p.hi): the 8-aligned interior through the TMA pipeline,
// the (< 8 + < 8) ragged ends per element by block 0.
template <int PT, int GT, bool SQ>
__global__ void __launch_bounds__(kTmaThreads, 1) k_fused_tma(const __grid_constant__ KParams p) {
  constexpr int P = PT;
  constexpr int NS = tma_stages(PT);
  constexpr int SB = tma_stage_bytes(PT);
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + NS * SB);
  uint64_t* empty = full + kMaxStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kMaxStages);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  bool bad = false;
  SumSq ss;

  const int64_t a0 = (p.lo + kVec - 1) / kVec * kVec;  // aligned interior [a0, a1)
  const int64_t a1 = p.hi / kVec * kVec > a0 ? p.hi / kVec * kVec : a0;
  const int64_t ntiles = (a1 - a0 + kTileE - 1) / kTileE;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol = evict_first_policy();
      int64_t issued = 0;
      bool ok = true;
      for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++issued) {
        const int s = static_cast<int>(issued % NS);
        if (issued >= NS &&
            !mbar_wait(&empty[s], static_cast<uint32_t>(((issued / NS) - 1) & 1), abort_flag)) {
          ok = false;
          break;
        }
        const int64_t e0 = a0 + t * kTileE;
        const int cnt = static_cast<int>(a1 - e0 < kTileE ? a1 - e0 : kTileE);
        unsigned char* st = smem + s * SB;
        mbar_expect_tx(&full[s], static_cast<uint32_t>(cnt) * (2u * P + 12u));
#pragma unroll
        for (int q = 0; q < P; ++q)
          bulk_load(st + q * kTileE * 2, grad_vec<GT>(p, q, e0), cnt * 2, &full[s], pol);
        unsigned char* sw = st + P * kTileE * 2;
        bulk_load(sw, p.w + e0, cnt * 4, &full[s], pol);
        bulk_load(sw + kTileE * 4, p.m + e0, cnt * 4, &full[s], pol);
        bulk_load(sw + 2 * kTileE * 4, p.v + e0, cnt * 4, &full[s], pol);
      }
      if (!ok) {
        if (p.status) atomicOr(p.status, ZDP_STATUS_TIMEOUT);
        *abort_flag = 1;
      }
      // No bulk copy may still be writing shared memory when the CTA exits:
      // wait (bounded) until the last copy of every stage has landed.
      const int64_t first = issued > NS ? issued - NS : 0;
      for (int64_t k = first; k < issued; ++k) {
        const int s = static_cast<int>(k % NS);
        const uint64_t t0 = global_ns();
        while (!mbar_test(&full[s], static_cast<uint32_t>((k / NS) & 1))) {
          if (global_ns() - t0 > kWaitLimitNs) {
            if (p.status) atomicOr(p.status, ZDP_STATUS_TIMEOUT);
            break;
          }
        }
      }
    }
  } else {
    const int c = threadIdx.x - 32;  // consumer thread 0..255
    int64_t k = 0;
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++k) {
      const int s = static_cast<int>(k % NS);
      if (!mbar_wait(&full[s], static_cast<uint32_t>((k / NS) & 1), abort_flag)) {
        if (p.status) atomicOr(p.status, ZDP_STATUS_TIMEOUT);
        *abort_flag = 1;
        break;
      }
      const int64_t e0 = a0 + t * kTileE;
      const int cnt = static_cast<int>(a1 - e0 < kTileE ? a1 - e0 : kTileE);
      const unsigned char* st = smem + s * SB;
      const bool active = c * kVec < cnt;
      const int64_t i0 = e0 + c * kVec;
      float w[kVec], m[kVec], v[kVec], g[kVec];
      if (active) {
        const float* sw = reinterpret_cast<const float*>(st + P * kTileE * 2);
        lds_f8(sw + c * kVec, w);
        lds_f8(sw + kTileE + c * kVec, m);
        lds_f8(sw + 2 * kTileE + c * kVec, v);
        const int r = owner_of(i0, p, P);
        if (i0 + kVec <= static_cast<int64_t>(r + 1) * p.S) {
          int q = ring_next(r, P);
          uint4 d[P];
#pragma unroll
          for (int j = 0; j < P; ++j) {
            d[j] = lds16<GT>(st + q * kTileE * 2 + c * 16);
            q = ring_next(q, P);
          }
          vec_set<GT>(g, d[0]);
#pragma unroll
          for (int j = 1; j < P; ++j) vec_add<GT>(g, d[j]);
        } else {
          // the vector straddles a shard boundary: per-element ring order
          const uint16_t* sg = reinterpret_cast<const uint16_t*>(st);
#pragma unroll 1
          for (int e = 0; e < kVec; ++e) {
            const int re = owner_of(i0 + e, p, P);
            int q = ring_next(re, P);
            float acc = widen1<GT>(sg[q * kTileE + c * kVec + e]);
            for (int j = 1; j < P; ++j) {
              q = ring_next(q, P);
              acc = __fadd_rn(acc, widen1<GT>(sg[q * kTileE + c * kVec + e]));
            }
            g[e] = acc;
          }
        }
      }
      // Every lane of the warp has read what it needs from stage s.
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      if (active) {
#pragma unroll
        for (int e = 0; e < kVec; ++e) g[e] = __fmul_rn(g[e], p.scale);
        account<SQ>(g, bad, ss);
#pragma unroll
        for (int e = 0; e < kVec; ++e) adamw(w[e], m[e], v[e], g[e], p.ad);
        st_f8(p.w + i0, w);
        st_f8(p.m + i0, m);
        st_f8(p.v + i0, v);
        const uint4 b = pack_bf16x8(w);
#pragma unroll
        for (int q = 0; q < P; ++q) st16(p.rep[q] + i0, b);
      }
    }
    // ragged ends of the range, outside the 8-aligned interior
    if (blockIdx.x == 0) {
      const int64_t head = a0 < p.hi ? a0 - p.lo : p.hi - p.lo;
      if (c < head) fused_elem<GT, SQ>(p, P, p.lo + c, bad, ss);
      const int64_t tail_lo = a1 > p.lo + head ? a1 : p.lo + head;
      if (c < p.hi - tail_lo) fused_elem<GT, SQ>(p, P, tail_lo + c, bad, ss);
    }
  }
  publish_n<SQ, kTmaThreads>(p, bad, ss);
}

// Reduce-scatter only: reduced gradients to gout.
template <int PT, int GT, bool SQ, bool VEC>
__global__ void __launch_bounds__(kThreads) k_reduce(const __grid_constant__ KParams p) {
  const int P = PT > 0 ? PT : p.P;
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
        ring_sum_vec<PT, GT>(p, P, r, i0, g);
#pragma unroll
        for (int k = 0; k < kVec; ++k) g[k] = __fmul_rn(g[k], p.scale);
        account<SQ>(g, bad, ss);
        st_f8(p.gout + (i0 - p.gout_base), g);
      } else {
        for (int k = 0; k < kVec; ++k) {
          const int64_t i = i0 + k;
          if (i >= p.lo && i < p.hi) {
            const float g = __fmul_rn(ring_sum_elem<GT>(p, P, owner_of(i, p, P), i), p.scale);
            account1<SQ>(g, bad, ss);
            p.gout[i - p.gout_base] = g;
          }
        }
      }
    }
  } else {
    for (int64_t i = p.lo + tid; i < p.hi; i += stride) {
      const float g = __fmul_rn(ring_sum_elem<GT>(p, P, owner_of(i, p, P), i), p.scale);
      account1<SQ>(g, bad, ss);
      p.gout[i - p.gout_base] = g;
    }
  }
  publish<SQ>(p, bad, ss);
}

// AdamW from reduced gradients gin, then cast + all-gather into nrep
// replicas.  With a gate, nothing is written when *gate != 0.
template <bool VEC>
__global__ void __launch_bounds__(kThreads) k_adam_gather(const __grid_constant__ KParams p) {
  if (p.gate && *p.gate) {  // uniform over the grid: the whole launch writes nothing
    if (blockIdx.x == 0 && threadIdx.x == 0 && p.flag) atomicOr(p.flag, 1);
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
        ld_f8(p.m + i0, m);
        ld_f8(p.v + i0, v);
        ld_f8(p.gin + (i0 - p.gin_base), g);
#pragma unroll
        for (int k = 0; k < kVec; ++k) adamw(w[k], m[k], v[k], g[k], p.ad);
        st_f8(p.w + i0, w);
        st_f8(p.m + i0, m);
        st_f8(p.v + i0, v);
        if (p.nrep > 0) {
          const uint4 b = pack_bf16x8(w);
          for (int q = 0; q < p.nrep; ++q) st16(p.rep[q] + i0, b);
        }
      } else {
        for (int k = 0; k < kVec; ++k) {
          const int64_t i = i0 + k;
          if (i >= p.lo && i < p.hi) {
            float w = p.w[i], m = p.m[i], v = p.v[i];
            adamw(w, m, v, p.gin[i - p.gin_base], p.ad);
            p.w[i] = w;
            p.m[i] = m;
            p.v[i] = v;
            const uint16_t b = to_bf16(w);
            for (int q = 0; q < p.nrep; ++q) p.rep[q][i] = b;
          }
        }
      }
    }
  } else {
    for (int64_t i = p.lo + tid; i < p.hi; i += stride) {
      float w = p.w[i], m = p.m[i], v = p.v[i];
      adamw(w, m, v, p.gin[i - p.gin_base], p.ad);
      p.w[i] = w;
      p.m[i] = m;
      p.v[i] = v;
      const uint16_t b = to_bf16(w);
      for (int q = 0; q < p.nrep; ++q) p.rep[q][i] = b;
    }
  }
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
