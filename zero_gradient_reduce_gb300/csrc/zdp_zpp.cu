// zdp_zpp.cu -- the ZeRO++ variant of the step (Fudan MLSys ch. 9, 9.4.3):
// gradients arrive quantized block-wise to int8 for the reduce-scatter, and
// the all-gather writes int8 replicas of the bf16 parameters.  Blocks are
// 256 consecutive elements (global index i in block i / 256); a block's scale
// is max|x| / 127, q = x / scale rounded half to even, clamped to +-127, and
// an all-zero block has scale 0.  Dequantization is q * scale in fp32.
//
// One warp owns one 256-element block at a time (lane l: elements
// 8l .. 8l+7), so the block maximum needed by the quantizer is one warp
// reduction; the loops over blocks are warp-uniform.
#include <algorithm>
#include <cstring>
#include <type_traits>

#include "zdp_kernels.cuh"

namespace zdp {
namespace {

constexpr int kQB = ZDP_QBLOCK;  // elements per quantization block (256 = 32 lanes x 8)

struct ZppParams {
  const int8_t* g[ZDP_MAX_P];   // rank q's int8 gradient of element i: g[q][i - off]
  const float* gs[ZDP_MAX_P];   // its scales: gs[q][i/256 - off/256]
  int8_t* rq[ZDP_MAX_P];        // rank q's int8 replica: rq[q][i]
  float* rs[ZDP_MAX_P];         // its scales: rs[q][i/256]
  float* w;
  void* m;
  void* v;
  int mt;
  int64_t n, S, off, lo, hi;
  float inv_s;
  int P;
  float scale;
  AdamK ad;
  int32_t* flag;
  double* sumsq;
};

__device__ __forceinline__ int zpp_owner(int64_t i, const ZppParams& p) {
  return owner_calc(i, p.S, p.inv_s, p.P);
}

__device__ __forceinline__ float dequant(int8_t q, float scale) {
  return __fmul_rn(__int2float_rn(q), scale);
}

// Reference form of the code: exact division, round half to even, clamp.  A
// NaN quotient (x / NaN, or inf / inf) clamps to -127: fmaxf returns its
// non-NaN operand.
__device__ __forceinline__ int quant_div(float x, float scale) {
  float r = rintf(__fdiv_rn(x, scale));
  r = fminf(fmaxf(r, -127.0f), 127.0f);
  return __float2int_rn(r);
}

// The same code from a multiply by rcp = fl(1/scale), without conversion
// instructions.  Adding 1.5 * 2^23 rounds y to an integer, half to even, and
// leaves that integer in the low mantissa bits.  Since |x| <= 128 * scale,
// y = fl(x * rcp) lies within 128 * 2^-23 < 2e-5 of x / scale, and
// fl(x / scale) within 128 * 2^-24 of it; unless y is within 1e-4 of a
// half-integer both round to the same integer.  Otherwise (and for NaN) the
// exact division decides.  The caller guarantees scale != 0 and rcp finite.
__device__ __forceinline__ int quant_rcp(float x, float scale, float rcp) {
  const float y = __fmul_rn(x, rcp);
  const float t = __fadd_rn(y, 12582912.0f);
  const float d = __fsub_rn(y, __fsub_rn(t, 12582912.0f));  // exact: y minus its rounding
  if (fabsf(__fsub_rn(fabsf(d), 0.5f)) > 1e-4f) {
    const int q = __float_as_int(t) - 0x4B400000;
    return q < -127 ? -127 : (q > 127 ? 127 : q);
  }
  return quant_div(x, scale);
}

// Codes of 8 values sharing one block scale (0 for an all-zero block).
// With a normal, finite scale (the usual case) every |x| <= 127 * scale is
// finite and rcp = fl(1/scale) is within 2^-24 of 1/scale, so
// |y| = |fl(x * rcp)| < 127 * (1 + 2^-22) < 127.5 and the rounded code needs
// no clamp; the 8 codes take the multiply path with one test for all of
// them (none of the 8 within 1e-4 of a half-integer), the same test as
// quant_rcp's per element.  ONE_TEST = false keeps the per-element form
// (quant_rcp) throughout: the kernels of 16 or more ranks spill registers
// with the other.
template <bool ONE_TEST = true>
__device__ __forceinline__ void quant8(const float (&x)[kVec], float scale, int (&q)[kVec]) {
  const float rcp = __frcp_rn(scale);
  if (ONE_TEST && scale >= 0x1p-126f && scale <= 3.40282347e38f) {
    float t[kVec];
    bool near_tie = false;
#pragma unroll
    for (int e = 0; e < kVec; ++e) {
      const float y = __fmul_rn(x[e], rcp);
      t[e] = __fadd_rn(y, 12582912.0f);
      const float d = __fsub_rn(y, __fsub_rn(t[e], 12582912.0f));  // exact: |d| <= 0.5
      near_tie |= !(fabsf(d) < 0.4999f);
    }
    if (!near_tie) {
#pragma unroll
      for (int e = 0; e < kVec; ++e) q[e] = __float_as_int(t[e]) - 0x4B400000;
      return;
    }
#pragma unroll
    for (int e = 0; e < kVec; ++e) q[e] = quant_rcp(x[e], scale, rcp);
  } else if (scale == 0.0f) {
#pragma unroll
    for (int e = 0; e < kVec; ++e) q[e] = 0;
  } else if (isfinite(rcp)) {
#pragma unroll
    for (int e = 0; e < kVec; ++e) q[e] = quant_rcp(x[e], scale, rcp);
  } else {
#pragma unroll
    for (int e = 0; e < kVec; ++e) q[e] = quant_div(x[e], scale);
  }
}

// |x| as its bit pattern.  These patterns order like the magnitudes, with
// every NaN above +inf, so an unsigned maximum over them propagates a NaN
// (fmaxf would drop it): a block holding a NaN gets a NaN scale, one holding
// an infinity an infinite scale, and either dequantizes to non-finite values.
__device__ __forceinline__ uint32_t abs_bits(float x) { return __float_as_uint(x) & 0x7fffffffu; }

// Warp maximum of magnitudes given as abs_bits patterns, as a float.
__device__ __forceinline__ float warp_absmax(uint32_t a) {
  return __uint_as_float(__reduce_max_sync(0xffffffffu, a));
}

__device__ __forceinline__ uint2 pack_i8x8(const int (&q)[kVec]) {
  uint32_t lo = 0, hi = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    lo |= (static_cast<uint32_t>(q[k]) & 0xffu) << (8 * k);
    hi |= (static_cast<uint32_t>(q[k + 4]) & 0xffu) << (8 * k);
  }
  return make_uint2(lo, hi);
}

__device__ __forceinline__ uint2 ld8(const void* ptr) {
  uint2 x;
  asm volatile("ld.global.cs.v2.u32 {%0, %1}, [%2];" : "=r"(x.x), "=r"(x.y) : "l"(ptr));
  return x;
}
__device__ __forceinline__ void st8(void* ptr, uint2 x) {
  asm volatile("st.global.cs.v2.u32 [%0], {%1, %2};" ::"l"(ptr), "r"(x.x), "r"(x.y) : "memory");
}

// Ring-order sum of the dequantized gradients of the 8 elements at i0, all
// owned by r.  PT > 0: P = PT known at compile time (PT <= 8, or a multiple
// of 8 taken in exact groups of 8); PT = 0: any P, the last group partial.
template <int PT>
__device__ __forceinline__ void zpp_ring_vec(const ZppParams& p, int P, int r, int64_t i0,
                                             int64_t blk, float (&acc)[kVec]) {
  int q = ring_next(r, P);
  // The generic kernel (PT = 0) loads 4 ranks at a time: with 8 its predicated
  // loads spilled 644 bytes and it ran 0.08 of the copy ceiling slower (P = 10..20).
  constexpr int U = PT > 0 && PT < 8 ? PT : (PT == 0 ? 4 : 8);
  constexpr bool EXACT = PT > 0;
#pragma unroll 1
  for (int base = 0; base < P; base += U) {
    uint2 d[U];
    float sc[U];
    const int cnt = P - base < U ? P - base : U;
#pragma unroll
    for (int k = 0; k < U; ++k) {
      if (EXACT || k < cnt) {
        d[k] = ld8(p.g[q] + (i0 - p.off));
        sc[k] = p.gs[q][blk];
        q = ring_next(q, P);
      }
    }
#pragma unroll
    for (int k = 0; k < U; ++k) {
      if (EXACT || k < cnt) {
        float v8[kVec];  // the int8 codes, converted exactly
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          v8[e] = __int2float_rn(static_cast<int8_t>((d[k].x >> (8 * e)) & 0xffu));
          v8[e + 4] = __int2float_rn(static_cast<int8_t>((d[k].y >> (8 * e)) & 0xffu));
        }
#pragma unroll
        for (int e = 0; e < kVec; ++e) {
          const float x = __fmul_rn(v8[e], sc[k]);
          acc[e] = (base == 0 && k == 0) ? x : __fadd_rn(acc[e], x);
        }
      }
    }
  }
}

// Resident blocks the register allocation must allow (measured best on
// GB300): 8 (64 registers) for P <= 8 and the generic kernel, 6 (80
// registers) for the exact multiples of 8 above 8, which keep two groups of
// eight ranks' loads in flight.
#ifndef ZDP_ZPP_MIN_BLOCKS
#define ZDP_ZPP_MIN_BLOCKS 8
#endif
#ifndef ZDP_ZPP_MIN_BLOCKS_WIDE
#define ZDP_ZPP_MIN_BLOCKS_WIDE 6
#endif

// The sum of squares accumulated straight in fp64: the square of an fp32
// value has at most 48 significant bits and an exponent within fp64's range,
// so it is exact in fp64 and each step rounds once (no worse than the
// compensated fp32 SumSq).  It costs one fp64 fma per element where SumSq
// spends about ten fp32 instructions.  GB300's fp64 rate is low, so which
// form is faster depends on what else the kernel keeps busy; see
// zpp_f64_sumsq.
struct SumSqF64 {
  double total = 0.0;
  __device__ __forceinline__ void add(float g) {
    const double d = static_cast<double>(g);
    total = __fma_rn(d, d, total);
  }
};

__device__ __forceinline__ void account(const float (&g)[kVec], bool sq, bool& bad,
                                        SumSqF64& ss) {
#pragma unroll
  for (int k = 0; k < kVec; ++k) bad |= non_finite(g[k]);
  if (sq) {
#pragma unroll
    for (int k = 0; k < kVec; ++k) ss.add(g[k]);
  }
}

__device__ __forceinline__ void account1(float g, bool sq, bool& bad, SumSqF64& ss) {
  bad |= non_finite(g);
  if (sq) ss.add(g);
}

__device__ __forceinline__ void publish_to(int32_t* flag, double* sumsq, bool bad,
                                           SumSqF64& acc) {
  SumSq whole;  // carries the fp64 total through the block reduction
  whole.total = acc.total;
  publish_to(flag, sumsq, bad, whole);
}

// MT: the moment type when fixed at compile time (the bf16-moment kernels), or
// -1 to follow p.mt; MINB: the resident blocks per SM the register allocation
// must allow.
template <int PT, bool F64SQ, int MT = -1,
          int MINB = (PT > 8 ? ZDP_ZPP_MIN_BLOCKS_WIDE : ZDP_ZPP_MIN_BLOCKS)>
__global__ void __launch_bounds__(kThreads, MINB) k_zpp(const __grid_constant__ ZppParams p) {
  const int P = PT > 0 ? PT : p.P;
  const int mt = MT >= 0 ? MT : p.mt;
  const bool sq = p.sumsq != nullptr;
  const int lane = threadIdx.x & 31;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * kThreads) >> 5;
  bool bad = false;
  typename std::conditional<F64SQ, SumSqF64, SumSq>::type ss;
  const int64_t b0 = p.lo / kQB, b1 = (p.hi + kQB - 1) / kQB;  // p.lo is block aligned
  for (int64_t b = b0 + warp; b < b1; b += nwarps) {               // warp-uniform
    const int64_t i0 = b * kQB + lane * kVec;
    const int64_t gb = b - p.off / kQB;                             // gradient scale index
    int cnt = static_cast<int>(p.hi - i0);
    cnt = cnt < 0 ? 0 : (cnt > kVec ? kVec : cnt);
    float pv[kVec];  // the new bf16 parameters as fp32
#pragma unroll
    for (int e = 0; e < kVec; ++e) pv[e] = 0.0f;
    if (cnt > 0) {
      const int r = zpp_owner(i0, p);
      float g[kVec];
      const bool full = cnt == kVec && i0 + kVec <= static_cast<int64_t>(r + 1) * p.S;
      if (full) {
        zpp_ring_vec<PT>(p, P, r, i0, gb, g);
      } else {
#pragma unroll
        for (int e = 0; e < kVec; ++e) {
          if (e < cnt) {
            const int64_t i = i0 + e;
            int q = ring_next(zpp_owner(i, p), P);
            float acc = dequant(p.g[q][i - p.off], p.gs[q][gb]);
            for (int k = 1; k < P; ++k) {
              q = ring_next(q, P);
              acc = __fadd_rn(acc, dequant(p.g[q][i - p.off], p.gs[q][gb]));
            }
            g[e] = acc;
          }
        }
      }
      if (full) {
        float w[kVec], m[kVec], v[kVec];
        ld_f8(p.w + i0, w);
        ld_moments8(p.m, p.v, mt, i0, m, v);
#pragma unroll
        for (int e = 0; e < kVec; ++e) {
          g[e] = __fmul_rn(g[e], p.scale);
          adamw(w[e], m[e], v[e], g[e], p.ad);
        }
        vec_set<ZDP_BF16>(pv, pack_bf16x8(w));  // the bf16 parameters, widened
        account(g, sq, bad, ss);
        st_f8(p.w + i0, w);
        st_moments8(p.m, p.v, mt, i0, m, v);
      } else {
#pragma unroll
        for (int e = 0; e < kVec; ++e) {
          if (e < cnt) {
            const int64_t i = i0 + e;
            const float ge = __fmul_rn(g[e], p.scale);
            account1(ge, sq, bad, ss);
            float w = p.w[i], m = ld_moment(p.m, i, mt), v = ld_moment(p.v, i, mt);
            adamw(w, m, v, ge, p.ad);
            p.w[i] = w;
            st_moment(p.m, i, mt, m);
            st_moment(p.v, i, mt, v);
            pv[e] = widen1<ZDP_BF16>(to_bf16(w));
          }
        }
      }
    }
    uint32_t abits = 0;
#pragma unroll
    for (int e = 0; e < kVec; ++e) abits = max(abits, abs_bits(pv[e]));
    const float sc = __fdiv_rn(warp_absmax(abits), 127.0f);
    int qv[kVec];
    quant8<(PT <= 8)>(pv, sc, qv);
    if (cnt == kVec) {
      const uint2 packed = pack_i8x8(qv);
      for (int q = 0; q < P; ++q) st8(p.rq[q] + i0, packed);
    } else {
      for (int q = 0; q < P; ++q) {
#pragma unroll
        for (int e = 0; e < kVec; ++e)
          if (e < cnt) p.rq[q][i0 + e] = static_cast<int8_t>(qv[e]);
      }
    }
    if (lane == 0)
      for (int q = 0; q < P; ++q) p.rs[q][b] = sc;
  }
  publish_to(p.flag, p.sumsq, bad, ss);
}

// Block quantization of a bf16 / fp16 / fp32 array (the producer's side).
template <int XT>  // 0 bf16, 1 fp16, 2 fp32
__global__ void __launch_bounds__(kThreads) k_quantize(const void* x, int64_t n, int8_t* q,
                                                       float* scales) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * kThreads) >> 5;
  for (int64_t b = warp; b * kQB < n; b += nwarps) {
    const int64_t i0 = b * kQB + lane * kVec;
    float v[kVec];
    uint32_t abits = 0;
#pragma unroll
    for (int e = 0; e < kVec; ++e) {
      const int64_t i = i0 + e;
      float xv = 0.0f;
      if (i < n) {
        if constexpr (XT == 0) {
          xv = widen1<ZDP_BF16>(static_cast<const uint16_t*>(x)[i]);
        } else if constexpr (XT == 1) {
          xv = widen1<ZDP_FP16>(static_cast<const uint16_t*>(x)[i]);
        } else {
          xv = static_cast<const float*>(x)[i];
        }
      }
      v[e] = xv;
      abits = max(abits, abs_bits(xv));
    }
    const float sc = __fdiv_rn(warp_absmax(abits), 127.0f);
    int qv[kVec];
    quant8(v, sc, qv);
#pragma unroll
    for (int e = 0; e < kVec; ++e)
      if (i0 + e < n) q[i0 + e] = static_cast<int8_t>(qv[e]);
    if (lane == 0) scales[b] = sc;
  }
}

// Dequantization back to bf16 (the receiver's side): bf16(q * scale).
__global__ void __launch_bounds__(kThreads) k_dequantize(const int8_t* q, const float* scales,
                                                         int64_t n, uint16_t* out) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < n; i += stride)
    out[i] = to_bf16(dequant(q[i], scales[i / kQB]));
}

#ifndef ZDP_CAP_ZPP
#define ZDP_CAP_ZPP 8
#endif

// One wave of at most `cap` resident blocks per SM, capped by the work (one
// warp per 256-element block).
int grid_warps(const void* kernel, int64_t warps_needed, int num_sms, int cap) {
  const int64_t blocks = (warps_needed * 32 + kThreads - 1) / kThreads;
  const int res = resident_blocks(kernel);
  const int64_t full = static_cast<int64_t>(num_sms) * (res < cap ? res : cap);
  return static_cast<int>(std::max<int64_t>(1, std::min(blocks, full)));
}

template <int PT>
const void* zpp_kernel(bool f64) {
  return f64 ? reinterpret_cast<const void*>(&k_zpp<PT, true>)
             : reinterpret_cast<const void*>(&k_zpp<PT, false>);
}

// Whether the step with the sum of squares accumulates it in fp64
// (SumSqF64) rather than compensated fp32 (SumSq), for P ranks and the
// moment type: the faster form measured on GB300 with the sum of squares
// asked for (time of the compensated form / time of the fp64 form, fp32
// moments and bf16 moments): P = 2: 1.02, 1.06; 4: 1.07, 1.08; 5: 1.06,
// 1.10; 8: 0.98, 1.12; 12 (the generic kernel): 1.09, 1.05; 16: 0.98, 0.96
// (the wide template spills 76 bytes with the fp64 form; P = 32 shares
// it); 64: 1.03, 0.99.  ZDP_ZPP_F64SQ = 0 or 1 forces one form (for tuning).
#ifndef ZDP_ZPP_F64SQ
#define ZDP_ZPP_F64SQ -1
#endif
bool zpp_f64_sumsq(int P, int mt) {
  if (ZDP_ZPP_F64SQ >= 0) return ZDP_ZPP_F64SQ != 0;
  const bool f32 = mt == ZDP_MOMENTS_F32;
  if (P == 16 || P == 32) return false;
  if (P == 8) return !f32;
  if (P == 64) return f32;
  return true;
}

// The kernels with the moment type fixed at compile time, for the P, moment
// type (and sum-of-squares form) where they measured faster on GB300 than the
// kernel that reads the moment type at run time; nullptr elsewhere.  The
// resident blocks per SM asked of the register allocator are the measured
// best.  Fraction of the copy ceiling, flat n = 2^28, run-time -> fixed
// moment type (blocks per SM):
//   bf16 moments: P = 1: 0.594 -> 0.603 (7); 2: 0.570 -> 0.593 (6); 3: 0.647
//   -> 0.684 (8); 4: 0.685 -> 0.754 (8); 5: 0.716 -> 0.753 (8); 6: 0.745 ->
//   0.804 (6); 7: 0.790 -> 0.846 (8); 8: 0.795 -> 0.852 (7); 12, the generic
//   kernel: 0.710 -> 0.733 (8); 16: 0.719 -> 0.725 (6); 64: 0.808 -> 0.816
//   (6); P = 32 keeps the run-time kernel (0.806 against 0.790).
//   fp32 moments: P = 1: 0.846 -> 0.862 (7); 2: 0.775 -> 0.799 (6); 3: 0.834
//   -> 0.885 (8); 4: 0.895 -> 0.910 (8); 5: 0.908 -> 0.918 (6); 6: 0.918 ->
//   0.943 (8); P = 7, 8 and above keep the run-time kernel (P = 8: 0.873
//   against 0.864 at 8 blocks).
// With the sum of squares in the other form than the one measured, the
// run-time kernel serves.
const void* zpp_kernel_fixed(int P, int mt, bool f64) {
  constexpr int B = ZDP_MOMENTS_BF16, F = ZDP_MOMENTS_F32;
  auto k = [](auto kernel) { return reinterpret_cast<const void*>(kernel); };
  if (f64 != zpp_f64_sumsq(P, mt)) return nullptr;
  if (mt == F) {
    switch (P) {
      case 1: return k(&k_zpp<1, true, F, 7>);
      case 2: return k(&k_zpp<2, true, F, 6>);
      case 3: return k(&k_zpp<3, true, F, 8>);
      case 4: return k(&k_zpp<4, true, F, 8>);
      case 5: return k(&k_zpp<5, true, F, 6>);
      case 6: return k(&k_zpp<6, true, F, 8>);
      default: return nullptr;
    }
  }
  switch (P) {
    case 1: return k(&k_zpp<1, true, B, 7>);
    case 2: return k(&k_zpp<2, true, B, 6>);
    case 3: return k(&k_zpp<3, true, B, 8>);
    case 4: return k(&k_zpp<4, true, B, 8>);
    case 5: return k(&k_zpp<5, true, B, 8>);
    case 6: return k(&k_zpp<6, true, B, 6>);
    case 7: return k(&k_zpp<7, true, B, 8>);
    case 8: return k(&k_zpp<8, true, B, 7>);
    case 16: return k(&k_zpp<16, false, B, 6>);
    case 32: return nullptr;
    case 64: return k(&k_zpp<64, false, B, 6>);
    default: return k(&k_zpp<0, true, B, 8>);
  }
}

}  // namespace

cudaError_t launch_zpp(const zdp_zpp_args* a, const AdamK& ad, int num_sms, cudaStream_t s) {
  ZppParams p;
  std::memset(&p, 0, sizeof p);
  const int P = a->P;
  for (int q = 0; q < P; ++q) {
    p.g[q] = a->grads[q];
    p.gs[q] = a->grad_scales[q];
    p.rq[q] = a->replicas[q];
    p.rs[q] = a->replica_scales[q];
  }
  p.w = a->master;
  p.m = a->m;
  p.v = a->v;
  p.mt = a->moment_dtype;
  p.n = a->n;
  p.S = (a->n + P - 1) / P;
  p.inv_s = 1.0f / static_cast<float>(p.S);
  p.off = a->off;
  p.lo = a->off;
  p.hi = a->off + a->len;
  p.P = P;
  p.scale = a->scale;
  p.ad = ad;
  p.flag = a->d_overflow;
  p.sumsq = a->d_sumsq;
  const int64_t blocks = (a->len + kQB - 1) / kQB;
  if (blocks == 0) return cudaSuccess;
  const bool f64 = p.sumsq != nullptr && zpp_f64_sumsq(P, p.mt);
  const void* fn = zpp_kernel_fixed(P, p.mt, f64);
  if (!fn) switch (P) {
    case 1: fn = zpp_kernel<1>(f64); break;
    case 2: fn = zpp_kernel<2>(f64); break;
    case 3: fn = zpp_kernel<3>(f64); break;
    case 4: fn = zpp_kernel<4>(f64); break;
    case 5: fn = zpp_kernel<5>(f64); break;
    case 6: fn = zpp_kernel<6>(f64); break;
    case 7: fn = zpp_kernel<7>(f64); break;
    case 8: fn = zpp_kernel<8>(f64); break;
    case 16: fn = zpp_kernel<16>(f64); break;
    case 32: fn = zpp_kernel<32>(f64); break;
    case 64: fn = zpp_kernel<64>(f64); break;
    default: fn = zpp_kernel<0>(f64); break;
  }
  void* args[] = {&p};
  // 6 blocks per SM at P = 2 (0.90 of the copy ceiling against 0.88 with 8);
  // every other P measured best at the register-limited 8 (or 6 above P = 8).
  const int cap = P == 2 ? 6 : ZDP_CAP_ZPP;
  return cudaLaunchKernel(fn, dim3(grid_warps(fn, blocks, num_sms, cap)), dim3(kThreads), args,
                          0, s);
}

cudaError_t launch_quantize(const void* x, int xdt, int64_t n, int8_t* q, float* scales,
                            int num_sms, cudaStream_t s) {
  const int64_t blocks = (n + kQB - 1) / kQB;
  const void* fn = xdt == 0   ? reinterpret_cast<const void*>(&k_quantize<0>)
                   : xdt == 1 ? reinterpret_cast<const void*>(&k_quantize<1>)
                              : reinterpret_cast<const void*>(&k_quantize<2>);
  const int grid = grid_warps(fn, blocks, num_sms, 8);
  if (xdt == 0) {
    k_quantize<0><<<grid, kThreads, 0, s>>>(x, n, q, scales);
  } else if (xdt == 1) {
    k_quantize<1><<<grid, kThreads, 0, s>>>(x, n, q, scales);
  } else {
    k_quantize<2><<<grid, kThreads, 0, s>>>(x, n, q, scales);
  }
  return cudaGetLastError();
}

cudaError_t launch_dequantize(const int8_t* q, const float* scales, int64_t n, uint16_t* out,
                              int num_sms, cudaStream_t s) {
  const int64_t need = (n + kThreads - 1) / kThreads;
  const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(need, num_sms * 8)));
  k_dequantize<<<grid, kThreads, 0, s>>>(q, scales, n, out);
  return cudaGetLastError();
}

}  // namespace zdp
