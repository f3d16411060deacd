// zdp_ring.cu -- zdp_step_ring: the ZeRO step run as the literal ring
// schedule, one launch per ring step, for comparison with the fused pass.
//
// Ring schedule (Fudan MLSys ch. 9, 9.3.6; CS336 Lecture 7 notes, 4.2), in
// the owner labelling: at reduce-scatter step s (s = 0 .. P-2) rank i sends
// its partial sum of chunk c = (i - s - 1) mod P to rank i+1, which adds its
// own chunk c; after P-1 steps rank i holds the complete chunk i.  Here the
// P ranks' messages are P fp32 chunk buffers in one HBM, double-buffered
// (step s reads the messages of step s-1 and writes its own), so the
// reduce-scatter is P-1 launches over P*S elements each.  The owner's last
// add is fused with the scale, the AdamW update and the bf16 write of the
// owner's own replica chunk; the all-gather is then P-1 launches, step s
// copying chunk (i - s) mod P of replica i into replica i+1.
//
// Every fp32 add happens in the same order as the fused kernel's (ring order
// starting after the owner), so the results are bit-identical to zdp_step.
// Elements at or beyond n (the padding of the last chunk) read as zero.
// Grids are 2-D: blockIdx.y is the rank, x walks the S elements of a chunk.
#include <algorithm>
#include <cstring>

#include "zdp_kernels.cuh"

namespace zdp {
namespace {

struct RingParams {
  const void* g[ZDP_MAX_P];  // rank q's gradient of global element i: g[q][i]
  uint16_t* rep[ZDP_MAX_P];
  float* w;
  float* m;
  float* v;
  const float* msg_in;  // P * S: message of rank q at msg_in[q*S + e]
  float* msg_out;
  int64_t n, S;
  int P, step;
  float scale;
  AdamK ad;
  int32_t* flag;
  double* sumsq;
};

template <int GT>
__device__ __forceinline__ float grad_at(const RingParams& p, int q, int64_t i) {
  return i < p.n ? widen1<GT>(__ldcs(static_cast<const uint16_t*>(p.g[q]) + i)) : 0.0f;
}

__device__ __forceinline__ int prev_rank(int i, int P) { return i == 0 ? P - 1 : i - 1; }

// Reduce-scatter step s for rank i = blockIdx.y: its message for chunk
// c = (i - s - 1) mod P is the previous rank's message plus G_i's chunk c
// (at s = 0 just G_i's chunk c: the ring's first operand).
// VEC: S % 8 == 0 and 16-byte aligned buffers; whole 8-vectors inside [0, n).
template <int GT, bool VEC>
__global__ void __launch_bounds__(kThreads) k_ring_rs(const __grid_constant__ RingParams p) {
  const int i = blockIdx.y;
  const int c = ((i - p.step - 1) % p.P + p.P) % p.P;
  const int64_t base = static_cast<int64_t>(c) * p.S;
  const float* in = p.msg_in + static_cast<int64_t>(prev_rank(i, p.P)) * p.S;
  float* out = p.msg_out + static_cast<int64_t>(i) * p.S;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  if constexpr (VEC) {
    for (int64_t e0 = tid * kVec; e0 < p.S; e0 += stride * kVec) {
      float acc[kVec];
      if (base + e0 + kVec <= p.n) {
        const uint4 d = ld16(static_cast<const uint16_t*>(p.g[i]) + base + e0);
        vec_set<GT>(acc, d);
      } else {
#pragma unroll
        for (int k = 0; k < kVec; ++k) acc[k] = grad_at<GT>(p, i, base + e0 + k);
      }
      if (p.step > 0) {
        float prev[kVec];
        ld_f8(in + e0, prev);
#pragma unroll
        for (int k = 0; k < kVec; ++k) acc[k] = __fadd_rn(prev[k], acc[k]);
      }
      st_f8(out + e0, acc);
    }
  } else {
    for (int64_t e = tid; e < p.S; e += stride) {
      float x = grad_at<GT>(p, i, base + e);
      if (p.step > 0) x = __fadd_rn(__ldcs(in + e), x);
      __stcs(out + e, x);
    }
  }
}

// Rank r = blockIdx.y finishes its own chunk from rank r-1's last message,
// then scale, flag, AdamW and the owner's replica chunk.
template <int GT, bool VEC>
__global__ void __launch_bounds__(kThreads) k_ring_final(const __grid_constant__ RingParams p) {
  const int r = blockIdx.y;
  const int64_t base = static_cast<int64_t>(r) * p.S;
  const float* in = p.msg_in + static_cast<int64_t>(prev_rank(r, p.P)) * p.S;
  const bool sq = p.sumsq != nullptr;
  bool bad = false;
  SumSq ss;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  if constexpr (VEC) {
    for (int64_t e0 = tid * kVec; e0 < p.S; e0 += stride * kVec) {
      const int64_t i0 = base + e0;
      if (i0 >= p.n) break;
      if (i0 + kVec <= p.n) {
        float g[kVec], w[kVec], m[kVec], v[kVec];
        vec_set<GT>(g, ld16(static_cast<const uint16_t*>(p.g[r]) + i0));
        if (p.P > 1) {
          float prev[kVec];
          ld_f8(in + e0, prev);
#pragma unroll
          for (int k = 0; k < kVec; ++k) g[k] = __fadd_rn(prev[k], g[k]);
        }
#pragma unroll
        for (int k = 0; k < kVec; ++k) g[k] = __fmul_rn(g[k], p.scale);
        account(g, sq, bad, ss);
        ld_f8(p.w + i0, w);
        ld_f8(p.m + i0, m);
        ld_f8(p.v + i0, v);
#pragma unroll
        for (int k = 0; k < kVec; ++k) adamw(w[k], m[k], v[k], g[k], p.ad);
        st_f8(p.w + i0, w);
        st_f8(p.m + i0, m);
        st_f8(p.v + i0, v);
        st16(p.rep[r] + i0, pack_bf16x8(w));
        continue;
      }
      for (int k = 0; k < kVec && i0 + k < p.n; ++k) {
        float g = grad_at<GT>(p, r, i0 + k);
        if (p.P > 1) g = __fadd_rn(in[e0 + k], g);
        g = __fmul_rn(g, p.scale);
        account1(g, sq, bad, ss);
        float w = p.w[i0 + k], m = p.m[i0 + k], v = p.v[i0 + k];
        adamw(w, m, v, g, p.ad);
        p.w[i0 + k] = w;
        p.m[i0 + k] = m;
        p.v[i0 + k] = v;
        p.rep[r][i0 + k] = to_bf16(w);
      }
    }
  } else {
    for (int64_t e = tid; e < p.S && base + e < p.n; e += stride) {
      const int64_t i = base + e;
      float g = grad_at<GT>(p, r, i);
      if (p.P > 1) g = __fadd_rn(__ldcs(in + e), g);
      g = __fmul_rn(g, p.scale);
      account1(g, sq, bad, ss);
      float w = p.w[i], m = p.m[i], v = p.v[i];
      adamw(w, m, v, g, p.ad);
      p.w[i] = w;
      p.m[i] = m;
      p.v[i] = v;
      p.rep[r][i] = to_bf16(w);
    }
  }
  publish_to(p.flag, p.sumsq, bad, ss);
}

// All-gather step s: replica i+1 receives chunk (i - s) mod P of replica i
// (i = blockIdx.y).
template <bool VEC>
__global__ void __launch_bounds__(kThreads) k_ring_ag(const __grid_constant__ RingParams p) {
  const int i = blockIdx.y;
  const int c = ((i - p.step) % p.P + p.P) % p.P;
  const int64_t base = static_cast<int64_t>(c) * p.S;
  const uint16_t* src = p.rep[i];
  uint16_t* dst = p.rep[i + 1 == p.P ? 0 : i + 1];
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  if constexpr (VEC) {
    for (int64_t e0 = tid * kVec; e0 < p.S; e0 += stride * kVec) {
      const int64_t i0 = base + e0;
      if (i0 + kVec <= p.n) {
        st16(dst + i0, ld16(src + i0));
      } else {
        for (int k = 0; k < kVec && i0 + k < p.n; ++k) dst[i0 + k] = src[i0 + k];
      }
    }
  } else {
    for (int64_t e = tid; e < p.S && base + e < p.n; e += stride) dst[base + e] = src[base + e];
  }
}

dim3 grid_2d(int64_t S, int P, int num_sms, bool vec) {
  const int64_t work = vec ? (S + kVec - 1) / kVec : S;
  const int64_t need = (work + kThreads - 1) / kThreads;
  // about 4 resident blocks of 128 threads per SM over all P ranks
  const int64_t per_rank = std::max<int64_t>(1, static_cast<int64_t>(num_sms) * 4 / P);
  return dim3(static_cast<unsigned>(std::max<int64_t>(1, std::min(need, per_rank))),
              static_cast<unsigned>(P));
}

template <int GT, bool VEC>
cudaError_t run(RingParams& p, float* const buf[2], int num_sms, cudaStream_t s) {
  void* args[] = {&p};
  const dim3 grid = grid_2d(p.S, p.P, num_sms, VEC);
  cudaError_t e = cudaSuccess;
  for (int step = 0; step + 1 < p.P; ++step) {  // P-1 reduce-scatter launches
    p.step = step;
    p.msg_in = buf[(step & 1) ^ 1];
    p.msg_out = buf[step & 1];
    e = cudaLaunchKernel(reinterpret_cast<const void*>(&k_ring_rs<GT, VEC>), grid,
                         dim3(kThreads), args, 0, s);
    if (e != cudaSuccess) return e;
  }
  p.msg_in = buf[(p.P - 2) & 1];  // the last reduce-scatter step's messages (unused at P = 1)
  e = cudaLaunchKernel(reinterpret_cast<const void*>(&k_ring_final<GT, VEC>), grid,
                       dim3(kThreads), args, 0, s);
  if (e != cudaSuccess) return e;
  for (int step = 0; step + 1 < p.P; ++step) {  // P-1 all-gather launches
    p.step = step;
    e = cudaLaunchKernel(reinterpret_cast<const void*>(&k_ring_ag<VEC>), grid, dim3(kThreads),
                         args, 0, s);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_ring(const zdp_step_args* a, const AdamK& ad, float* ws, bool vec,
                        int num_sms, cudaStream_t s) {
  RingParams p;
  std::memset(&p, 0, sizeof p);
  const int P = a->P;
  for (int q = 0; q < P; ++q) {
    p.g[q] = a->grads[q];
    p.rep[q] = a->replicas[q];
  }
  p.w = a->master;
  p.m = static_cast<float*>(a->m);  // the ring mode takes fp32 moments only
  p.v = static_cast<float*>(a->v);
  p.n = a->n;
  p.S = (a->n + P - 1) / P;
  p.P = P;
  p.scale = a->scale;
  p.ad = ad;
  p.flag = a->d_overflow;
  p.sumsq = a->d_sumsq;
  float* const buf[2] = {ws, ws + static_cast<int64_t>(P) * p.S};
  vec = vec && p.S % kVec == 0;
  if (a->gdt == ZDP_BF16) {
    return vec ? run<ZDP_BF16, true>(p, buf, num_sms, s) : run<ZDP_BF16, false>(p, buf, num_sms, s);
  }
  return vec ? run<ZDP_FP16, true>(p, buf, num_sms, s) : run<ZDP_FP16, false>(p, buf, num_sms, s);
}

}  // namespace zdp
