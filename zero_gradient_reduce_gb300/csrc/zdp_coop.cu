// zdp_coop.cu -- the overflow-checked step in one cooperative launch, for
// ranges whose reduced gradients fit in the registers of one resident wave.
//
// The checked step may write nothing unless every reduced gradient of the
// range is finite, so the update must wait for a decision that depends on the
// whole range.  The two-pass form writes the reduced gradients to a workspace
// and reads them back (8 more bytes per parameter, two launches and a memset).
// Here every thread keeps the reduced gradients of its vectors in registers,
// the blocks OR their flags into a device word and meet at a grid barrier,
// and after the barrier every block reads the word and either updates its
// vectors or writes nothing.  The launch is cooperative, so every block is
// resident and the barrier completes.  The wait is still bounded: after
// `timeout_ns` a block gives up, writes nothing and raises ZDP_FLAG_TIMEOUT
// in the caller's flag word.
#include <algorithm>
#include <cstdlib>

#include "zdp_kernels.cuh"

namespace zdp {
namespace {

constexpr int kCoopV = 2;  // 8-element vectors per thread held in registers

struct CoopParams {
  KParams k;
  int32_t* ws_flag;      // device word: OR of every block's overflow, zeroed before launch
  uint32_t* arrived;     // device word: blocks that reached the barrier, zeroed before launch
  uint32_t expected;     // arrivals the barrier waits for (gridDim.x)
  uint64_t timeout_ns;   // how long a block waits at the barrier
};

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ int32_t ld_acquire(const int32_t* p) {
  int32_t v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Vector vi of this thread is "full" when its 8 elements lie in the range and
// in one shard; otherwise its elements are handled one by one.
__device__ __forceinline__ bool full_vec(const KParams& p, int64_t i0, int r) {
  return i0 >= p.lo && i0 + kVec <= p.hi && i0 + kVec <= static_cast<int64_t>(r + 1) * p.S;
}

template <int PT, int GT>
__global__ void __launch_bounds__(kThreads) k_step_coop(const __grid_constant__ CoopParams c) {
  const KParams& p = c.k;
  constexpr int P = PT;
  const bool sq = p.sumsq != nullptr;
  bool bad = false;
  SumSq ss;
  const int64_t T = static_cast<int64_t>(gridDim.x) * kThreads;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  const int64_t vlo = p.lo / kVec, vhi = (p.hi + kVec - 1) / kVec;

  // Phase 1: the reduced gradients of this thread's vectors, kept in registers.
  float g[kCoopV][kVec];
#pragma unroll
  for (int j = 0; j < kCoopV; ++j) {
    const int64_t vi = vlo + tid + j * T;
    if (vi >= vhi) continue;
    const int64_t i0 = vi * kVec;
    const int r = owner_of(i0, p, P);
    if (full_vec(p, i0, r)) {
      ring_sum_vec<PT, true, GT>(p, P, r, i0, g[j]);
#pragma unroll
      for (int k = 0; k < kVec; ++k) g[j][k] = __fmul_rn(g[j][k], p.scale);
      account(g[j], sq, bad, ss);
    } else {
#pragma unroll
      for (int k = 0; k < kVec; ++k) {
        const int64_t i = i0 + k;
        if (i >= p.lo && i < p.hi) {
          g[j][k] = __fmul_rn(ring_sum_elem<GT>(p, P, owner_of(i, p, P), i), p.scale);
          account1(g[j][k], sq, bad, ss);
        }
      }
    }
  }
  publish_to(c.ws_flag, p.sumsq, bad, ss);

  // Grid barrier: thread 0 of each block arrives after its flag is visible
  // and waits, bounded, for every block.
  __shared__ int s_go;
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(c.arrived, 1u);
    const uint64_t t0 = globaltimer_ns();
    bool met = false;
    for (uint32_t polls = 0;; ++polls) {
      if (ld_acquire(c.arrived) >= c.expected) {
        met = true;
        break;
      }
      if (globaltimer_ns() - t0 > c.timeout_ns) break;
      if (polls >= 64) __nanosleep(64);  // spin first: the last arrival is usually close
    }
    const bool clean = met && ld_acquire(c.ws_flag) == 0;
    if (p.flag) {
      if (!met) atomicOr(p.flag, ZDP_FLAG_TIMEOUT);
      if (met && !clean && blockIdx.x == 0) atomicOr(p.flag, ZDP_FLAG_OVERFLOW);
    }
    s_go = clean ? 1 : 0;
  }
  __syncthreads();
  if (!s_go) return;

  // Phase 2: AdamW, the bf16 cast and every replica, from the registers.
#pragma unroll
  for (int j = 0; j < kCoopV; ++j) {
    const int64_t vi = vlo + tid + j * T;
    if (vi >= vhi) continue;
    const int64_t i0 = vi * kVec;
    const int r = owner_of(i0, p, P);
    if (full_vec(p, i0, r)) {
      float w[kVec], m[kVec], v[kVec];
      ld_f8(p.w + i0, w);
      ld_moments8(p.m, p.v, p.mt, i0, m, v);
#pragma unroll
      for (int k = 0; k < kVec; ++k) adamw(w[k], m[k], v[k], g[j][k], p.ad);
      st_f8(p.w + i0, w);
      st_moments8(p.m, p.v, p.mt, i0, m, v);
      const uint4 b = pack_bf16x8(w);
#pragma unroll 8
      for (int q = 0; q < P; ++q) st16(p.rep[q] + i0, b);
    } else {
#pragma unroll
      for (int k = 0; k < kVec; ++k) {
        const int64_t i = i0 + k;
        if (i >= p.lo && i < p.hi) {
          float w = p.w[i], m = ld_moment(p.m, i, p.mt), v = ld_moment(p.v, i, p.mt);
          adamw(w, m, v, g[j][k], p.ad);
          p.w[i] = w;
          st_moment(p.m, i, p.mt, m);
          st_moment(p.v, i, p.mt, v);
          const uint16_t b = to_bf16(w);
          for (int q = 0; q < P; ++q) p.rep[q][i] = b;
        }
      }
    }
  }
}

template <int GT>
const void* coop_kernel(int P) {
  switch (P) {
    case 1: return reinterpret_cast<const void*>(&k_step_coop<1, GT>);
    case 2: return reinterpret_cast<const void*>(&k_step_coop<2, GT>);
    case 3: return reinterpret_cast<const void*>(&k_step_coop<3, GT>);
    case 4: return reinterpret_cast<const void*>(&k_step_coop<4, GT>);
    case 5: return reinterpret_cast<const void*>(&k_step_coop<5, GT>);
    case 6: return reinterpret_cast<const void*>(&k_step_coop<6, GT>);
    case 7: return reinterpret_cast<const void*>(&k_step_coop<7, GT>);
    case 8: return reinterpret_cast<const void*>(&k_step_coop<8, GT>);
    case 16: return reinterpret_cast<const void*>(&k_step_coop<16, GT>);
    case 32: return reinterpret_cast<const void*>(&k_step_coop<32, GT>);
    case 64: return reinterpret_cast<const void*>(&k_step_coop<64, GT>);
    default: return nullptr;
  }
}

int64_t env_int(const char* name, int64_t fallback) {
  const char* s = std::getenv(name);
  if (!s || !*s) return fallback;
  char* end = nullptr;
  const long long v = std::strtoll(s, &end, 10);
  return (end && *end == '\0') ? static_cast<int64_t>(v) : fallback;
}

}  // namespace

cudaError_t launch_step_coop(const KParams& p, int gdt, int num_sms, void* ws, cudaStream_t s,
                             bool* launched) {
  *launched = false;
  if (env_int("ZDP_COOP", 1) == 0) return cudaSuccess;
  const void* fn = gdt == ZDP_BF16 ? coop_kernel<ZDP_BF16>(p.P) : coop_kernel<ZDP_FP16>(p.P);
  if (!fn) return cudaSuccess;
  const int res = resident_blocks(fn);
  const int64_t nvec = (p.hi + kVec - 1) / kVec - p.lo / kVec;
  // One vector per thread while the range fits one resident wave of threads
  // (most latency hiding), up to kCoopV per thread beyond that.
  const int64_t most = static_cast<int64_t>(res) * num_sms;
  if (nvec <= 0 || nvec > most * kThreads * kCoopV) return cudaSuccess;  // does not fit
  const int grid = static_cast<int>(std::min(most, (nvec + kThreads - 1) / kThreads));
  CoopParams c;
  c.k = p;
  c.ws_flag = static_cast<int32_t*>(ws);
  c.arrived = reinterpret_cast<uint32_t*>(static_cast<char*>(ws) + 4);
  // A test hook: extra arrivals that never come make the barrier time out.
  // (never fewer than grid: the barrier must not open before every block arrived)
  const int64_t extra = std::max<int64_t>(0, env_int("ZDP_TEST_COOP_EXTRA_ARRIVALS", 0));
  c.expected = static_cast<uint32_t>(grid + std::min<int64_t>(extra, 1 << 20));
  c.timeout_ns = static_cast<uint64_t>(
      std::max<int64_t>(1000, env_int("ZDP_COOP_TIMEOUT_NS", 1000000000)));
  cudaError_t e = cudaMemsetAsync(ws, 0, 8, s);
  if (e != cudaSuccess) return e;
  void* args[] = {&c};
  e = cudaLaunchCooperativeKernel(fn, dim3(grid), dim3(kThreads), args, 0, s);
  if (e == cudaSuccess) *launched = true;
  return e;
}

}  // namespace zdp
