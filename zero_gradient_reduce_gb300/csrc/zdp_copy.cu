// zdp_copy.cu -- a plain 128-bit device copy with the step's own access
// pattern (16-byte ld.global.cs / st.global.cs, persistent grid-stride grid
// of 128-thread blocks).  It has no counterpart on the pages: it measures the
// copy ceiling that the streaming kernels are held against.
#include <algorithm>

#include "zdp_kernels.cuh"

namespace zdp {
namespace {

// 5 resident blocks per SM with 4 vectors in flight per thread (40 KB of
// loads in flight per SM) measured best of caps 2..16 and unrolls 2, 4, 8 on
// GB300: 6.6-6.7 TB/s, against 3.6 TB/s at 2 x 2 and 6.2 TB/s at 16 x 4.
#ifndef ZDP_COPY_UNROLL
#define ZDP_COPY_UNROLL 4
#endif
constexpr int kCopyUnroll = ZDP_COPY_UNROLL;  // 16-byte vectors in flight per thread

#ifndef ZDP_CAP_COPY
#define ZDP_CAP_COPY 5
#endif

// dst, src: `nvec` 16-byte vectors, both 16-byte aligned, not overlapping.
__global__ void __launch_bounds__(kThreads) k_copy16(uint4* __restrict__ dst,
                                                     const uint4* __restrict__ src,
                                                     int64_t nvec) {
  const int64_t T = static_cast<int64_t>(gridDim.x) * kThreads;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  const int64_t chunk = T * kCopyUnroll;
  int64_t base = 0;
  for (; base + chunk <= nvec; base += chunk) {  // whole chunks: all loads, then all stores
    uint4 x[kCopyUnroll];
#pragma unroll
    for (int k = 0; k < kCopyUnroll; ++k) x[k] = ld16(src + base + k * T + t);
#pragma unroll
    for (int k = 0; k < kCopyUnroll; ++k) st16(dst + base + k * T + t, x[k]);
  }
  for (int64_t i = base + t; i < nvec; i += T) st16(dst + i, ld16(src + i));
}

}  // namespace

cudaError_t launch_copy(void* dst, const void* src, int64_t bytes, int num_sms, cudaStream_t s) {
  const int64_t nvec = bytes / 16;
  if (nvec == 0) return cudaSuccess;
  const void* fn = reinterpret_cast<const void*>(&k_copy16);
  const int res = resident_blocks(fn);
  const int64_t per_sm = std::max(1, std::min(res, ZDP_CAP_COPY));
  const int64_t need = (nvec + kThreads - 1) / kThreads;
  const int grid = static_cast<int>(std::max<int64_t>(1, std::min(need, num_sms * per_sm)));
  k_copy16<<<grid, kThreads, 0, s>>>(static_cast<uint4*>(dst), static_cast<const uint4*>(src),
                                     nvec);
  return cudaGetLastError();
}

}  // namespace zdp
