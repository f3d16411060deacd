// zdp_internal.h -- declarations shared by the host API (zdp_api.cu) and the
// kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "zdp.h"

namespace zdp {

#ifndef ZDP_THREADS
#define ZDP_THREADS 128
#endif
constexpr int kThreads = ZDP_THREADS;  // threads per block of the streaming kernels

// Resident blocks per SM for each streaming kernel (at most; fewer if the
// kernel's registers do not allow it).  HBM throughput of these kernels
// peaks at a moderate number of loads in flight per SM and falls again when
// more threads are resident; the caps are the measured optima on GB300
// (fused step: see fused_cap; reduce-scatter, which keeps only its gradient
// loads in flight: see reduce_cap; AdamW 640 threads per SM; AdamW with the
// replica stores: see adam_gather_cap; all-gather: see gather_cap).
#ifndef ZDP_CAP_FUSED_BF16M_SMALL_P
#define ZDP_CAP_FUSED_BF16M_SMALL_P 12
#endif
#ifndef ZDP_CAP_ADAM_GATHER_BF16M
#define ZDP_CAP_ADAM_GATHER_BF16M 7
#endif

// Blocks per SM of the fused step for P ranks and the moment type.  With
// fp32 moments, measured over caps 2..8 for P = 1..16, 24, 32, 40, 48, 56, 64
// (fraction of the copy ceiling at the chosen cap): P = 1: 5 (0.94); 2: 6
// (0.95; 5 gave 0.87); 3: 5 (0.96); 4: 4 (0.95); 5..7: 5 (0.97-0.98); 8: 4
// (0.97); 9..15, the partial-group template: 3 (0.95-0.99); 16..32: 4
// (0.94-0.99); above 32: 3 (0.98-0.99 at 40, 48, 56, 64).  The optimum is
// not monotonic in P: it follows each template's registers and bytes in
// flight.  bf16 moments leave fewer bytes in flight per thread and want more
// threads: 12 blocks at P <= 3, 8 at P = 4..7, 7 at P = 8..15, 6 above.
inline int fused_cap(int P, int mt) {
  if (mt == ZDP_MOMENTS_F32) {
    if (P <= 8) return P == 2 ? 6 : ((P == 4 || P == 8) ? 4 : 5);
    return P < 16 ? 3 : (P <= 32 ? 4 : 3);
  }
  if (P <= 3) return ZDP_CAP_FUSED_BF16M_SMALL_P;
  return P < 8 ? 8 : (P < 16 ? 7 : 6);
}

// Whether the fused step with the sum of squares tests the squares' range per
// vector (k_fused<..., SQV = true>) rather than per element, for P ranks and
// the moment type.  Both give the same bits; which is faster depends on the
// compiled kernel.  Measured on GB300 (time per element / time per vector),
// fp32 moments: P = 1: 1.016, 2: 0.996, 3: 0.989, 4: 1.018, 5: 0.999, 6:
// 1.001, 7: 0.994, 8: 1.009, 12: 0.988, 16: 0.987, 24: 0.996, 32: 1.000, 40:
// 1.011, 48: 1.007, 56: 1.006, 64: 1.005; bf16 moments: P = 2: 1.009, 4:
// 0.988, 8: 0.989, 64: 1.004.  Chosen where the gain is at least 0.5 %.
// (Of these, P = 1, 4 and 8 with fp32 moments and P = 2 with bf16 moments now
// run k_fused_mt, which tests per vector; see pick_fused_mt.)
inline bool fused_sqv(int P, int mt) {
  if (mt != ZDP_MOMENTS_F32) return P == 2;
  return P == 1 || P == 4 || P == 8 || P == 40 || P == 48 || P == 56 || P == 64;
}

// Blocks per SM of the reduce-scatter for P ranks; measured fractions of the
// copy ceiling at the chosen caps: P = 2: 8 blocks, 0.95; P = 4: 16, 0.99
// (12: 0.96); P = 8, 16, 64: 12, 0.98-0.99.
inline int reduce_cap(int P) { return P <= 3 ? 8 : (P < 8 ? 16 : 12); }
#ifndef ZDP_CAP_ADAM
#define ZDP_CAP_ADAM 5
#endif

// Blocks per SM of the flag-gated AdamW + all-gather (the checked step's
// second pass) for P replicas and the moment type; with fp32 moments,
// measured on the two-pass checked step: P = 2: 5 (0.92 of the copy
// ceiling; 4 gave 0.87); P = 4: 4 (0.98); P = 8 and 16: 3 (0.94, 0.93);
// P = 64: any cap, 0.92.  bf16 moments: 7.
inline int adam_gather_cap(int P, int mt) {
  if (mt != ZDP_MOMENTS_F32) return ZDP_CAP_ADAM_GATHER_BF16M;
  return P <= 2 ? 5 : (P <= 4 ? 4 : 3);
}

// Blocks per SM of the all-gather for P replicas.  A thread reads 32 bytes
// and writes 16P per vector, so small P needs more threads for the same
// bytes in flight; measured fractions of the copy ceiling at the chosen caps:
// P = 1 and 2: 8 blocks, 0.97 and 1.00 (3 blocks: 0.64 at P = 2); P = 4: 6,
// 0.94; P = 8: 3, 0.93; P >= 16: 2, 0.88-0.89.
inline int gather_cap(int P) { return P <= 2 ? 8 : (P <= 4 ? 6 : (P <= 8 ? 3 : 2)); }
constexpr int kVec = 8;        // elements per vector: 16 B of bf16, 32 B of fp32

// AdamW constants, prepared once per call on the host.
struct AdamK {
  float lr, b1, b2, eps;
  float one_minus_b1, one_minus_b2;  // fp32 1-b1, 1-b2
  float lr_wd;                       // fp32 lr*wd
  float bc1, bc2;                    // fp32 rounding of the double 1-b^t
};

// Everything a kernel needs, passed by value as a __grid_constant__ parameter.
// Element indices are global (0..n); each pointer family says how it maps a
// global index to an address.
struct KParams {
  // rank q's gradient of global element i: g[q] + (i - goff) * esize
  const void* g[ZDP_MAX_P];
  // rank q's replica of global element i: rep[q][i]
  uint16_t* rep[ZDP_MAX_P];
  float* w;  // master: w[i]
  void* m;   // first moment m[i]: fp32, or bf16 when mt == ZDP_MOMENTS_BF16
  void* v;   // second moment v[i], same type
  int mt;    // zdp_moment_dtype of m and v
  const float* gin;  // reduced gradient input: gin[i - gin_base]
  float* gout;       // reduced gradient output: gout[i - gout_base]
  int64_t goff, gin_base, gout_base;
  int64_t S;       // shard size; owner of i is i / S
  int64_t lo, hi;  // this launch processes global elements [lo, hi)
  float inv_s;     // fp32 1/S, for the owner estimate
  int P;           // ranks whose gradients are summed
  int nrep;        // replicas written (0..P)
  float scale;
  AdamK ad;
  int32_t* flag;       // nullable: OR-ed with 1 on a non-finite reduced gradient
  double* sumsq;       // nullable: fp64 sum of squares of reduced gradients added
  const int32_t* gate; // nullable: when *gate != 0 the launch writes nothing
};

// Launchers, one per kernel family.  `vec` selects the 16-byte-access
// kernels (every buffer's element 0 on a 16-byte boundary).  The grid is a
// persistent grid-stride grid: `num_sms` times the kernel's resident blocks
// per SM, capped by the work.  Each returns the launch status.
// The fused and reduce kernels add the sum of squares when p.sumsq is set.
// overlap_prev: launch with programmatic stream serialization, so that the
// blocks of this launch may start while the previous launch on the stream
// (a launch of the same kernel over a disjoint range) drains.  k_fused,
// k_reduce and k_adam_gather wait for that launch before exiting, so stream
// order still holds for whatever follows.
cudaError_t launch_kernel(const void* fn, int grid, void** args, cudaStream_t s,
                          bool overlap_prev);
cudaError_t launch_fused(const KParams& p, int gdt, bool vec, int num_sms, cudaStream_t s,
                         bool overlap_prev = false);
cudaError_t launch_reduce(const KParams& p, int gdt, bool vec, int num_sms, cudaStream_t s,
                          bool overlap_prev = false);
cudaError_t launch_adam_gather(const KParams& p, bool vec, int num_sms, cudaStream_t s,
                               bool overlap_prev = false);
// The overflow-checked step in one cooperative launch over [p.lo, p.hi)
// (16-byte vector path only).  ws: the call's workspace, whose first 8 bytes
// it zeroes and uses.  Sets *launched = false, launching nothing, when the
// range does not fit one resident wave, P has no template, or ZDP_COOP=0.
cudaError_t launch_step_coop(const KParams& p, int gdt, int num_sms, void* ws, cudaStream_t s,
                             bool* launched);
cudaError_t launch_gather(const KParams& p, bool vec, int num_sms, cudaStream_t s);

// The literal ring schedule of zdp_step_ring (zdp_ring.cu); `ws` holds the
// 2 * P * S fp32 messages.
cudaError_t launch_ring(const zdp_step_args* a, const AdamK& ad, float* ws, bool vec, int num_sms,
                        cudaStream_t s);

// ZeRO++ kernels (zdp_zpp.cu).
cudaError_t launch_zpp(const zdp_zpp_args* a, const AdamK& ad, int num_sms, cudaStream_t s);
cudaError_t launch_quantize(const void* x, int xdt, int64_t n, int8_t* q, float* scales,
                            int num_sms, cudaStream_t s);
cudaError_t launch_copy(void* dst, const void* src, int64_t bytes, int num_sms, cudaStream_t s);
cudaError_t launch_dequantize(const int8_t* q, const float* scales, int64_t n, uint16_t* out,
                              int num_sms, cudaStream_t s);

// Sets this host thread's zdp_last_error() message; returns `code`.
int report_error(int code, const char* msg);

// Blocks of kThreads threads of `kernel` that fit on one SM (queried once
// per kernel, then cached).  A persistent grid larger than one wave of them
// would leave a partial last wave.
int resident_blocks(const void* kernel);

// Grid size for `kernel` over the elements [p.lo, p.hi): min(resident
// blocks per SM (queried once per kernel and cached), cap) times num_sms,
// capped by the work.
int grid_for(const void* kernel, const KParams& p, bool vec, int num_sms, int cap);

}  // namespace zdp
