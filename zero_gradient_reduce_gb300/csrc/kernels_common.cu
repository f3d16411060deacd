// Kernels that do not read rank gradients (AdamW from reduced gradients,
// cast + all-gather), the per-type dispatch, and grid sizing.
#include <mutex>
#include <unordered_map>

#include "zdp_kernels.cuh"

namespace zdp {

cudaError_t launch_fused_bf16(const KParams& p, bool vec, int num_sms, cudaStream_t s,
                              bool overlap_prev);
cudaError_t launch_fused_fp16(const KParams& p, bool vec, int num_sms, cudaStream_t s,
                              bool overlap_prev);
cudaError_t launch_reduce_bf16(const KParams& p, bool vec, int num_sms, cudaStream_t s,
                               bool overlap_prev);
cudaError_t launch_step_coop_bf16(const KParams& p, int num_sms, void* ws, cudaStream_t s,
                                  bool* launched);
cudaError_t launch_step_coop_fp16(const KParams& p, int num_sms, void* ws, cudaStream_t s,
                                  bool* launched);
cudaError_t launch_reduce_fp16(const KParams& p, bool vec, int num_sms, cudaStream_t s,
                               bool overlap_prev);

int resident_blocks(const void* kernel) {
  static std::mutex mu;
  static std::unordered_map<const void*, int> resident;
  std::lock_guard<std::mutex> lock(mu);
  auto it = resident.find(kernel);
  if (it != resident.end()) return it->second;
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, kThreads, 0) != cudaSuccess ||
      occ < 1) {
    occ = 1;
  }
  resident[kernel] = occ;
  return occ;
}

int grid_for(const void* kernel, const KParams& p, bool vec, int num_sms, int cap) {
  const int64_t work = vec ? (p.hi + kVec - 1) / kVec - p.lo / kVec : p.hi - p.lo;
  if (work <= 0) return 0;
  int occ = resident_blocks(kernel);
  // The caps pay off when every thread walks many vectors; a launch too
  // small to give each capped thread two of them is latency-bound and runs
  // at full occupancy instead (tiny step: 14.4 against 16.2 us).
  const int64_t capped = static_cast<int64_t>(num_sms) * (occ < cap ? occ : cap);
  if (work >= 2 * capped * kThreads && occ > cap) occ = cap;
  const int64_t full = static_cast<int64_t>(num_sms) * occ;
  const int64_t need = (work + kThreads - 1) / kThreads;
  return static_cast<int>(need < full ? need : full);
}

cudaError_t launch_kernel(const void* fn, int grid, void** args, cudaStream_t s,
                          bool overlap_prev) {
  if (!ZDP_PDL || !overlap_prev) return cudaLaunchKernel(fn, dim3(grid), dim3(kThreads), args, 0, s);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

namespace {
cudaError_t launch_fn(const void* fn, const KParams& p, bool vec, int num_sms, int cap,
                      cudaStream_t s, bool overlap_prev = false) {
  const int grid = grid_for(fn, p, vec, num_sms, cap);
  if (grid == 0) return cudaSuccess;
  void* args[] = {const_cast<KParams*>(&p)};
  return launch_kernel(fn, grid, args, s, overlap_prev);
}
}  // namespace

cudaError_t launch_fused(const KParams& p, int gdt, bool vec, int num_sms, cudaStream_t s,
                         bool overlap_prev) {
  return gdt == ZDP_BF16 ? launch_fused_bf16(p, vec, num_sms, s, overlap_prev)
                         : launch_fused_fp16(p, vec, num_sms, s, overlap_prev);
}

cudaError_t launch_step_coop(const KParams& p, int gdt, int num_sms, void* ws, cudaStream_t s,
                             bool* launched) {
  return gdt == ZDP_BF16 ? launch_step_coop_bf16(p, num_sms, ws, s, launched)
                         : launch_step_coop_fp16(p, num_sms, ws, s, launched);
}

cudaError_t launch_reduce(const KParams& p, int gdt, bool vec, int num_sms, cudaStream_t s,
                          bool overlap_prev) {
  return gdt == ZDP_BF16 ? launch_reduce_bf16(p, vec, num_sms, s, overlap_prev)
                         : launch_reduce_fp16(p, vec, num_sms, s, overlap_prev);
}

cudaError_t launch_adam_gather(const KParams& p, bool vec, int num_sms, cudaStream_t s,
                               bool overlap_prev) {
  if (vec && p.nrep == 8 && p.mt == ZDP_MOMENTS_F32)
    return launch_fn(reinterpret_cast<const void*>(&k_adam_gather_mt<8, ZDP_MOMENTS_F32>), p, vec,
                     num_sms, adam_gather_cap(p.nrep, p.mt), s, overlap_prev);
  const void* fn = vec ? reinterpret_cast<const void*>(&k_adam_gather<true>)
                       : reinterpret_cast<const void*>(&k_adam_gather<false>);
  const int cap = p.nrep == 0 ? ZDP_CAP_ADAM : adam_gather_cap(p.nrep, p.mt);
  return launch_fn(fn, p, vec, num_sms, cap, s, overlap_prev);
}

cudaError_t launch_gather(const KParams& p, bool vec, int num_sms, cudaStream_t s) {
  const void* fn = vec ? reinterpret_cast<const void*>(&k_gather<true>)
                       : reinterpret_cast<const void*>(&k_gather<false>);
  return launch_fn(fn, p, vec, num_sms, gather_cap(p.nrep), s);
}

}  // namespace zdp
