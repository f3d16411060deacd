// zdp_api.cu -- the C ABI of libzdp: argument checks, kernel parameters and
// launches.  Declarations and their documentation are in include/zdp.h.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "zdp_internal.h"

namespace {

thread_local std::string g_err;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}

int ok() {
  g_err.clear();
  return ZDP_OK;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(ZDP_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool valid_p(int P) { return P >= 1 && P <= ZDP_MAX_P; }

int64_t shard(int64_t n, int P) { return (n + P - 1) / P; }

uintptr_t addr(const void* p) { return reinterpret_cast<uintptr_t>(p); }

// Byte ranges of the buffers a call touches; any overlap between two of them
// (outputs among themselves or with inputs) is rejected.
struct Range {
  uintptr_t lo, hi;
  const char* what;
  int index;
};

int check_disjoint(std::vector<Range>& rs) {
  std::sort(rs.begin(), rs.end(), [](const Range& a, const Range& b) { return a.lo < b.lo; });
  for (size_t k = 1; k < rs.size(); ++k) {
    if (rs[k].lo < rs[k - 1].hi) {
      return fail(ZDP_ERR_INVALID, "buffers overlap: %s[%d] and %s[%d]", rs[k - 1].what,
                  rs[k - 1].index, rs[k].what, rs[k].index);
    }
  }
  return ZDP_OK;
}

void add_range(std::vector<Range>& rs, const void* p, int64_t bytes, const char* what, int idx) {
  if (p && bytes > 0) rs.push_back({addr(p), addr(p) + static_cast<uintptr_t>(bytes), what, idx});
}

// SM count of the current device, cached per device (any host thread may call).
int num_sms(int* out) {
  static std::atomic<int> cache[128];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  const bool cached = dev >= 0 && dev < 128;
  if (cached) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) {
      *out = c;
      return ZDP_OK;
    }
  }
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
  if (cached) cache[dev].store(sms, std::memory_order_relaxed);
  *out = sms;
  return ZDP_OK;
}

zdp::AdamK make_adam(float lr, float b1, float b2, float eps, float wd, int t) {
  zdp::AdamK a;
  a.lr = lr;
  a.b1 = b1;
  a.b2 = b2;
  a.eps = eps;
  // fp32 arithmetic on fp32 operands, each result rounded once.
  volatile float one = 1.0f;
  a.one_minus_b1 = one - b1;
  a.one_minus_b2 = one - b2;
  volatile float lrv = lr;
  a.lr_wd = lrv * wd;
  a.bc1 = static_cast<float>(1.0 - std::pow(static_cast<double>(b1), static_cast<double>(t)));
  a.bc2 = static_cast<float>(1.0 - std::pow(static_cast<double>(b2), static_cast<double>(t)));
  return a;
}

void init_params(zdp::KParams& p) { std::memset(&p, 0, sizeof p); }

bool aligned16(const void* p) { return (addr(p) & 15u) == 0; }

}  // namespace

namespace zdp {
// Records `msg` as this thread's zdp_last_error() text and returns `code`.
int report_error(int code, const char* msg) { return fail(code, "%s", msg); }
}  // namespace zdp

extern "C" {

int zdp_version(void) { return 100; }

const char* zdp_last_error(void) { return g_err.c_str(); }

int64_t zdp_shard_size(int64_t n, int P) {
  if (n < 1 || !valid_p(P)) return -1;
  return shard(n, P);
}

int zdp_reduce_scatter(const void* const* grads, int gdt, float* shards, int64_t n, int P,
                       float scale, int32_t* d_overflow, double* d_sumsq, void* stream) {
  if (!valid_p(P)) return fail(ZDP_ERR_INVALID, "P=%d outside 1..%d", P, ZDP_MAX_P);
  if (n < 1) return fail(ZDP_ERR_INVALID, "n=%lld must be >= 1", static_cast<long long>(n));
  if (gdt != ZDP_BF16 && gdt != ZDP_FP16) return fail(ZDP_ERR_INVALID, "bad gradient type %d", gdt);
  if (!grads) return fail(ZDP_ERR_INVALID, "grads is NULL");
  if (!shards) return fail(ZDP_ERR_INVALID, "shards is NULL");
  if ((addr(shards) & 3u) != 0) return fail(ZDP_ERR_INVALID, "shards not 4-byte aligned");
  const int64_t S = shard(n, P);
  bool vec = aligned16(shards);
  for (int q = 0; q < P; ++q) {
    if (!grads[q]) return fail(ZDP_ERR_INVALID, "grads[%d] is NULL", q);
    if ((addr(grads[q]) & 1u) != 0) return fail(ZDP_ERR_INVALID, "grads[%d] not 2-byte aligned", q);
    vec = vec && aligned16(grads[q]);
  }
  // Ranks may share one gradient buffer (inputs); outputs may not touch them.
  {
    std::vector<Range> outs;
    add_range(outs, shards, P * S * 4, "shards", 0);
    add_range(outs, d_overflow, 4, "d_overflow", 0);
    add_range(outs, d_sumsq, 8, "d_sumsq", 0);
    if (check_disjoint(outs) != ZDP_OK) return ZDP_ERR_INVALID;
    for (int q = 0; q < P; ++q) {
      for (const Range& o : outs) {
        const uintptr_t lo = addr(grads[q]), hi = lo + static_cast<uintptr_t>(n * 2);
        if (lo < o.hi && o.lo < hi)
          return fail(ZDP_ERR_INVALID, "buffers overlap: grads[%d] and %s", q, o.what);
      }
    }
  }
  int sms = 0;
  if (num_sms(&sms) != ZDP_OK) return ZDP_ERR_CUDA;
  zdp::KParams p;
  init_params(p);
  for (int q = 0; q < P; ++q) p.g[q] = grads[q];
  p.goff = 0;
  p.gout = shards;
  p.gout_base = 0;
  p.S = S;
  p.inv_s = 1.0f / static_cast<float>(S);
  p.lo = 0;
  p.hi = n;
  p.P = P;
  p.scale = scale;
  p.flag = d_overflow;
  p.sumsq = d_sumsq;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = zdp::launch_reduce(p, gdt, vec, sms, s);
  if (e != cudaSuccess) return cuda_fail(e, "reduce-scatter launch");
  if (P * S > n) {
    e = cudaMemsetAsync(shards + n, 0, static_cast<size_t>(P * S - n) * 4, s);
    if (e != cudaSuccess) return cuda_fail(e, "padding memset");
  }
  return ok();
}

int zdp_adamw_shard(float* master, float* m, float* v, const float* grad_shard, int64_t count,
                    float lr, float b1, float b2, float eps, float wd, int t, void* stream) {
  if (count < 0) return fail(ZDP_ERR_INVALID, "count=%lld < 0", static_cast<long long>(count));
  if (t < 1) return fail(ZDP_ERR_INVALID, "t=%d must be >= 1", t);
  if (count == 0) return ok();
  if (!master || !m || !v || !grad_shard) return fail(ZDP_ERR_INVALID, "NULL buffer");
  const void* bufs[4] = {master, m, v, grad_shard};
  for (const void* b : bufs)
    if ((addr(b) & 3u) != 0) return fail(ZDP_ERR_INVALID, "fp32 buffer not 4-byte aligned");
  std::vector<Range> rs;
  add_range(rs, master, count * 4, "master", 0);
  add_range(rs, m, count * 4, "m", 0);
  add_range(rs, v, count * 4, "v", 0);
  add_range(rs, grad_shard, count * 4, "grad_shard", 0);
  if (check_disjoint(rs) != ZDP_OK) return ZDP_ERR_INVALID;
  int sms = 0;
  if (num_sms(&sms) != ZDP_OK) return ZDP_ERR_CUDA;
  zdp::KParams p;
  init_params(p);
  p.w = master;
  p.m = m;
  p.v = v;
  p.mt = ZDP_MOMENTS_F32;
  p.gin = grad_shard;
  p.gin_base = 0;
  p.lo = 0;
  p.hi = count;
  p.nrep = 0;
  p.ad = make_adam(lr, b1, b2, eps, wd, t);
  const bool vec = aligned16(master) && aligned16(m) && aligned16(v) && aligned16(grad_shard);
  cudaError_t e = zdp::launch_adam_gather(p, vec, sms, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "adamw launch");
  return ok();
}

int zdp_all_gather(const float* master, uint16_t* const* replicas, int64_t n, int P,
                   void* stream) {
  if (!valid_p(P)) return fail(ZDP_ERR_INVALID, "P=%d outside 1..%d", P, ZDP_MAX_P);
  if (n < 1) return fail(ZDP_ERR_INVALID, "n=%lld must be >= 1", static_cast<long long>(n));
  if (!master) return fail(ZDP_ERR_INVALID, "master is NULL");
  if (!replicas) return fail(ZDP_ERR_INVALID, "replicas is NULL");
  if ((addr(master) & 3u) != 0) return fail(ZDP_ERR_INVALID, "master not 4-byte aligned");
  std::vector<Range> rs;
  add_range(rs, master, n * 4, "master", 0);
  bool vec = aligned16(master);
  for (int q = 0; q < P; ++q) {
    if (!replicas[q]) return fail(ZDP_ERR_INVALID, "replicas[%d] is NULL", q);
    if ((addr(replicas[q]) & 1u) != 0)
      return fail(ZDP_ERR_INVALID, "replicas[%d] not 2-byte aligned", q);
    vec = vec && aligned16(replicas[q]);
    add_range(rs, replicas[q], n * 2, "replicas", q);
  }
  if (check_disjoint(rs) != ZDP_OK) return ZDP_ERR_INVALID;
  int sms = 0;
  if (num_sms(&sms) != ZDP_OK) return ZDP_ERR_CUDA;
  zdp::KParams p;
  init_params(p);
  p.w = const_cast<float*>(master);
  for (int q = 0; q < P; ++q) p.rep[q] = replicas[q];
  p.nrep = P;
  p.lo = 0;
  p.hi = n;
  cudaError_t e = zdp::launch_gather(p, vec, sms, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "all-gather launch");
  return ok();
}

int zdp_copy(void* dst, const void* src, int64_t bytes, void* stream) {
  if (bytes < 0 || bytes % 16 != 0)
    return fail(ZDP_ERR_INVALID, "bytes=%lld must be a non-negative multiple of 16",
                static_cast<long long>(bytes));
  if (bytes == 0) return ok();
  if (!dst || !src) return fail(ZDP_ERR_INVALID, "dst or src is NULL");
  if (!aligned16(dst) || !aligned16(src))
    return fail(ZDP_ERR_INVALID, "dst and src must be 16-byte aligned");
  std::vector<Range> rs;
  add_range(rs, dst, bytes, "dst", 0);
  add_range(rs, src, bytes, "src", 0);
  if (check_disjoint(rs) != ZDP_OK) return ZDP_ERR_INVALID;
  int sms = 0;
  if (num_sms(&sms) != ZDP_OK) return ZDP_ERR_CUDA;
  cudaError_t e = zdp::launch_copy(dst, src, bytes, sms, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "copy launch");
  return ok();
}

size_t zdp_step_workspace_bytes(const zdp_step_args* a) {
  if (!a || !a->check_overflow || a->len <= 0) return 0;
  // 256 B for the device flag, then the reduced gradients of the range,
  // starting at the global multiple of 8 at or below `off`.
  const size_t body = static_cast<size_t>(a->len + 8) * 4;
  return 256 + ((body + 255) / 256) * 256;
}

}  // extern "C"

namespace {

// Checks of zdp_step / zdp_step_ring arguments; `ws_need` is the workspace the
// call needs (0: none).  Sets *vec when every buffer's element 0 is 16-byte
// aligned.  Returns ZDP_OK, or ZDP_ERR_INVALID with the message set.
int validate_step(const zdp_step_args* a, size_t ws_need, bool* vec_out) {
  if (!a) return fail(ZDP_ERR_INVALID, "args is NULL");
  const int P = a->P;
  if (!valid_p(P)) return fail(ZDP_ERR_INVALID, "P=%d outside 1..%d", P, ZDP_MAX_P);
  if (a->n < 1) return fail(ZDP_ERR_INVALID, "n=%lld must be >= 1", static_cast<long long>(a->n));
  if (a->off < 0 || a->len < 0 || a->off > a->n || a->len > a->n - a->off)
    return fail(ZDP_ERR_INVALID, "range [%lld, %lld+%lld) outside [0, n=%lld)",
                static_cast<long long>(a->off), static_cast<long long>(a->off),
                static_cast<long long>(a->len), static_cast<long long>(a->n));
  if (a->gdt != ZDP_BF16 && a->gdt != ZDP_FP16)
    return fail(ZDP_ERR_INVALID, "bad gradient type %d", a->gdt);
  if (a->t < 1) return fail(ZDP_ERR_INVALID, "t=%d must be >= 1", a->t);
  if (a->bucket_elems < 0) return fail(ZDP_ERR_INVALID, "bucket_elems < 0");
  if (!a->grads || !a->replicas) return fail(ZDP_ERR_INVALID, "grads or replicas is NULL");
  if (!a->master || !a->m || !a->v) return fail(ZDP_ERR_INVALID, "master, m or v is NULL");
  if (a->moment_dtype != ZDP_MOMENTS_F32 && a->moment_dtype != ZDP_MOMENTS_BF16)
    return fail(ZDP_ERR_INVALID, "bad moment type %d", a->moment_dtype);
  const int64_t n = a->n, off = a->off, len = a->len;
  const int64_t mbytes = a->moment_dtype == ZDP_MOMENTS_F32 ? 4 : 2;
  if ((addr(a->master) & 3u) != 0) return fail(ZDP_ERR_INVALID, "master not 4-byte aligned");
  if ((addr(a->m) & (mbytes - 1)) != 0 || (addr(a->v) & (mbytes - 1)) != 0)
    return fail(ZDP_ERR_INVALID, "m or v not aligned to its element size");
  bool vec = aligned16(a->master) && aligned16(a->m) && aligned16(a->v);
  std::vector<Range> outs;
  add_range(outs, a->master, n * 4, "master", 0);
  add_range(outs, a->m, n * mbytes, "m", 0);
  add_range(outs, a->v, n * mbytes, "v", 0);
  for (int q = 0; q < P; ++q) {
    if (!a->grads[q]) return fail(ZDP_ERR_INVALID, "grads[%d] is NULL", q);
    if (!a->replicas[q]) return fail(ZDP_ERR_INVALID, "replicas[%d] is NULL", q);
    if ((addr(a->grads[q]) & 1u) != 0)
      return fail(ZDP_ERR_INVALID, "grads[%d] not 2-byte aligned", q);
    if ((addr(a->replicas[q]) & 1u) != 0)
      return fail(ZDP_ERR_INVALID, "replicas[%d] not 2-byte aligned", q);
    // element off of rank q's gradient must sit where a global multiple of 8 would be 16-B aligned
    vec = vec && ((addr(a->grads[q]) - static_cast<uintptr_t>(off) * 2u) & 15u) == 0;
    vec = vec && aligned16(a->replicas[q]);
    add_range(outs, a->replicas[q], n * 2, "replicas", q);
  }
  add_range(outs, a->d_overflow, 4, "d_overflow", 0);
  add_range(outs, a->d_sumsq, 8, "d_sumsq", 0);
  if (ws_need > 0) {
    if (!a->workspace) return fail(ZDP_ERR_INVALID, "this call needs a workspace");
    if (a->workspace_bytes < ws_need)
      return fail(ZDP_ERR_INVALID, "workspace of %zu bytes, need %zu", a->workspace_bytes, ws_need);
    if (!aligned16(a->workspace)) return fail(ZDP_ERR_INVALID, "workspace not 16-byte aligned");
    add_range(outs, a->workspace, static_cast<int64_t>(ws_need), "workspace", 0);
  }
  if (check_disjoint(outs) != ZDP_OK) return ZDP_ERR_INVALID;
  for (int q = 0; q < P; ++q) {
    const uintptr_t lo = addr(a->grads[q]), hi = lo + static_cast<uintptr_t>(len * 2);
    for (const Range& o : outs)
      if (lo < o.hi && o.lo < hi)
        return fail(ZDP_ERR_INVALID, "buffers overlap: grads[%d] and %s[%d]", q, o.what, o.index);
  }
  *vec_out = vec;
  return ZDP_OK;
}

}  // namespace

extern "C" {

int zdp_step(const zdp_step_args* a, void* stream) {
  if (a && a->len == 0 && a->P >= 1 && a->P <= ZDP_MAX_P && a->n >= 1 && a->off >= 0 &&
      a->off <= a->n && a->t >= 1 && a->grads && a->replicas && a->master && a->m && a->v &&
      (a->gdt == ZDP_BF16 || a->gdt == ZDP_FP16) && a->bucket_elems >= 0 &&
      (a->moment_dtype == ZDP_MOMENTS_F32 || a->moment_dtype == ZDP_MOMENTS_BF16))
    return ok();
  bool vec = false;
  if (validate_step(a, zdp_step_workspace_bytes(a), &vec) != ZDP_OK) return ZDP_ERR_INVALID;
  const int P = a->P;
  const int64_t n = a->n, off = a->off, len = a->len;
  int sms = 0;
  if (num_sms(&sms) != ZDP_OK) return ZDP_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t S = shard(n, P);

  zdp::KParams p;
  init_params(p);
  for (int q = 0; q < P; ++q) {
    p.g[q] = a->grads[q];
    p.rep[q] = a->replicas[q];
  }
  p.goff = off;
  p.w = a->master;
  p.m = a->m;
  p.v = a->v;
  p.mt = a->moment_dtype;
  p.S = S;
  p.inv_s = 1.0f / static_cast<float>(S);
  p.P = P;
  p.nrep = P;
  p.scale = a->scale;
  p.ad = make_adam(a->lr, a->b1, a->b2, a->eps, a->wd, a->t);
  const int64_t bucket = a->bucket_elems > 0 ? a->bucket_elems : len;

  if (!a->check_overflow) {
    p.flag = a->d_overflow;
    p.sumsq = a->d_sumsq;
    for (int64_t lo = off; lo < off + len; lo += bucket) {
      p.lo = lo;
      p.hi = std::min(off + len, lo + bucket);
      cudaError_t e = zdp::launch_fused(p, a->gdt, vec, sms, s, lo != off);
      if (e != cudaSuccess) return cuda_fail(e, "fused step launch");
    }
    return ok();
  }

  if (vec) {  // one cooperative launch when the range fits one resident wave
    p.lo = off;
    p.hi = off + len;
    p.flag = a->d_overflow;
    p.sumsq = a->d_sumsq;
    bool launched = false;
    cudaError_t e = zdp::launch_step_coop(p, a->gdt, sms, a->workspace, s, &launched);
    if (e != cudaSuccess) return cuda_fail(e, "single-pass checked step launch");
    if (launched) return ok();
  }

  // Two passes: reduced gradients and a device flag, then the gated update.
  int32_t* ws_flag = static_cast<int32_t*>(a->workspace);
  float* ws_g = reinterpret_cast<float*>(static_cast<char*>(a->workspace) + 256);
  const int64_t gbase = off & ~static_cast<int64_t>(7);
  cudaError_t e = cudaMemsetAsync(ws_flag, 0, 4, s);
  if (e != cudaSuccess) return cuda_fail(e, "flag reset");
  p.gout = ws_g;
  p.gout_base = gbase;
  p.flag = ws_flag;
  p.sumsq = a->d_sumsq;
  for (int64_t lo = off; lo < off + len; lo += bucket) {
    p.lo = lo;
    p.hi = std::min(off + len, lo + bucket);
    e = zdp::launch_reduce(p, a->gdt, vec, sms, s, lo != off);
    if (e != cudaSuccess) return cuda_fail(e, "reduce pass launch");
  }
  p.gout = nullptr;
  p.sumsq = nullptr;
  p.gin = ws_g;
  p.gin_base = gbase;
  p.gate = ws_flag;
  p.flag = a->d_overflow;  // the gated pass forwards a raised flag to the caller
  for (int64_t lo = off; lo < off + len; lo += bucket) {
    p.lo = lo;
    p.hi = std::min(off + len, lo + bucket);
    e = zdp::launch_adam_gather(p, vec, sms, s, lo != off);
    if (e != cudaSuccess) return cuda_fail(e, "update pass launch");
  }
  return ok();
}

size_t zdp_step_ring_workspace_bytes(const zdp_step_args* a) {
  if (!a || !valid_p(a->P) || a->n < 1) return 0;
  const size_t msgs = 2u * static_cast<size_t>(a->P) * static_cast<size_t>(shard(a->n, a->P)) * 4u;
  return (msgs + 255) / 256 * 256;
}

int zdp_step_ring(const zdp_step_args* a, void* stream) {
  if (!a) return fail(ZDP_ERR_INVALID, "args is NULL");
  if (a->off != 0 || a->len != a->n)
    return fail(ZDP_ERR_INVALID, "the ring schedule covers the whole model: off = 0, len = n");
  if (a->check_overflow) return fail(ZDP_ERR_INVALID, "zdp_step_ring has no overflow check");
  if (a->bucket_elems != 0) return fail(ZDP_ERR_INVALID, "zdp_step_ring takes no buckets");
  if (a->moment_dtype != ZDP_MOMENTS_F32)
    return fail(ZDP_ERR_INVALID, "zdp_step_ring takes fp32 moments only");
  bool vec = false;
  if (validate_step(a, zdp_step_ring_workspace_bytes(a), &vec) != ZDP_OK) return ZDP_ERR_INVALID;
  int sms = 0;
  if (num_sms(&sms) != ZDP_OK) return ZDP_ERR_CUDA;
  const zdp::AdamK ad = make_adam(a->lr, a->b1, a->b2, a->eps, a->wd, a->t);
  cudaError_t e = zdp::launch_ring(a, ad, static_cast<float*>(a->workspace), vec, sms,
                                   static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "ring step launch");
  return ok();
}

int zdp_quantize_blocks(const void* x, int xdt, int64_t n, int8_t* q, float* scales,
                        void* stream) {
  if (n < 1) return fail(ZDP_ERR_INVALID, "n=%lld must be >= 1", static_cast<long long>(n));
  if (xdt != ZDP_BF16 && xdt != ZDP_FP16 && xdt != ZDP_F32)
    return fail(ZDP_ERR_INVALID, "bad input type %d", xdt);
  if (!x || !q || !scales) return fail(ZDP_ERR_INVALID, "NULL buffer");
  const int64_t xb = xdt == ZDP_F32 ? 4 : 2;
  if ((addr(x) & (xb - 1)) != 0 || (addr(scales) & 3u) != 0)
    return fail(ZDP_ERR_INVALID, "misaligned buffer");
  std::vector<Range> rs;
  add_range(rs, x, n * xb, "x", 0);
  add_range(rs, q, n, "q", 0);
  add_range(rs, scales, (n + ZDP_QBLOCK - 1) / ZDP_QBLOCK * 4, "scales", 0);
  if (check_disjoint(rs) != ZDP_OK) return ZDP_ERR_INVALID;
  int sms = 0;
  if (num_sms(&sms) != ZDP_OK) return ZDP_ERR_CUDA;
  cudaError_t e = zdp::launch_quantize(x, xdt, n, q, scales, sms, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "quantize launch");
  return ok();
}

int zdp_dequantize_blocks(const int8_t* q, const float* scales, int64_t n, uint16_t* out,
                          void* stream) {
  if (n < 1) return fail(ZDP_ERR_INVALID, "n=%lld must be >= 1", static_cast<long long>(n));
  if (!q || !scales || !out) return fail(ZDP_ERR_INVALID, "NULL buffer");
  if ((addr(out) & 1u) != 0 || (addr(scales) & 3u) != 0)
    return fail(ZDP_ERR_INVALID, "misaligned buffer");
  std::vector<Range> rs;
  add_range(rs, q, n, "q", 0);
  add_range(rs, scales, (n + ZDP_QBLOCK - 1) / ZDP_QBLOCK * 4, "scales", 0);
  add_range(rs, out, n * 2, "out", 0);
  if (check_disjoint(rs) != ZDP_OK) return ZDP_ERR_INVALID;
  int sms = 0;
  if (num_sms(&sms) != ZDP_OK) return ZDP_ERR_CUDA;
  cudaError_t e = zdp::launch_dequantize(q, scales, n, out, sms, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "dequantize launch");
  return ok();
}

int zdp_step_zpp(const zdp_zpp_args* a, void* stream) {
  if (!a) return fail(ZDP_ERR_INVALID, "args is NULL");
  const int P = a->P;
  if (!valid_p(P)) return fail(ZDP_ERR_INVALID, "P=%d outside 1..%d", P, ZDP_MAX_P);
  if (a->n < 1) return fail(ZDP_ERR_INVALID, "n=%lld must be >= 1", static_cast<long long>(a->n));
  if (a->off < 0 || a->len < 0 || a->off > a->n || a->len > a->n - a->off)
    return fail(ZDP_ERR_INVALID, "range [%lld, %lld+%lld) outside [0, n=%lld)",
                static_cast<long long>(a->off), static_cast<long long>(a->off),
                static_cast<long long>(a->len), static_cast<long long>(a->n));
  if (a->off % ZDP_QBLOCK != 0 || ((a->off + a->len) % ZDP_QBLOCK != 0 && a->off + a->len != a->n))
    return fail(ZDP_ERR_INVALID, "the range must start on a %d-element block and end on one or at n",
                ZDP_QBLOCK);
  if (a->t < 1) return fail(ZDP_ERR_INVALID, "t=%d must be >= 1", a->t);
  if (a->moment_dtype != ZDP_MOMENTS_F32 && a->moment_dtype != ZDP_MOMENTS_BF16)
    return fail(ZDP_ERR_INVALID, "bad moment type %d", a->moment_dtype);
  if (!a->grads || !a->grad_scales || !a->replicas || !a->replica_scales)
    return fail(ZDP_ERR_INVALID, "a pointer array is NULL");
  if (!a->master || !a->m || !a->v) return fail(ZDP_ERR_INVALID, "master, m or v is NULL");
  if (a->len == 0) return ok();
  const int64_t n = a->n, len = a->len;
  const int64_t nb = (n + ZDP_QBLOCK - 1) / ZDP_QBLOCK;
  const int64_t lb = (len + ZDP_QBLOCK - 1) / ZDP_QBLOCK;
  const int64_t mbytes = a->moment_dtype == ZDP_MOMENTS_F32 ? 4 : 2;
  if (!aligned16(a->master) || !aligned16(a->m) || !aligned16(a->v))
    return fail(ZDP_ERR_INVALID, "master, m and v must be 16-byte aligned");
  std::vector<Range> outs;
  add_range(outs, a->master, n * 4, "master", 0);
  add_range(outs, a->m, n * mbytes, "m", 0);
  add_range(outs, a->v, n * mbytes, "v", 0);
  for (int q = 0; q < P; ++q) {
    if (!a->grads[q] || !a->grad_scales[q] || !a->replicas[q] || !a->replica_scales[q])
      return fail(ZDP_ERR_INVALID, "a rank-%d pointer is NULL", q);
    if (!aligned16(a->grads[q]) || !aligned16(a->replicas[q]))
      return fail(ZDP_ERR_INVALID, "grads[%d] and replicas[%d] must be 16-byte aligned", q, q);
    if ((addr(a->grad_scales[q]) & 3u) != 0 || (addr(a->replica_scales[q]) & 3u) != 0)
      return fail(ZDP_ERR_INVALID, "scales of rank %d not 4-byte aligned", q);
    add_range(outs, a->replicas[q], n, "replicas", q);
    add_range(outs, a->replica_scales[q], nb * 4, "replica_scales", q);
  }
  add_range(outs, a->d_overflow, 4, "d_overflow", 0);
  add_range(outs, a->d_sumsq, 8, "d_sumsq", 0);
  if (check_disjoint(outs) != ZDP_OK) return ZDP_ERR_INVALID;
  for (int q = 0; q < P; ++q) {
    const Range ins[2] = {{addr(a->grads[q]), addr(a->grads[q]) + static_cast<uintptr_t>(len), "grads", q},
                          {addr(a->grad_scales[q]),
                           addr(a->grad_scales[q]) + static_cast<uintptr_t>(lb * 4), "grad_scales", q}};
    for (const Range& in : ins)
      for (const Range& o : outs)
        if (in.lo < o.hi && o.lo < in.hi)
          return fail(ZDP_ERR_INVALID, "buffers overlap: %s[%d] and %s[%d]", in.what, q, o.what,
                      o.index);
  }
  int sms = 0;
  if (num_sms(&sms) != ZDP_OK) return ZDP_ERR_CUDA;
  const zdp::AdamK ad = make_adam(a->lr, a->b1, a->b2, a->eps, a->wd, a->t);
  cudaError_t e = zdp::launch_zpp(a, ad, sms, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "ZeRO++ step launch");
  return ok();
}

}  // extern "C"
