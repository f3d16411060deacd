// zdp_noalloc.cu -- zdp_step_noalloc: the overflow-checked step with its
// scratch in a static device array instead of a caller-provided workspace,
// for callers that cannot allocate device memory.
//
// The scratch has exactly the layout zdp_step_workspace_bytes() describes: a
// 256-byte slot whose first 8 bytes hold the device overflow flag (and, for
// the single cooperative launch, the grid barrier's arrival counter), then,
// for the two-pass form, the reduced gradients of the call's range (len + 8
// fp32 values, starting at the multiple of 8 at or below `off`).  The array
// is sized for ZDP_NOALLOC_MAX_LEN elements.
#include <cuda.h>

#include <cstdio>
#include <mutex>

#include "zdp_internal.h"

namespace {

constexpr size_t kScratchBytes =
    256 + ((static_cast<size_t>(ZDP_NOALLOC_MAX_LEN) + 8) * 4 + 255) / 256 * 256;

// Lives in the memory of every GPU on which this library's module is loaded,
// until the process exits.  In host code the name is only a stand-in for the
// symbol, never a device address: the address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// The context handle and its process-unique id come from the driver API,
// reached through the runtime's entry-point query so that the library does
// not link the driver library directly.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

struct DriverEntryPoints {
  CtxGetCurrentFn get_current = nullptr;
  CtxGetIdFn get_id = nullptr;
};

const DriverEntryPoints& driver_entry_points() {
  static const DriverEntryPoints eps = [] {
    DriverEntryPoints d;
    auto query = [](const char* name) -> void* {
      void* f = nullptr;
      cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
      const cudaError_t e = cudaGetDriverEntryPointByVersion(name, &f, 12000, cudaEnableDefault, &q);
      if (e != cudaSuccess) {
        cudaGetLastError();  // clear this query's own (non-sticky) error, nothing older
        return nullptr;
      }
      return q == cudaDriverEntryPointSuccess ? f : nullptr;
    };
    d.get_current = reinterpret_cast<CtxGetCurrentFn>(query("cuCtxGetCurrent"));
    d.get_id = reinterpret_cast<CtxGetIdFn>(query("cuCtxGetId"));
    return d;
  }();
  return eps;
}

// Process-unique id of the calling thread's current CUDA context; 0 when no
// context is current yet or the driver cannot tell.  Context handles can be
// reused after a context is destroyed; these ids are never reused.
unsigned long long current_context_id() {
  const DriverEntryPoints& d = driver_entry_points();
  if (!d.get_current || !d.get_id) return 0;
  CUcontext ctx = nullptr;
  if (d.get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  unsigned long long id = 0;
  if (d.get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

int lookup_failed(cudaError_t e) {
  // The failed lookup's error is reported here; clear it from the runtime so
  // that a later call's launch check does not take it for its own.
  if (e != cudaSuccess) cudaGetLastError();
  char msg[200];
  std::snprintf(msg, sizeof msg, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
  return zdp::report_error(ZDP_ERR_CUDA, msg);
}

// Device address of the scratch in the current context.  Each context that
// loads this library's module (normally the primary context of a device)
// holds its own instance of the array, so the address is looked up with
// cudaGetSymbolAddress once per context, with that context current, and
// cached under the context's unique id.  A context created later on the same
// device, after cudaDeviceReset or as a separate (e.g. green) context, gets
// its own lookup instead of a stale address.  The first lookup in a context
// may load the library's module there.
int scratch_address(void** out) {
  constexpr int kSlots = 64;
  static std::mutex mu;
  static unsigned long long ids[kSlots] = {0};
  static void* addrs[kSlots] = {nullptr};
  static int next = 0;

  unsigned long long id = current_context_id();
  void* p = nullptr;
  if (id == 0) {
    // No context is current on this thread yet: the lookup binds the current
    // device's primary context, whose id can then be read.
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) return lookup_failed(e);
    id = current_context_id();
    if (id == 0) {  // the driver does not report context ids: no caching
      *out = p;
      return ZDP_OK;
    }
  }
  std::lock_guard<std::mutex> lock(mu);
  for (int k = 0; k < kSlots; ++k) {
    if (ids[k] == id) {
      *out = addrs[k];
      return ZDP_OK;
    }
  }
  if (p == nullptr) {
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) return lookup_failed(e);
  }
  ids[next] = id;
  addrs[next] = p;
  next = (next + 1) % kSlots;
  *out = p;
  return ZDP_OK;
}

}  // namespace

extern "C" int zdp_step_noalloc(const zdp_step_args* args, void* stream) {
  if (!args) return zdp::report_error(ZDP_ERR_INVALID, "args is NULL");
  if (args->len > ZDP_NOALLOC_MAX_LEN) {
    char msg[200];
    std::snprintf(msg, sizeof msg,
                  "len=%lld exceeds ZDP_NOALLOC_MAX_LEN=%lld, the size of the static scratch; "
                  "split the range into several calls or use zdp_step with a workspace",
                  static_cast<long long>(args->len), static_cast<long long>(ZDP_NOALLOC_MAX_LEN));
    return zdp::report_error(ZDP_ERR_INVALID, msg);
  }
  void* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != ZDP_OK) return rc;
  zdp_step_args a = *args;
  a.check_overflow = 1;
  a.workspace = scratch;
  a.workspace_bytes = kScratchBytes;
  return zdp_step(&a, stream);
}
