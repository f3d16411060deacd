// zdp_noalloc.cu -- zdp_step_noalloc: the overflow-checked two-pass step with
// its scratch in a static device array instead of a caller-provided
// workspace, for callers that cannot allocate device memory.
//
// The scratch holds what the two passes exchange: a 256-byte slot for the
// device overflow flag, then the reduced gradients of the call's range
// (len + 8 fp32 values, starting at the multiple of 8 at or below `off`),
// exactly the layout zdp_step_workspace_bytes() describes.  The array is
// sized for ZDP_NOALLOC_MAX_LEN elements.
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

constexpr int kMaxDevices = 256;

// Device address of the scratch on the current device.  Looked up once per
// device, with that device current, and cached; the first lookup on a device
// may load the library's module there.
int scratch_address(void** out) {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {nullptr};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    char msg[200];
    std::snprintf(msg, sizeof msg, "cudaGetDevice: %s", cudaGetErrorString(e));
    return zdp::report_error(ZDP_ERR_CUDA, msg);
  }
  if (dev < 0 || dev >= kMaxDevices)
    return zdp::report_error(ZDP_ERR_CUDA, "device ordinal outside the scratch table");
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      char msg[200];
      std::snprintf(msg, sizeof msg, "cudaGetSymbolAddress(scratch): %s",
                    cudaGetErrorString(e));
      return zdp::report_error(ZDP_ERR_CUDA, msg);
    }
    addr[dev] = p;
  }
  *out = addr[dev];
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
