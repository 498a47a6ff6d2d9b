// Gradient clipping for callers that cannot allocate device memory.
//
// zero_clip_grad_norm needs a caller-provided device workspace.  Some callers
// cannot provide one: code that runs where the allocator must not be entered
// (inside a custom allocator or an out-of-memory handler, a real-time loop
// that forbids allocation, an embedding that has no allocation API of its own
// to offer).  zero_clip_grad_norm_static gives them the same computation with
// its scratch in a fixed array that lives in the library's own device memory:
// the array below, kStaticClipBytes long, is created on every GPU that loads
// the library and held until the process exits.  The call allocates nothing.
//
// The array is shared by every call on a device and keeps the last call's
// contents.  Nothing in it has to start at zero: each call writes every chunk
// partial it later reads, and writes the norm and coefficient itself.  Calls
// whose device work can overlap (different streams, different contexts) race
// on it; the coefficient one call leaves there is read by that context's next
// zero_step, so no other static-scratch clip may run between the two unless
// all of them are ordered on one stream.

#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "zero_flatstep.h"
#include "zero_internal.h"

namespace {

// 1 MiB: the 32-byte header plus 131,068 chunk partials of 16,384 elements,
// i.e. layouts of up to about 2.1 billion padded elements.
constexpr long long kStaticClipBytes = 1LL << 20;

static __device__ __align__(256) unsigned char g_clip_scratch[kStaticClipBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_address[kMaxDevices] = {};

}  // namespace

extern "C" zero_status zero_clip_grad_norm_static(zero_ctx* ctx, float max_norm, void* stream) {
  if (!ctx) return static_cast<zero_status>(zfs_report_error(nullptr, ZERO_EINVAL, "ctx is NULL"));
  int64_t need = 0;
  zero_status st = zero_clip_workspace_bytes(ctx, &need);
  if (st != ZERO_OK) return st;
  if (need > kStaticClipBytes) {
    char msg[256];
    std::snprintf(msg, sizeof msg,
                  "layout needs %lld bytes of clip scratch; the static scratch holds %lld "
                  "(about 2.1e9 padded elements): use zero_clip_grad_norm with a workspace",
                  static_cast<long long>(need), kStaticClipBytes);
    return static_cast<zero_status>(zfs_report_error(ctx, ZERO_EINVAL, msg));
  }
  int device = -1;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess || device < 0 || device >= kMaxDevices) {
    return static_cast<zero_status>(zfs_report_error(ctx, ZERO_ECUDA, "cannot query the current device"));
  }
  void* scratch = nullptr;
  {
    // Set-up, once per device, with that device current: in host code the
    // array's name only stands in for the device object, so its device
    // address is looked up here and passed to the kernels.
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_address[device]) {
      void* address = nullptr;
      e = cudaGetSymbolAddress(&address, g_clip_scratch);
      if (e != cudaSuccess || !address) {
        char msg[256];
        std::snprintf(msg, sizeof msg, "cudaGetSymbolAddress of the static clip scratch failed: %s",
                      cudaGetErrorString(e));
        return static_cast<zero_status>(zfs_report_error(ctx, ZERO_ECUDA, msg));
      }
      g_scratch_address[device] = address;
    }
    scratch = g_scratch_address[device];
  }
  return zero_clip_grad_norm(ctx, max_norm, scratch, kStaticClipBytes, stream);
}
