// Gradient clipping for callers that cannot allocate device memory.
//
// zero_clip_grad_norm needs a caller-provided device workspace.  Some callers
// cannot provide one: code that runs where the allocator must not be entered
// (inside a custom allocator or an out-of-memory handler, a real-time loop
// that forbids allocation, an embedding that has no allocation API of its own
// to offer).  zero_clip_grad_norm_static gives them the same computation with
// its scratch in a fixed array that lives in the library's own device memory:
// the array below, kStaticClipBytes long, is created in every CUDA context
// that loads the library's device code and held until that context ends.
// The call allocates nothing.
//
// The array is shared by every call in a context and keeps the last call's
// contents.  Nothing in it has to start at zero: each call writes every chunk
// partial it later reads, and writes the norm and coefficient itself.  Calls
// whose device work can overlap (different streams) race on it; the
// coefficient one call leaves there is read by that zero_ctx's next
// zero_step, so no other static-scratch clip may run between the two unless
// all of them are ordered on one stream.
//
// Each CUDA context has its own copy of a __device__ array, at its own
// address.  The address is therefore looked up once per context — keyed on
// the context's unique id, which the driver never reuses within a process —
// and not once per device ordinal: a non-primary context, or the primary
// context created again after cudaDeviceReset, gets its own lookup.

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

// Addresses of the array in the contexts seen so far (a small ring: an
// evicted context is simply looked up again).
constexpr int kCachedContexts = 64;
struct CachedAddress {
  unsigned long long ctx_id;
  void* address;
};
std::mutex g_mutex;
CachedAddress g_cache[kCachedContexts] = {};
int g_cache_next = 0;

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
  if (cudaGetDevice(&device) != cudaSuccess || device < 0) {
    return static_cast<zero_status>(zfs_report_error(ctx, ZERO_ECUDA, "cannot query the current device"));
  }
  void* scratch = nullptr;
  unsigned long long ctx_id = 0;
  bool have_id = zfs::current_context_id(&ctx_id);
  std::lock_guard<std::mutex> lock(g_mutex);
  if (have_id) {
    for (const CachedAddress& c : g_cache) {
      if (c.address && c.ctx_id == ctx_id) {
        scratch = c.address;
        break;
      }
    }
  }
  if (!scratch) {
    // Set-up, once per context, with the caller's device current: in host
    // code the array's name only stands in for the device object, so its
    // device address is looked up here and passed to the kernels.  The first
    // lookup in a context may load the library's device code into it.
    void* address = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&address, g_clip_scratch);
    if (e != cudaSuccess || !address) {
      char msg[256];
      std::snprintf(msg, sizeof msg, "cudaGetSymbolAddress of the static clip scratch failed: %s",
                    cudaGetErrorString(e));
      return static_cast<zero_status>(zfs_report_error(ctx, ZERO_ECUDA, msg));
    }
    cudaPointerAttributes attr{};
    e = cudaPointerGetAttributes(&attr, address);
    if (e != cudaSuccess || attr.type != cudaMemoryTypeDevice || attr.device != device) {
      return static_cast<zero_status>(zfs_report_error(
          ctx, ZERO_ECUDA, "the static clip scratch is not device memory of the current device"));
    }
    scratch = address;
    if (!have_id) have_id = zfs::current_context_id(&ctx_id);  // the lookup may have made the context current
    if (have_id) {
      g_cache[g_cache_next] = CachedAddress{ctx_id, address};
      g_cache_next = (g_cache_next + 1) % kCachedContexts;
    }
  }
  return zero_clip_grad_norm(ctx, max_norm, scratch, kStaticClipBytes, stream);
}
