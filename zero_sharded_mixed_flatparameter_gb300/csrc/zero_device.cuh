// Device helpers shared by the step kernels and the auxiliary kernels of the
// ZeRO flat-parameter library: bf16 bit conversions, streaming (evict-first)
// 16-byte accesses and the grid-stride start index.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace zfs {

// Debug builds (-DZFS_DEBUG_CHECKS) check every index before the access it
// guards: a failed check counts in this file's counter and the access is
// skipped (no trap, no out-of-range access).  Release builds compile the
// checks away.
#ifdef ZFS_DEBUG_CHECKS
static __device__ unsigned int g_debug_failures = 0;
__device__ __forceinline__ bool debug_check(bool ok) {
  if (!ok) atomicAdd(&g_debug_failures, 1u);
  return ok;
}
#define ZFS_CHECK(cond) (::zfs::debug_check(static_cast<bool>(cond)))
#else
#define ZFS_CHECK(cond) true
#endif

__device__ __forceinline__ float bf16_lo(uint32_t word) { return __uint_as_float(word << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t word) { return __uint_as_float(word & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);  // .x = lo (low half), .y = hi
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint16_t to_bf16_bits(float x) {
  __nv_bfloat16 h = __float2bfloat16_rn(x);
  return *reinterpret_cast<uint16_t*>(&h);
}

// Streaming (evict-first) global accesses: every byte is touched once per step.
__device__ __forceinline__ uint4 ld_stream(const void* p) { return __ldcs(reinterpret_cast<const uint4*>(p)); }
__device__ __forceinline__ float4 ld_stream_f4(const float* p) { return __ldcs(reinterpret_cast<const float4*>(p)); }
__device__ __forceinline__ void st_stream_f4(float* p, float4 x) { __stcs(reinterpret_cast<float4*>(p), x); }
__device__ __forceinline__ void st_stream(void* p, uint4 x) { __stcs(reinterpret_cast<uint4*>(p), x); }

// How many of kN reduced gradients are inf or NaN (the step's overflow
// count): one comparison and one add per value, no branch, so that the
// kernels' loads are not held behind it; the sum reaches the caller's counter
// only when counting is on (flush_nonfinite).
template <int kN>
__device__ __forceinline__ unsigned tally_nonfinite(const float* g) {
  unsigned c = 0;
#pragma unroll
  for (int e = 0; e < kN; ++e) c += (fabsf(g[e]) <= 0x1.fffffep127f) ? 0u : 1u;
  return c;
}

// Adds a thread's overflow count to the caller's counter (none when zero).
__device__ __forceinline__ void flush_nonfinite(unsigned long long* counter, unsigned count) {
  if (count != 0u && counter != nullptr) atomicAdd(counter, static_cast<unsigned long long>(count));
}

// First index >= 0 congruent to (tid - start) modulo stride: walking a
// segment from there in steps of `stride` makes the launch's grid-stride
// loop run over all segments as one concatenated index space.
__device__ __forceinline__ long long first_index(long long tid, long long start, long long stride) {
  long long r = (tid - start) % stride;
  return r < 0 ? r + stride : r;
}

}  // namespace zfs
