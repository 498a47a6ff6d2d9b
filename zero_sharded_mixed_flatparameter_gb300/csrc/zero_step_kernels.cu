// sm_103a kernels of the fused ZeRO flat-parameter optimizer step.
//
// The step is a pure HBM stream: per element it reads N replica gradients
// (bf16 or fp32), the fp32 master, m and v, and writes master, m, v and the
// bf16 parameter — (2N + 26) bytes per element for bf16 gradients, with about
// N + 15 flops.  Nothing is a contraction, so there are no tensor cores here;
// what matters is coalesced 16-byte accesses, enough bytes in flight per SM
// and a grid that fills all SMs.  Each thread handles 8 consecutive elements
// per iteration (one 16-byte load per bf16 replica, two per fp32 array).
//
// Arithmetic follows the Adam update of the CMU 15-779 Lecture 13 notes §2.1
// with the fixed rank-order fp32 reduction of §3.4; every operation is an
// explicitly rounded IEEE fp32 intrinsic (no FMA contraction; IEEE division
// and square root), so the result is reproducible bit for bit.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "zero_device.cuh"
#include "zero_internal.h"

namespace zfs {
namespace {

// Adam / AdamW on one element (decay == 1 exactly for plain Adam).
__device__ __forceinline__ void adam(const StepArgs& a, float g, float& w, float& m, float& v) {
  w = __fmul_rn(w, a.decay);
  m = __fadd_rn(__fmul_rn(a.beta1, m), __fmul_rn(a.omb1, g));
  v = __fadd_rn(__fmul_rn(a.beta2, v), __fmul_rn(a.omb2, __fmul_rn(g, g)));
  const float m_hat = __fdiv_rn(m, a.bc1);
  const float v_hat = __fdiv_rn(v, a.bc2);
  const float denom = __fadd_rn(__fsqrt_rn(v_hat), a.eps);
  w = __fsub_rn(w, __fmul_rn(a.lr, __fdiv_rn(m_hat, denom)));
}

// Reduced gradient of one element k of segment s, any N, any alignment.
__device__ __forceinline__ float reduce_scalar(const StepArgs& a, const Seg& s, long long k) {
  float acc;
  if (a.grad_fp32) {
    acc = __ldcs(static_cast<const float*>(s.g[0]) + k);
    for (int r = 1; r < a.n_ranks; ++r) acc = __fadd_rn(acc, __ldcs(static_cast<const float*>(s.g[r]) + k));
  } else {
    acc = __uint_as_float(static_cast<uint32_t>(__ldcs(static_cast<const unsigned short*>(s.g[0]) + k)) << 16);
    for (int r = 1; r < a.n_ranks; ++r) {
      const uint32_t h = __ldcs(static_cast<const unsigned short*>(s.g[r]) + k);
      acc = __fadd_rn(acc, __uint_as_float(h << 16));
    }
  }
  return __fmul_rn(acc, a.inv_n);
}

__device__ __forceinline__ void step_scalar_element(const StepArgs& a, const Seg& s, long long k, float clip) {
  const long long j = s.base + k;
  const float g = __fmul_rn(reduce_scalar(a, s, k), clip);
  float w = a.master[j], m = a.m[j], v = a.v[j];
  adam(a, g, w, m, v);
  a.master[j] = w;
  a.m[j] = m;
  a.v[j] = v;
  a.p16[j] = to_bf16_bits(w);
}

// ---------------------------------------------------------------------------
// Vector kernel: 8 elements per thread-iteration.
// ---------------------------------------------------------------------------
template <int N, bool kFp32>
__device__ __forceinline__ void step_vec8(const StepArgs& a, const Seg& s, long long vi, float clip) {
  const long long j = s.base + vi * kVec;
  float g[kVec];
  if constexpr (!kFp32) {
    uint4 raw[N];
#pragma unroll
    for (int r = 0; r < N; ++r) raw[r] = ld_stream(static_cast<const uint4*>(s.g[r]) + vi);
    g[0] = bf16_lo(raw[0].x); g[1] = bf16_hi(raw[0].x);
    g[2] = bf16_lo(raw[0].y); g[3] = bf16_hi(raw[0].y);
    g[4] = bf16_lo(raw[0].z); g[5] = bf16_hi(raw[0].z);
    g[6] = bf16_lo(raw[0].w); g[7] = bf16_hi(raw[0].w);
#pragma unroll
    for (int r = 1; r < N; ++r) {
      g[0] = __fadd_rn(g[0], bf16_lo(raw[r].x)); g[1] = __fadd_rn(g[1], bf16_hi(raw[r].x));
      g[2] = __fadd_rn(g[2], bf16_lo(raw[r].y)); g[3] = __fadd_rn(g[3], bf16_hi(raw[r].y));
      g[4] = __fadd_rn(g[4], bf16_lo(raw[r].z)); g[5] = __fadd_rn(g[5], bf16_hi(raw[r].z));
      g[6] = __fadd_rn(g[6], bf16_lo(raw[r].w)); g[7] = __fadd_rn(g[7], bf16_hi(raw[r].w));
    }
  } else {
    float4 raw[N][2];
#pragma unroll
    for (int r = 0; r < N; ++r) {
      const float* base = static_cast<const float*>(s.g[r]) + vi * kVec;
      raw[r][0] = ld_stream_f4(base);
      raw[r][1] = ld_stream_f4(base + 4);
    }
    g[0] = raw[0][0].x; g[1] = raw[0][0].y; g[2] = raw[0][0].z; g[3] = raw[0][0].w;
    g[4] = raw[0][1].x; g[5] = raw[0][1].y; g[6] = raw[0][1].z; g[7] = raw[0][1].w;
#pragma unroll
    for (int r = 1; r < N; ++r) {
      g[0] = __fadd_rn(g[0], raw[r][0].x); g[1] = __fadd_rn(g[1], raw[r][0].y);
      g[2] = __fadd_rn(g[2], raw[r][0].z); g[3] = __fadd_rn(g[3], raw[r][0].w);
      g[4] = __fadd_rn(g[4], raw[r][1].x); g[5] = __fadd_rn(g[5], raw[r][1].y);
      g[6] = __fadd_rn(g[6], raw[r][1].z); g[7] = __fadd_rn(g[7], raw[r][1].w);
    }
  }
  const float4 w0 = ld_stream_f4(a.master + j), w1 = ld_stream_f4(a.master + j + 4);
  const float4 m0 = ld_stream_f4(a.m + j), m1 = ld_stream_f4(a.m + j + 4);
  const float4 v0 = ld_stream_f4(a.v + j), v1 = ld_stream_f4(a.v + j + 4);
  float w[kVec] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
  float m[kVec] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
  float v[kVec] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
  for (int e = 0; e < kVec; ++e) adam(a, __fmul_rn(__fmul_rn(g[e], a.inv_n), clip), w[e], m[e], v[e]);
  st_stream_f4(a.master + j, make_float4(w[0], w[1], w[2], w[3]));
  st_stream_f4(a.master + j + 4, make_float4(w[4], w[5], w[6], w[7]));
  st_stream_f4(a.m + j, make_float4(m[0], m[1], m[2], m[3]));
  st_stream_f4(a.m + j + 4, make_float4(m[4], m[5], m[6], m[7]));
  st_stream_f4(a.v + j, make_float4(v[0], v[1], v[2], v[3]));
  st_stream_f4(a.v + j + 4, make_float4(v[4], v[5], v[6], v[7]));
  uint4 out;
  out.x = pack_bf16x2(w[0], w[1]);
  out.y = pack_bf16x2(w[2], w[3]);
  out.z = pack_bf16x2(w[4], w[5]);
  out.w = pack_bf16x2(w[6], w[7]);
  st_stream(a.p16 + j, out);
}

// Minimum of one resident CTA in the bounds lets each thread keep all of its
// 16-byte loads in flight before the first use (about 94 registers at N = 8);
// the grid then caps residency at kStepCtasPerSm CTAs per SM (see launch_step_vec).
template <int N, bool kFp32>
__global__ void __launch_bounds__(kStepThreads, 1) step_vec_kernel(const __grid_constant__ StepArgs a) {
  const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  // Clip coefficient of the global norm (x 1 is exact when not clipping).
  const float clip = a.clip ? *a.clip : 1.0f;
  for (int s = 0; s < a.nseg; ++s) {
    const Seg& seg = a.seg[s];
    const long long nvec = seg.len / kVec;
    for (long long vi = first_index(tid, seg.vec_start, stride); vi < nvec; vi += stride) {
      step_vec8<N, kFp32>(a, seg, vi, clip);
    }
  }
  // Ragged ends (fewer than 8 elements per segment), element by element.
  for (int s = 0; s < a.nseg; ++s) {
    const Seg& seg = a.seg[s];
    const long long done = (seg.len / kVec) * kVec;
    const long long k = done + tid - static_cast<long long>(s) * kVec;
    if (tid >= static_cast<long long>(s) * kVec && k < seg.len && k < done + kVec) {
      step_scalar_element(a, seg, k, clip);
    }
  }
}

// ---------------------------------------------------------------------------
// Scalar kernel: one element per thread-iteration, any alignment, any N.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kStepThreads) step_scalar_kernel(const __grid_constant__ StepArgs a) {
  const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  const float clip = a.clip ? *a.clip : 1.0f;
  long long start = 0;
  for (int s = 0; s < a.nseg; ++s) {
    const Seg& seg = a.seg[s];
    for (long long k = first_index(tid, start, stride); k < seg.len; k += stride) {
      step_scalar_element(a, seg, k, clip);
    }
    start += seg.len;
  }
}

// ---------------------------------------------------------------------------
// Launch configuration.
// ---------------------------------------------------------------------------
using StepKernel = void (*)(StepArgs);

template <bool kFp32>
StepKernel vec_kernel_for(int n) {
  switch (n) {
    case 1: return step_vec_kernel<1, kFp32>;
    case 2: return step_vec_kernel<2, kFp32>;
    case 3: return step_vec_kernel<3, kFp32>;
    case 4: return step_vec_kernel<4, kFp32>;
    case 5: return step_vec_kernel<5, kFp32>;
    case 6: return step_vec_kernel<6, kFp32>;
    case 7: return step_vec_kernel<7, kFp32>;
    case 8: return step_vec_kernel<8, kFp32>;
    case 9: return step_vec_kernel<9, kFp32>;
    case 10: return step_vec_kernel<10, kFp32>;
    case 11: return step_vec_kernel<11, kFp32>;
    case 12: return step_vec_kernel<12, kFp32>;
    case 13: return step_vec_kernel<13, kFp32>;
    case 14: return step_vec_kernel<14, kFp32>;
    case 15: return step_vec_kernel<15, kFp32>;
    case 16: return step_vec_kernel<16, kFp32>;
    default: return nullptr;
  }
}

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  int sms = 0;
  int vec_blocks_per_sm[2][kMaxRanks + 1] = {};
  int scalar_blocks_per_sm = 0;
};

std::mutex g_info_mutex;
DeviceInfo g_info[kMaxDevices];

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) dev = 0;
  return dev;
}

int cached_sms(int dev) {
  std::lock_guard<std::mutex> lock(g_info_mutex);
  if (g_info[dev].sms == 0) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = 1;
    g_info[dev].sms = sms;
  }
  return g_info[dev].sms;
}

int resident_blocks(int* slot, const void* kernel) {
  std::lock_guard<std::mutex> lock(g_info_mutex);
  if (*slot == 0) {
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kernel, kStepThreads, 0) != cudaSuccess || b <= 0) b = 1;
    *slot = b;
  }
  return *slot;
}

}  // namespace

long long grid_for(long long work_items, int sms, int blocks_per_sm) {
  const long long full = static_cast<long long>(sms) * blocks_per_sm;
  long long need = (work_items + kStepThreads - 1) / kStepThreads;
  if (need < 1) need = 1;
  return need < full ? need : full;
}


int sm_count() { return cached_sms(current_device()); }

cudaError_t launch_step_vec(const StepArgs& a, cudaStream_t stream) {
  StepKernel k = a.grad_fp32 ? vec_kernel_for<true>(a.n_ranks) : vec_kernel_for<false>(a.n_ranks);
  if (!k) return cudaErrorInvalidValue;
  const int dev = current_device();
  const int sms = cached_sms(dev);
  int bps = resident_blocks(&g_info[dev].vec_blocks_per_sm[a.grad_fp32 ? 1 : 0][a.n_ranks],
                            reinterpret_cast<const void*>(k));
  // 512 resident threads per SM: measured on GB300 to give the best DRAM
  // efficiency across N = 1..16 (more threads widen the address window the
  // grid streams through at once and lower row-buffer locality; fewer leave
  // too few bytes in flight).
  if (bps > kStepCtasPerSm) bps = kStepCtasPerSm;
  long long work = a.total_vec;
  if (work < static_cast<long long>(a.nseg) * kVec) work = static_cast<long long>(a.nseg) * kVec;
  const long long grid = grid_for(work, sms, bps);
  k<<<static_cast<unsigned>(grid), kStepThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_step_scalar(const StepArgs& a, cudaStream_t stream) {
  const int dev = current_device();
  const int sms = cached_sms(dev);
  const int bps = resident_blocks(&g_info[dev].scalar_blocks_per_sm,
                                  reinterpret_cast<const void*>(step_scalar_kernel));
  const long long grid = grid_for(a.total_elems, sms, bps);
  step_scalar_kernel<<<static_cast<unsigned>(grid), kStepThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace zfs
