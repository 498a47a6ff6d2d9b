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
__device__ __forceinline__ void adam(const StepArgs& a, float bc1, float bc2, float g, float& w, float& m,
                                     float& v) {
  w = __fmul_rn(w, a.decay);
  m = __fadd_rn(__fmul_rn(a.beta1, m), __fmul_rn(a.omb1, g));
  v = __fadd_rn(__fmul_rn(a.beta2, v), __fmul_rn(a.omb2, __fmul_rn(g, g)));
  const float m_hat = __fdiv_rn(m, bc1);
  const float v_hat = __fdiv_rn(v, bc2);
  const float denom = __fadd_rn(__fsqrt_rn(v_hat), a.eps);
  w = __fsub_rn(w, __fmul_rn(a.lr, __fdiv_rn(m_hat, denom)));
}

// The bias corrections of this step.  kDevBias (capturable steps): the step
// count lives on the device and the host's table holds bc1, bc2 for every t
// up to dev_steps; a count past the table gives false (the step is skipped,
// the table is never read out of range).  Otherwise the launch carries them.
template <bool kDevBias>
__device__ __forceinline__ bool step_bias(const StepArgs& a, float* bc1, float* bc2) {
  if constexpr (kDevBias) {
    const long long t = *a.dev_t + 1;
    if (t < 1 || t > a.dev_steps) return false;
    *bc1 = a.dev_bias[2 * (t - 1)];
    *bc2 = a.dev_bias[2 * (t - 1) + 1];
  } else {
    *bc1 = a.bc1;
    *bc2 = a.bc2;
  }
  return true;
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

__device__ __forceinline__ void step_scalar_element(const StepArgs& a, const Seg& s, long long k, float clip,
                                                    float bc1, float bc2, unsigned& nf) {
  const long long j = s.base + k;
  if (!ZFS_CHECK(k >= 0 && k < s.len && j < a.total_padded)) return;
  const float r = reduce_scalar(a, s, k);
  nf += tally_nonfinite<1>(&r);
  const float g = __fmul_rn(r, clip);
  float w = a.master[j], m = a.m[j], v = a.v[j];
  adam(a, bc1, bc2, g, w, m, v);
  a.master[j] = w;
  a.m[j] = m;
  a.v[j] = v;
  a.p16[j] = to_bf16_bits(w);
}

// ---------------------------------------------------------------------------
// Vector kernel: 8 elements per thread-iteration.
// ---------------------------------------------------------------------------
template <int N, bool kFp32>
__device__ __forceinline__ void step_vec8(const StepArgs& a, const Seg& s, long long vi, float clip, float bc1,
                                          float bc2, unsigned& nf) {
  const long long j = s.base + vi * kVec;
  if (!ZFS_CHECK(vi >= 0 && (vi + 1) * kVec <= s.len && j + kVec <= a.total_padded)) return;
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
  nf += tally_nonfinite<kVec>(g);  // the sum is non-finite exactly when g / N is
#pragma unroll
  for (int e = 0; e < kVec; ++e) adam(a, bc1, bc2, __fmul_rn(__fmul_rn(g[e], a.inv_n), clip), w[e], m[e], v[e]);
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
template <int N, bool kFp32, bool kDevBias>
__global__ void __launch_bounds__(kStepThreads, 1) step_vec_kernel(const __grid_constant__ StepArgs a) {
  const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  float bc1, bc2;
  if (!step_bias<kDevBias>(a, &bc1, &bc2)) return;
  // Clip coefficient of the global norm (x 1 is exact when not clipping).
  const float clip = a.clip ? *a.clip : 1.0f;
  unsigned nf = 0;  // non-finite reduced gradients seen by this thread
  for (int s = 0; s < a.nseg; ++s) {
    const Seg& seg = a.seg[s];
    const long long nvec = seg.len / kVec;
    for (long long vi = first_index(tid, seg.vec_start, stride); vi < nvec; vi += stride) {
      step_vec8<N, kFp32>(a, seg, vi, clip, bc1, bc2, nf);
    }
  }
  // Ragged ends (fewer than 8 elements per segment), element by element.
  for (int s = 0; s < a.nseg; ++s) {
    const Seg& seg = a.seg[s];
    const long long done = (seg.len / kVec) * kVec;
    const long long k = done + tid - static_cast<long long>(s) * kVec;
    if (tid >= static_cast<long long>(s) * kVec && k < seg.len && k < done + kVec) {
      step_scalar_element(a, seg, k, clip, bc1, bc2, nf);
    }
  }
  flush_nonfinite(a.nonfinite, nf);
}

// ---------------------------------------------------------------------------
// Staged kernel for many replicas: TMA (1-D bulk copy) of whole tiles.
//
// With N >= 13 bf16 replicas (N = 8 or 9 fp32) the step is
// read-heavy and has 3 + N input streams.  Here one thread per CTA moves each
// kTmaTile-element tile of every input stream into shared memory with one
// cp.async.bulk per stream (4-8 KB contiguous requests), completing on an
// mbarrier; kTmaStages tiles are in flight per CTA.  Measured on GB300 over a
// 100 M-element buffer (GB/s, staged against register-staged): bf16 N = 11
// 6770 / 6645, N = 12 6942 / 6640, N = 13 7059 / 6653, N = 14 7178 / 6645,
// N = 16 7200 / 6618; fp32 N = 8 7164 / 6651, N = 9 7190 / 6634.  At bf16
// N <= 10 (N = 8: 6143 / 6806), fp32 N = 7 and fp32 N >= 10 the
// register-staged kernel is as fast or faster than this kernel (fp32 N = 7,
// N >= 10 and bf16 N = 1..4 have their own staged shapes, step_tma4_kernel,
// and bf16 N = 7..12 the pipelined step_pipe_kernel, faster than this one
// from N = 11 on as well);
// so it does for launches of fewer than kTmaMinElems elements, where one CTA
// per SM works through too few tiles to hide the latency of each (N = 16
// bf16: 2363 / 3152 GB/s at 1 M elements, 5481 / 5479 at 6 M, 6179 / 5962
// at 12 M).
// The arithmetic and its order are those of step_vec8, so the results are
// bit-identical.  Every wait is bounded in time (kTmaWaitNs): a CTA that gives
// up (which needs a copy that never lands) counts it in g_step_timeouts,
// waits (bounded) for the copies it issued and leaves, with the rest of its
// tiles not updated; the host reads the counter with zero_kernel_timeouts.
// The test hook inject_missing_copy makes exactly this happen to the launch's
// first tile (its bytes are announced to the mbarrier, no copy is issued).
// ---------------------------------------------------------------------------
__device__ unsigned int g_step_timeouts = 0;

// Wait limits (device global timer, ns): a tile's copies land within
// microseconds; a second means they never will.  Draining after a give-up
// waits at most kTmaDrainNs per outstanding tile.
constexpr unsigned long long kTmaWaitNs = 1000000000ull;
constexpr unsigned long long kTmaDrainNs = 50000000ull;
constexpr int kTmaFastSpins = 64;  // try_wait attempts before the timed wait starts

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}
// The rest of a tile's wait after a first try_wait failed: a short spin
// (tiles usually land within a few tries), then tries until kTmaWaitNs have
// passed.  False: the copies never landed.  Out of line so that the rarely
// long wait does not weigh on the register allocation of the tile loop.
__device__ __noinline__ bool wait_tile(uint64_t* bar, uint32_t parity) {
  for (int i = 0; i < kTmaFastSpins; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
  }
  const unsigned long long t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() - t0 > kTmaWaitNs) return false;
  }
  return true;
}

// Global -> this CTA's shared memory; completes `bytes` on the mbarrier.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

template <int N, bool kFp32>
struct TmaTile {
  static constexpr uint32_t kGradBytes = kTmaTile * (kFp32 ? 4 : 2);
  static constexpr uint32_t kStateBytes = kTmaTile * 4;
  static constexpr uint32_t kStageBytes = N * kGradBytes + 3 * kStateBytes;
  static constexpr uint32_t kSmemBytes = kStageBytes * kTmaStages;
};

// Full tiles of a launch, segment after segment: tile id -> (segment, tile).
__device__ __forceinline__ void locate_tile(const StepArgs& a, long long id, int* si, long long* ti) {
  int s = 0;
  while (id >= a.seg[s].len / kTmaTile) {
    id -= a.seg[s].len / kTmaTile;
    ++s;
  }
  *si = s;
  *ti = id;
}

template <int N, bool kFp32, bool kDevBias>
__global__ void __launch_bounds__(kStepThreads, 1) step_tma_kernel(const __grid_constant__ StepArgs a) {
  float bc1, bc2;
  if (!step_bias<kDevBias>(a, &bc1, &bc2)) return;  // before any barrier or copy
  using L = TmaTile<N, kFp32>;
  static_assert(kTmaTile == kStepThreads * kVec, "8 elements per thread per tile");
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ __align__(8) uint64_t bars[kTmaStages];
  long long n_tiles = 0;
  for (int s = 0; s < a.nseg; ++s) n_tiles += a.seg[s].len / kTmaTile;
  const float clip = a.clip ? *a.clip : 1.0f;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kTmaStages; ++s) mbar_init(&bars[s], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  auto issue = [&](long long id, int stage) {  // thread 0 only
    int si;
    long long ti;
    locate_tile(a, id, &si, &ti);
    const Seg& sg = a.seg[si];
    unsigned char* st = smem + static_cast<size_t>(stage) * L::kStageBytes;
    const long long e0 = ti * kTmaTile;
    if (!ZFS_CHECK(ti >= 0 && e0 + kTmaTile <= sg.len && sg.base + e0 + kTmaTile <= a.total_padded)) {
      // complete the stage's phase without bytes: its stores are skipped below
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&bars[stage])) : "memory");
      return;
    }
    mbar_expect_tx(&bars[stage], L::kStageBytes);
    if (a.inject_missing_copy && id == 0) return;  // test hook: this tile's wait must run out
    for (int r = 0; r < N; ++r)
      bulk_load(st + r * L::kGradBytes, static_cast<const char*>(sg.g[r]) + e0 * (kFp32 ? 4 : 2), L::kGradBytes,
                &bars[stage]);
    const long long j0 = sg.base + e0;
    bulk_load(st + N * L::kGradBytes, a.master + j0, L::kStateBytes, &bars[stage]);
    bulk_load(st + N * L::kGradBytes + L::kStateBytes, a.m + j0, L::kStateBytes, &bars[stage]);
    bulk_load(st + N * L::kGradBytes + 2 * L::kStateBytes, a.v + j0, L::kStateBytes, &bars[stage]);
  };
  if (threadIdx.x == 0) {
    for (int i = 0; i < kTmaStages; ++i) {
      const long long id = blockIdx.x + static_cast<long long>(i) * gridDim.x;
      if (id < n_tiles) issue(id, i);
    }
  }
  long long gave_up_at = -1;  // the tile whose wait ran out, if any
  unsigned nf = 0;            // non-finite reduced gradients seen by this thread
  for (long long k = 0;; ++k) {
    const long long id = blockIdx.x + k * gridDim.x;
    if (id >= n_tiles) break;
    const int stage = static_cast<int>(k % kTmaStages);
    const uint32_t parity = static_cast<uint32_t>((k / kTmaStages) & 1);
    const bool mine = !mbar_try_wait(&bars[stage], parity) && !wait_tile(&bars[stage], parity);
    // Every thread reaches this barrier; the CTA gives up together or not at all.
    if (__syncthreads_or(mine ? 1 : 0)) {
      gave_up_at = k;
      if (threadIdx.x == 0) atomicAdd(&g_step_timeouts, 1u);
      break;
    }
    // Which 8 elements of the tile a thread takes.  bf16 gradients: 4t..4t+3
    // of each half of the tile, so every warp reads contiguous 256-512 B runs
    // of shared memory (no bank conflicts; measured +0.4-2.7 % at N = 14-16).
    // fp32 gradients: 8t..8t+7 with the loads and stores below in this
    // order, which measured 7-10 % faster at N = 8, 9 than the split mapping
    // and 4-7 % faster than this mapping with the two halves' stores
    // interleaved.  The arithmetic per element is the same either way.
    const unsigned char* st = smem + static_cast<size_t>(stage) * L::kStageBytes;
    constexpr int kHalf = kTmaTile / 2;
    const int e_lo = kFp32 ? threadIdx.x * kVec : threadIdx.x * 4;      // elements e_lo .. e_lo + 3
    const int e_hi = kFp32 ? threadIdx.x * kVec + 4 : kHalf + threadIdx.x * 4;  // and e_hi .. e_hi + 3
    float g[kVec];
    if constexpr (!kFp32) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int e0 = h ? e_hi : e_lo;
        float* gh = g + 4 * h;
        const uint2 r0 = *reinterpret_cast<const uint2*>(st + e0 * 2);
        gh[0] = bf16_lo(r0.x); gh[1] = bf16_hi(r0.x); gh[2] = bf16_lo(r0.y); gh[3] = bf16_hi(r0.y);
#pragma unroll
        for (int r = 1; r < N; ++r) {
          const uint2 x = *reinterpret_cast<const uint2*>(st + r * L::kGradBytes + e0 * 2);
          gh[0] = __fadd_rn(gh[0], bf16_lo(x.x)); gh[1] = __fadd_rn(gh[1], bf16_hi(x.x));
          gh[2] = __fadd_rn(gh[2], bf16_lo(x.y)); gh[3] = __fadd_rn(gh[3], bf16_hi(x.y));
        }
      }
    } else {
      const float* g0 = reinterpret_cast<const float*>(st) + e_lo;
#pragma unroll
      for (int e = 0; e < kVec; ++e) g[e] = g0[e];
#pragma unroll
      for (int r = 1; r < N; ++r) {
        const float* gr = reinterpret_cast<const float*>(st + r * L::kGradBytes) + e_lo;
        const float4 x0 = *reinterpret_cast<const float4*>(gr), x1 = *reinterpret_cast<const float4*>(gr + 4);
        g[0] = __fadd_rn(g[0], x0.x); g[1] = __fadd_rn(g[1], x0.y); g[2] = __fadd_rn(g[2], x0.z);
        g[3] = __fadd_rn(g[3], x0.w); g[4] = __fadd_rn(g[4], x1.x); g[5] = __fadd_rn(g[5], x1.y);
        g[6] = __fadd_rn(g[6], x1.z); g[7] = __fadd_rn(g[7], x1.w);
      }
    }
    const float* sw = reinterpret_cast<const float*>(st + N * L::kGradBytes);
    const float* sm = reinterpret_cast<const float*>(st + N * L::kGradBytes + L::kStateBytes);
    const float* sv = reinterpret_cast<const float*>(st + N * L::kGradBytes + 2 * L::kStateBytes);
    float w[kVec], m[kVec], v[kVec];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int e0 = h ? e_hi : e_lo;
      *reinterpret_cast<float4*>(w + 4 * h) = *reinterpret_cast<const float4*>(sw + e0);
      *reinterpret_cast<float4*>(m + 4 * h) = *reinterpret_cast<const float4*>(sm + e0);
      *reinterpret_cast<float4*>(v + 4 * h) = *reinterpret_cast<const float4*>(sv + e0);
    }
    __syncthreads();  // every thread holds its operands: the stage can be refilled
    if (threadIdx.x == 0) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      const long long next = id + static_cast<long long>(kTmaStages) * gridDim.x;
      if (next < n_tiles) issue(next, stage);
    }
    nf += tally_nonfinite<kVec>(g);
#pragma unroll
    for (int e = 0; e < kVec; ++e) adam(a, bc1, bc2, __fmul_rn(__fmul_rn(g[e], a.inv_n), clip), w[e], m[e], v[e]);
    int si;
    long long ti;
    locate_tile(a, id, &si, &ti);
    const long long j_lo = a.seg[si].base + ti * kTmaTile + e_lo;
    const long long j_hi = a.seg[si].base + ti * kTmaTile + e_hi;
    if (!ZFS_CHECK((ti + 1) * kTmaTile <= a.seg[si].len && a.seg[si].base + (ti + 1) * kTmaTile <= a.total_padded)) {
      continue;
    }
    if constexpr (kFp32) {
      st_stream_f4(a.master + j_lo, make_float4(w[0], w[1], w[2], w[3]));
      st_stream_f4(a.master + j_hi, make_float4(w[4], w[5], w[6], w[7]));
      st_stream_f4(a.m + j_lo, make_float4(m[0], m[1], m[2], m[3]));
      st_stream_f4(a.m + j_hi, make_float4(m[4], m[5], m[6], m[7]));
      st_stream_f4(a.v + j_lo, make_float4(v[0], v[1], v[2], v[3]));
      st_stream_f4(a.v + j_hi, make_float4(v[4], v[5], v[6], v[7]));
      uint4 out;
      out.x = pack_bf16x2(w[0], w[1]);
      out.y = pack_bf16x2(w[2], w[3]);
      out.z = pack_bf16x2(w[4], w[5]);
      out.w = pack_bf16x2(w[6], w[7]);
      st_stream(a.p16 + j_lo, out);
    } else {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const long long j = h ? j_hi : j_lo;
        st_stream_f4(a.master + j, make_float4(w[4 * h], w[4 * h + 1], w[4 * h + 2], w[4 * h + 3]));
        st_stream_f4(a.m + j, make_float4(m[4 * h], m[4 * h + 1], m[4 * h + 2], m[4 * h + 3]));
        st_stream_f4(a.v + j, make_float4(v[4 * h], v[4 * h + 1], v[4 * h + 2], v[4 * h + 3]));
        uint2 out;  // 4 contiguous bf16 per half: a warp writes 256 B runs
        out.x = pack_bf16x2(w[4 * h], w[4 * h + 1]);
        out.y = pack_bf16x2(w[4 * h + 2], w[4 * h + 3]);
        __stcs(reinterpret_cast<uint2*>(a.p16 + j), out);
      }
    }
  }
  if (gave_up_at >= 0) {
    // Copies may still be landing in this CTA's shared memory: the tiles
    // issued and not consumed are gave_up_at .. gave_up_at + kTmaStages - 1
    // (those that exist), tile j in stage j % kTmaStages with phase parity
    // (j / kTmaStages) & 1.  Wait for each, bounded, before leaving.
    for (long long j = gave_up_at; j < gave_up_at + kTmaStages; ++j) {
      if (blockIdx.x + j * gridDim.x >= n_tiles) break;
      const int s = static_cast<int>(j % kTmaStages);
      const uint32_t parity = static_cast<uint32_t>((j / kTmaStages) & 1);
      const unsigned long long t0 = global_ns();
      while (!mbar_try_wait(&bars[s], parity) && global_ns() - t0 < kTmaDrainNs) {
      }
    }
    flush_nonfinite(a.nonfinite, nf);
    return;
  }
  // The part of each segment after its last full tile (fewer than kTmaTile
  // elements), element by element.
  const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (int s = 0; s < a.nseg; ++s) {
    const Seg& sg = a.seg[s];
    for (long long k = (sg.len / kTmaTile) * kTmaTile + tid; k < sg.len; k += stride) {
      step_scalar_element(a, sg, k, clip, bc1, bc2, nf);
    }
  }
  flush_nonfinite(a.nonfinite, nf);
}

// ---------------------------------------------------------------------------
// Tile-staged kernel for many fp32 replicas (N = 10..16): tiles of 1,024
// elements, 4 per thread, so that two stages of N + 3 tiles of 4 KB fit one
// CTA's shared memory (2,048-element tiles do not from N = 10 on).  Thread t
// takes elements 4t..4t+3 of a tile: every warp reads contiguous 512-byte
// runs of shared memory.  Waits, give-up, test hook and index checks as in
// step_tma_kernel; the arithmetic per element is step_vec8's.
//
// Measured on GB300 over 400 M elements (step bytes / event time): one CTA
// per SM with three stages at N = 10, 11 (7,135 and 7,151 GB/s; two stages
// 7,076 / 7,123; two CTAs per SM 6,887 / 6,902) and two stages from N = 12
// on (7,133-7,179 GB/s; three stages 6,651-6,949), against 6,800-6,889 GB/s
// for the register-staged kernel at N = 10..16.
// ---------------------------------------------------------------------------
// Tile geometry: kThreads threads x 4 elements per tile, kStages tiles in
// flight per CTA.
template <int N, bool kFp32, int kThreads, int kStages>
struct Tma4Tile {
  static constexpr long long kElems = kThreads * 4;
  static constexpr uint32_t kGradBytes = kElems * (kFp32 ? 4 : 2);
  static constexpr uint32_t kStateBytes = kElems * 4;
  static constexpr uint32_t kStageBytes = N * kGradBytes + 3 * kStateBytes;
  static constexpr uint32_t kSmemBytes = kStageBytes * kStages;
};

// Full kElems-element tiles of a launch, segment after segment.
template <long long kElems>
__device__ __forceinline__ void locate_tile4(const StepArgs& a, long long id, int* si, long long* ti) {
  int s = 0;
  while (id >= a.seg[s].len / kElems) {
    id -= a.seg[s].len / kElems;
    ++s;
  }
  *si = s;
  *ti = id;
}

template <int N, bool kFp32, int kThreads, int kStages, bool kDevBias>
__global__ void __launch_bounds__(kThreads, 1) step_tma4_kernel(const __grid_constant__ StepArgs a) {
  float bc1, bc2;
  if (!step_bias<kDevBias>(a, &bc1, &bc2)) return;  // before any barrier or copy
  using L = Tma4Tile<N, kFp32, kThreads, kStages>;
  constexpr int S = kStages;
  constexpr long long T = L::kElems;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ __align__(8) uint64_t bars[S];
  long long n_tiles = 0;
  for (int s = 0; s < a.nseg; ++s) n_tiles += a.seg[s].len / T;
  const float clip = a.clip ? *a.clip : 1.0f;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  auto issue = [&](long long id, int stage) {  // thread 0 only
    int si;
    long long ti;
    locate_tile4<T>(a, id, &si, &ti);
    const Seg& sg = a.seg[si];
    unsigned char* st = smem + static_cast<size_t>(stage) * L::kStageBytes;
    const long long e0 = ti * T;
    if (!ZFS_CHECK(ti >= 0 && e0 + T <= sg.len && sg.base + e0 + T <= a.total_padded)) {
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&bars[stage])) : "memory");
      return;
    }
    mbar_expect_tx(&bars[stage], L::kStageBytes);
    if (a.inject_missing_copy && id == 0) return;  // test hook: this tile's wait must run out
    for (int r = 0; r < N; ++r)
      bulk_load(st + r * L::kGradBytes, static_cast<const unsigned char*>(sg.g[r]) + e0 * (kFp32 ? 4 : 2),
                L::kGradBytes, &bars[stage]);
    const long long j0 = sg.base + e0;
    unsigned char* st_state = st + N * L::kGradBytes;
    bulk_load(st_state, a.master + j0, L::kStateBytes, &bars[stage]);
    bulk_load(st_state + L::kStateBytes, a.m + j0, L::kStateBytes, &bars[stage]);
    bulk_load(st_state + 2 * L::kStateBytes, a.v + j0, L::kStateBytes, &bars[stage]);
  };
  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      const long long id = blockIdx.x + static_cast<long long>(i) * gridDim.x;
      if (id < n_tiles) issue(id, i);
    }
  }
  long long gave_up_at = -1;
  unsigned nf = 0;  // non-finite reduced gradients seen by this thread
  const int t4 = threadIdx.x * 4;
  for (long long k = 0;; ++k) {
    const long long id = blockIdx.x + k * gridDim.x;
    if (id >= n_tiles) break;
    const int stage = static_cast<int>(k % S);
    const uint32_t parity = static_cast<uint32_t>((k / S) & 1);
    const bool mine = !mbar_try_wait(&bars[stage], parity) && !wait_tile(&bars[stage], parity);
    if (__syncthreads_or(mine ? 1 : 0)) {
      gave_up_at = k;
      if (threadIdx.x == 0) atomicAdd(&g_step_timeouts, 1u);
      break;
    }
    const unsigned char* st = smem + static_cast<size_t>(stage) * L::kStageBytes;
    float gg[4];
    if constexpr (kFp32) {
      const float4 x0 = *reinterpret_cast<const float4*>(st + t4 * 4);
      gg[0] = x0.x; gg[1] = x0.y; gg[2] = x0.z; gg[3] = x0.w;
#pragma unroll
      for (int r = 1; r < N; ++r) {
        const float4 x = *reinterpret_cast<const float4*>(st + r * L::kGradBytes + t4 * 4);
        gg[0] = __fadd_rn(gg[0], x.x); gg[1] = __fadd_rn(gg[1], x.y);
        gg[2] = __fadd_rn(gg[2], x.z); gg[3] = __fadd_rn(gg[3], x.w);
      }
    } else {
      const uint2 x0 = *reinterpret_cast<const uint2*>(st + t4 * 2);
      gg[0] = bf16_lo(x0.x); gg[1] = bf16_hi(x0.x); gg[2] = bf16_lo(x0.y); gg[3] = bf16_hi(x0.y);
#pragma unroll
      for (int r = 1; r < N; ++r) {
        const uint2 x = *reinterpret_cast<const uint2*>(st + r * L::kGradBytes + t4 * 2);
        gg[0] = __fadd_rn(gg[0], bf16_lo(x.x)); gg[1] = __fadd_rn(gg[1], bf16_hi(x.x));
        gg[2] = __fadd_rn(gg[2], bf16_lo(x.y)); gg[3] = __fadd_rn(gg[3], bf16_hi(x.y));
      }
    }
    const unsigned char* st_state = st + N * L::kGradBytes;
    const float4 w4 = *reinterpret_cast<const float4*>(st_state + t4 * 4);
    const float4 m4 = *reinterpret_cast<const float4*>(st_state + L::kStateBytes + t4 * 4);
    const float4 v4 = *reinterpret_cast<const float4*>(st_state + 2 * L::kStateBytes + t4 * 4);
    __syncthreads();  // every thread holds its operands: the stage can be refilled
    if (threadIdx.x == 0) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      const long long next = id + static_cast<long long>(S) * gridDim.x;
      if (next < n_tiles) issue(next, stage);
    }
    float w[4] = {w4.x, w4.y, w4.z, w4.w}, m[4] = {m4.x, m4.y, m4.z, m4.w}, v[4] = {v4.x, v4.y, v4.z, v4.w};
    nf += tally_nonfinite<4>(gg);
#pragma unroll
    for (int e = 0; e < 4; ++e) adam(a, bc1, bc2, __fmul_rn(__fmul_rn(gg[e], a.inv_n), clip), w[e], m[e], v[e]);
    int si;
    long long ti;
    locate_tile4<T>(a, id, &si, &ti);
    if (!ZFS_CHECK((ti + 1) * T <= a.seg[si].len && a.seg[si].base + (ti + 1) * T <= a.total_padded)) {
      continue;
    }
    const long long j = a.seg[si].base + ti * T + t4;
    st_stream_f4(a.master + j, make_float4(w[0], w[1], w[2], w[3]));
    st_stream_f4(a.m + j, make_float4(m[0], m[1], m[2], m[3]));
    st_stream_f4(a.v + j, make_float4(v[0], v[1], v[2], v[3]));
    uint2 out;
    out.x = pack_bf16x2(w[0], w[1]);
    out.y = pack_bf16x2(w[2], w[3]);
    __stcs(reinterpret_cast<uint2*>(a.p16 + j), out);
  }
  if (gave_up_at >= 0) {
    for (long long jj = gave_up_at; jj < gave_up_at + S; ++jj) {
      if (blockIdx.x + jj * gridDim.x >= n_tiles) break;
      const int s = static_cast<int>(jj % S);
      const uint32_t parity = static_cast<uint32_t>((jj / S) & 1);
      const unsigned long long t0 = global_ns();
      while (!mbar_try_wait(&bars[s], parity) && global_ns() - t0 < kTmaDrainNs) {
      }
    }
    flush_nonfinite(a.nonfinite, nf);
    return;
  }
  // The part of each segment after its last full tile, element by element.
  const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (int s = 0; s < a.nseg; ++s) {
    const Seg& sg = a.seg[s];
    for (long long k = (sg.len / T) * T + tid; k < sg.len; k += stride) {
      step_scalar_element(a, sg, k, clip, bc1, bc2, nf);
    }
  }
  flush_nonfinite(a.nonfinite, nf);
}

// ---------------------------------------------------------------------------
// Kernel for segments the aligned kernels cannot take: the segment's flat
// base is not a multiple of 8, or a replica's gradient is not 16-byte aligned
// where the segment's 8-element vectors start.  Padding every unit to a
// multiple of N (CMU 15-779 Lecture 13 notes §3.6) moves later unit bases
// off 8-element boundaries for many layouts and rank counts, and gradients
// that arrive as one buffer per unit are each aligned on their own.
//
// The host peels the segment's first (8 - base % 8) % 8 elements (the head)
// so that the body's master, m, v and bf16 parameters are 16-byte aligned,
// and records per replica how many elements (phi) its gradient sits past a
// 16-byte boundary at the body's start.  A thread takes 8 body elements per
// iteration as step_vec8 does; for a replica with phi != 0 it loads the two
// aligned 16-byte words that hold the vector's elements and funnel-shifts
// them into place.  The second word is also the next lane's first: the
// duplicate request is served on chip, so DRAM traffic is that of the
// aligned kernel (measured against taking the word from the neighbouring
// lane by warp shuffle: level for bf16, +6 % for fp32 gradients at N = 3 —
// the shuffles and the bookkeeping of which lane loads cost more issue slots
// than the extra on-chip request).  The arithmetic and its order are
// step_vec8's, so the results are bit-identical.  Heads and ragged ends (at
// most 7 elements each per segment) go element by element.
// ---------------------------------------------------------------------------

// Elements phi .. phi + 7 of the 16 bf16 in (lo, hi), 0 <= phi < 8.
__device__ __forceinline__ uint4 shift_bf16x8(const uint4& lo, const uint4& hi, int phi) {
  const uint32_t u[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
  const int k = phi >> 1;  // whole 32-bit words
  uint32_t t[6], v[5];
#pragma unroll
  for (int i = 0; i < 6; ++i) t[i] = (k & 2) ? u[i + 2] : u[i];
#pragma unroll
  for (int i = 0; i < 5; ++i) v[i] = (k & 1) ? t[i + 1] : t[i];
  const uint32_t sh = static_cast<uint32_t>(phi & 1) * 16;  // and a half word
  return make_uint4(__funnelshift_r(v[0], v[1], sh), __funnelshift_r(v[1], v[2], sh),
                    __funnelshift_r(v[2], v[3], sh), __funnelshift_r(v[3], v[4], sh));
}

// Elements phi .. phi + 7 of the 12 fp32 in (w0, w1, w2), 0 <= phi < 4.
__device__ __forceinline__ void shift_f32x8(const float4& w0, const float4& w1, const float4& w2, int phi, float* x) {
  const float u[12] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w, w2.x, w2.y, w2.z, w2.w};
  float t[9];
#pragma unroll
  for (int i = 0; i < 9; ++i) t[i] = (phi & 2) ? u[i + 2] : u[i];
#pragma unroll
  for (int i = 0; i < kVec; ++i) x[i] = (phi & 1) ? t[i + 1] : t[i];
}

__device__ __forceinline__ float4 u4_as_f4(const uint4& w) {
  return make_float4(__uint_as_float(w.x), __uint_as_float(w.y), __uint_as_float(w.z), __uint_as_float(w.w));
}

// One iteration of the shifted-gradient kernel: vector vi of segment si (a
// whole vector of the body).  Every load of the iteration — the gradient
// words, master, m, v — is issued before any of them is used, as in
// step_vec8.  The word past the vector is loaded only for phi != 0: its
// first phi elements are the vector's last ones, so it starts inside the
// segment.
template <int N, bool kFp32>
__device__ __forceinline__ void shifted_vec8(const StepArgs& a, const Seg& s, int si, long long vi, float clip,
                                             float bc1, float bc2, unsigned& nf) {
  const long long j = s.base + vi * kVec;
  const bool ok = ZFS_CHECK(vi >= 0 && (vi + 1) * kVec <= s.len && j >= 0 && j + kVec <= a.total_padded);
  constexpr int kWords = kFp32 ? 2 : 1;  // 16-byte words per replica and vector
  uint4 w[N][kWords + 1];
#pragma unroll
  for (int r = 0; r < N; ++r) {
    const int phi = a.gshift[si][r];
    const uint4* base = reinterpret_cast<const uint4*>(static_cast<const char*>(s.g[r]) - phi * (kFp32 ? 4 : 2)) +
                        vi * kWords;
#pragma unroll
    for (int q = 0; q < kWords; ++q) w[r][q] = ok ? ld_stream(base + q) : make_uint4(0u, 0u, 0u, 0u);
    w[r][kWords] = (ok && phi != 0) ? ld_stream(base + kWords) : make_uint4(0u, 0u, 0u, 0u);
  }
  const float4 zero = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  const float4 w0 = ok ? ld_stream_f4(a.master + j) : zero, w1 = ok ? ld_stream_f4(a.master + j + 4) : zero;
  const float4 m0 = ok ? ld_stream_f4(a.m + j) : zero, m1 = ok ? ld_stream_f4(a.m + j + 4) : zero;
  const float4 v0 = ok ? ld_stream_f4(a.v + j) : zero, v1 = ok ? ld_stream_f4(a.v + j + 4) : zero;
  float g[kVec];
#pragma unroll
  for (int r = 0; r < N; ++r) {
    const int phi = a.gshift[si][r];  // uniform over the launch
    float x[kVec];
    if constexpr (!kFp32) {
      const uint4 y = phi != 0 ? shift_bf16x8(w[r][0], w[r][1], phi) : w[r][0];
      x[0] = bf16_lo(y.x); x[1] = bf16_hi(y.x); x[2] = bf16_lo(y.y); x[3] = bf16_hi(y.y);
      x[4] = bf16_lo(y.z); x[5] = bf16_hi(y.z); x[6] = bf16_lo(y.w); x[7] = bf16_hi(y.w);
    } else {
      shift_f32x8(u4_as_f4(w[r][0]), u4_as_f4(w[r][1]), u4_as_f4(w[r][2]), phi, x);
    }
    if (r == 0) {
#pragma unroll
      for (int e = 0; e < kVec; ++e) g[e] = x[e];
    } else {
#pragma unroll
      for (int e = 0; e < kVec; ++e) g[e] = __fadd_rn(g[e], x[e]);
    }
  }
  if (!ok) return;
  nf += tally_nonfinite<kVec>(g);
  float wv[kVec] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
  float mv[kVec] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
  float vv[kVec] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
  for (int e = 0; e < kVec; ++e) adam(a, bc1, bc2, __fmul_rn(__fmul_rn(g[e], a.inv_n), clip), wv[e], mv[e], vv[e]);
  st_stream_f4(a.master + j, make_float4(wv[0], wv[1], wv[2], wv[3]));
  st_stream_f4(a.master + j + 4, make_float4(wv[4], wv[5], wv[6], wv[7]));
  st_stream_f4(a.m + j, make_float4(mv[0], mv[1], mv[2], mv[3]));
  st_stream_f4(a.m + j + 4, make_float4(mv[4], mv[5], mv[6], mv[7]));
  st_stream_f4(a.v + j, make_float4(vv[0], vv[1], vv[2], vv[3]));
  st_stream_f4(a.v + j + 4, make_float4(vv[4], vv[5], vv[6], vv[7]));
  uint4 out;
  out.x = pack_bf16x2(wv[0], wv[1]);
  out.y = pack_bf16x2(wv[2], wv[3]);
  out.z = pack_bf16x2(wv[4], wv[5]);
  out.w = pack_bf16x2(wv[6], wv[7]);
  st_stream(a.p16 + j, out);
}

// One head or tail element k of the body (k < 0: the head) of segment si.
__device__ __forceinline__ void shifted_element(const StepArgs& a, const Seg& s, int si, long long k, float clip,
                                                float bc1, float bc2, unsigned& nf) {
  const long long j = s.base + k;
  if (!ZFS_CHECK(k >= -static_cast<long long>(a.head[si]) && k < s.len && j >= 0 && j < a.total_padded)) return;
  const float r = reduce_scalar(a, s, k);
  nf += tally_nonfinite<1>(&r);
  const float g = __fmul_rn(r, clip);
  float w = a.master[j], m = a.m[j], v = a.v[j];
  adam(a, bc1, bc2, g, w, m, v);
  a.master[j] = w;
  a.m[j] = m;
  a.v[j] = v;
  a.p16[j] = to_bf16_bits(w);
}

template <int N, bool kFp32, bool kDevBias>
__global__ void __launch_bounds__(kStepThreads, 1) step_shift_kernel(const __grid_constant__ StepArgs a) {
  const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  float bc1, bc2;
  if (!step_bias<kDevBias>(a, &bc1, &bc2)) return;  // the same for every thread
  const float clip = a.clip ? *a.clip : 1.0f;
  unsigned nf = 0;  // non-finite reduced gradients seen by this thread
  for (int si = 0; si < a.nseg; ++si) {
    const Seg& seg = a.seg[si];
    const long long nvec = seg.len / kVec;
    for (long long vi = first_index(tid, seg.vec_start, stride); vi < nvec; vi += stride) {
      shifted_vec8<N, kFp32>(a, seg, si, vi, clip, bc1, bc2, nf);
    }
  }
  // Heads and ragged ends: 16 threads per segment, at most 7 + 7 elements.
  for (int si = 0; si < a.nseg; ++si) {
    const Seg& seg = a.seg[si];
    const long long q = tid - static_cast<long long>(si) * 2 * kVec;
    if (q < 0 || q >= 2 * kVec) continue;
    const long long head = a.head[si];
    const long long k = q < head ? q - head : (seg.len / kVec) * kVec + (q - head);
    if (q < head || (q - head < kVec && k < seg.len)) shifted_element(a, seg, si, k, clip, bc1, bc2, nf);
  }
  flush_nonfinite(a.nonfinite, nf);
}

// ---------------------------------------------------------------------------
// Tile-staged kernel without a CTA barrier in its loop (bf16 N = 7..12).
//
// step_tma4_kernel synchronises the whole CTA twice per tile: a give-up
// decision after the wait, and a barrier after every thread has read the
// stage so that thread 0 may refill it.  Here every stage also has an
// "empty" mbarrier on which each warp arrives once it has read its part of
// the stage; thread 0 refills the stage consumed in the previous iteration
// after waiting (bounded) on that barrier, so no warp waits for the others
// and the next tiles stay in flight while the slowest warp finishes.
// Give-up decisions are warp-uniform (a warp meets __syncwarp below); a CTA
// whose producer or consumers give up counts one timeout, thread 0 waits
// (bounded) for every copy it issued, and the CTA leaves with the rest of its
// tiles not updated, as in the other staged kernels.  Tile geometry, the test
// hook, the index checks and the per-element arithmetic are
// step_tma4_kernel's, so results are bit-identical.
//
// Measured on GB300 over 100 M bf16 elements (step GB/s against the kernel
// each N took before): 512 threads with four stages of 2,048-element tiles at
// N = 7 6902-6903 / 6771-6814 (register-staged) and N = 8 7003-7012 /
// 6827-6830 (7001-7012 against 6826-6827 in another run; three stages
// 6872; the 73.4 M-param Llama-1024 layout 6972 / 6798-6799), three stages
// (four do not fit) at N = 9 6966 / 6748-6759, N = 10 7025-7038 / 6753-6764,
// N = 11 7119-7121 / 6778-6787 (2,048-element staged kernel), N = 12 7173 /
// 6914-6915.  256-thread CTAs (two per SM, four stages), 384 threads with
// four stages, 768 or 1,024 threads with two stages and 512 threads with two
// stages measured 1-20 % slower at N = 8..10; at N <= 6 (four or five stages
// as well), N >= 13 (two stages fit) and for fp32 gradients this kernel was
// slower than the kernels those take.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_arrive1(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

template <int N, bool kFp32, int kThreads, int kStages, bool kDevBias>
__global__ void __launch_bounds__(kThreads, 1) step_pipe_kernel(const __grid_constant__ StepArgs a) {
  float bc1, bc2;
  if (!step_bias<kDevBias>(a, &bc1, &bc2)) return;
  using L = Tma4Tile<N, kFp32, kThreads, kStages>;
  constexpr int S = kStages;
  constexpr long long T = L::kElems;
  constexpr int kWarps = kThreads / 32;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ __align__(8) uint64_t full[S];
  __shared__ __align__(8) uint64_t empty[S];
  __shared__ int cta_gave_up;  // some warp of the CTA gave up (counted once, below)
  long long n_tiles = 0;
  for (int s = 0; s < a.nseg; ++s) n_tiles += a.seg[s].len / T;
  const float clip = a.clip ? *a.clip : 1.0f;
  if (threadIdx.x == 0) {
    cta_gave_up = 0;
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  auto issue = [&](long long id, int stage) {  // thread 0 only
    int si;
    long long ti;
    locate_tile4<T>(a, id, &si, &ti);
    const Seg& sg = a.seg[si];
    unsigned char* st = smem + static_cast<size_t>(stage) * L::kStageBytes;
    const long long e0 = ti * T;
    if (!ZFS_CHECK(ti >= 0 && e0 + T <= sg.len && sg.base + e0 + T <= a.total_padded)) {
      mbar_arrive1(&full[stage]);
      return;
    }
    mbar_expect_tx(&full[stage], L::kStageBytes);
    if (a.inject_missing_copy && id == 0) return;
    for (int r = 0; r < N; ++r)
      bulk_load(st + r * L::kGradBytes, static_cast<const unsigned char*>(sg.g[r]) + e0 * (kFp32 ? 4 : 2),
                L::kGradBytes, &full[stage]);
    const long long j0 = sg.base + e0;
    unsigned char* st_state = st + N * L::kGradBytes;
    bulk_load(st_state, a.master + j0, L::kStateBytes, &full[stage]);
    bulk_load(st_state + L::kStateBytes, a.m + j0, L::kStateBytes, &full[stage]);
    bulk_load(st_state + 2 * L::kStateBytes, a.v + j0, L::kStateBytes, &full[stage]);
  };
  long long issued = 0;  // tiles issued by thread 0 (k-indices 0 .. issued-1)
  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      const long long id = blockIdx.x + static_cast<long long>(i) * gridDim.x;
      if (id < n_tiles) {
        issue(id, i);
        issued = i + 1;
      }
    }
  }
  bool gave_up = false;
  unsigned nf = 0;
  const int t4 = threadIdx.x * 4;
  const int lane = threadIdx.x & 31;
  long long k = 0;
  for (;; ++k) {
    const long long id = blockIdx.x + k * gridDim.x;
    if (id >= n_tiles) break;
    const int stage = static_cast<int>(k % S);
    const uint32_t parity = static_cast<uint32_t>((k / S) & 1);
    const bool got = mbar_try_wait(&full[stage], parity) || wait_tile(&full[stage], parity);
    if (!__all_sync(0xffffffffu, got)) {  // the warp gives up together (it meets __syncwarp below)
      gave_up = true;
      if (lane == 0) cta_gave_up = 1;
      break;
    }
    const unsigned char* st = smem + static_cast<size_t>(stage) * L::kStageBytes;
    float gg[4];
    if constexpr (kFp32) {
      const float4 x0 = *reinterpret_cast<const float4*>(st + t4 * 4);
      gg[0] = x0.x; gg[1] = x0.y; gg[2] = x0.z; gg[3] = x0.w;
#pragma unroll
      for (int r = 1; r < N; ++r) {
        const float4 x = *reinterpret_cast<const float4*>(st + r * L::kGradBytes + t4 * 4);
        gg[0] = __fadd_rn(gg[0], x.x); gg[1] = __fadd_rn(gg[1], x.y);
        gg[2] = __fadd_rn(gg[2], x.z); gg[3] = __fadd_rn(gg[3], x.w);
      }
    } else {
      const uint2 x0 = *reinterpret_cast<const uint2*>(st + t4 * 2);
      gg[0] = bf16_lo(x0.x); gg[1] = bf16_hi(x0.x); gg[2] = bf16_lo(x0.y); gg[3] = bf16_hi(x0.y);
#pragma unroll
      for (int r = 1; r < N; ++r) {
        const uint2 x = *reinterpret_cast<const uint2*>(st + r * L::kGradBytes + t4 * 2);
        gg[0] = __fadd_rn(gg[0], bf16_lo(x.x)); gg[1] = __fadd_rn(gg[1], bf16_hi(x.x));
        gg[2] = __fadd_rn(gg[2], bf16_lo(x.y)); gg[3] = __fadd_rn(gg[3], bf16_hi(x.y));
      }
    }
    const unsigned char* st_state = st + N * L::kGradBytes;
    const float4 w4 = *reinterpret_cast<const float4*>(st_state + t4 * 4);
    const float4 m4 = *reinterpret_cast<const float4*>(st_state + L::kStateBytes + t4 * 4);
    const float4 v4 = *reinterpret_cast<const float4*>(st_state + 2 * L::kStateBytes + t4 * 4);
    __syncwarp();
    if (lane == 0) mbar_arrive1(&empty[stage]);  // this warp has read the stage
    // Thread 0 refills the stage consumed in the previous iteration.
    if (threadIdx.x == 0 && k >= 1) {
      const long long kp = k - 1;
      const long long nid = blockIdx.x + (kp + S) * gridDim.x;
      if (nid < n_tiles) {
        const int ps = static_cast<int>(kp % S);
        const uint32_t pp = static_cast<uint32_t>((kp / S) & 1);
        if (!mbar_try_wait(&empty[ps], pp) && !wait_tile(&empty[ps], pp)) {
          gave_up = true;
        } else {
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          issue(nid, ps);
          issued = kp + S + 1;
        }
      }
    }
    if (threadIdx.x < 32) gave_up = __shfl_sync(0xffffffffu, gave_up, 0);  // warp 0 leaves together
    if (threadIdx.x == 0 && gave_up) cta_gave_up = 1;
    float w[4] = {w4.x, w4.y, w4.z, w4.w}, m[4] = {m4.x, m4.y, m4.z, m4.w}, v[4] = {v4.x, v4.y, v4.z, v4.w};
    nf += tally_nonfinite<4>(gg);
#pragma unroll
    for (int e = 0; e < 4; ++e) adam(a, bc1, bc2, __fmul_rn(__fmul_rn(gg[e], a.inv_n), clip), w[e], m[e], v[e]);
    int si;
    long long ti;
    locate_tile4<T>(a, id, &si, &ti);
    if (ZFS_CHECK((ti + 1) * T <= a.seg[si].len && a.seg[si].base + (ti + 1) * T <= a.total_padded)) {
      const long long j = a.seg[si].base + ti * T + t4;
      st_stream_f4(a.master + j, make_float4(w[0], w[1], w[2], w[3]));
      st_stream_f4(a.m + j, make_float4(m[0], m[1], m[2], m[3]));
      st_stream_f4(a.v + j, make_float4(v[0], v[1], v[2], v[3]));
      uint2 out;
      out.x = pack_bf16x2(w[0], w[1]);
      out.y = pack_bf16x2(w[2], w[3]);
      __stcs(reinterpret_cast<uint2*>(a.p16 + j), out);
    }
    if (gave_up) break;  // thread 0 could not refill: warp 0 leaves after this tile
  }
  // Every thread gets here once (every wait above is bounded): whether any
  // warp gave up is then known to all.
  __syncthreads();
  if (cta_gave_up) {
    if (threadIdx.x == 0) {
      atomicAdd(&g_step_timeouts, 1u);
      // every tile issued and not consumed by thread 0: wait (bounded) for its copies
      for (long long j = k; j < issued; ++j) {
        const int s = static_cast<int>(j % S);
        const uint32_t parity = static_cast<uint32_t>((j / S) & 1);
        const unsigned long long t0 = global_ns();
        while (!mbar_try_wait(&full[s], parity) && global_ns() - t0 < kTmaDrainNs) {
        }
      }
    }
    flush_nonfinite(a.nonfinite, nf);
    return;
  }
  const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (int s = 0; s < a.nseg; ++s) {
    const Seg& sg = a.seg[s];
    for (long long kk = (sg.len / T) * T + tid; kk < sg.len; kk += stride) {
      step_scalar_element(a, sg, kk, clip, bc1, bc2, nf);
    }
  }
  flush_nonfinite(a.nonfinite, nf);
}

// Capturable steps: the device step count advances after the step's launches.
__global__ void count_step_kernel(long long* t) { *t += 1; }

// ---------------------------------------------------------------------------
// Launch configuration.
// ---------------------------------------------------------------------------
using StepKernel = void (*)(StepArgs);

template <bool kFp32, bool kDevBias>
StepKernel vec_kernel_for(int n) {
  switch (n) {
    case 1: return step_vec_kernel<1, kFp32, kDevBias>;
    case 2: return step_vec_kernel<2, kFp32, kDevBias>;
    case 3: return step_vec_kernel<3, kFp32, kDevBias>;
    case 4: return step_vec_kernel<4, kFp32, kDevBias>;
    case 5: return step_vec_kernel<5, kFp32, kDevBias>;
    case 6: return step_vec_kernel<6, kFp32, kDevBias>;
    case 7: return step_vec_kernel<7, kFp32, kDevBias>;
    case 8: return step_vec_kernel<8, kFp32, kDevBias>;
    case 9: return step_vec_kernel<9, kFp32, kDevBias>;
    case 10: return step_vec_kernel<10, kFp32, kDevBias>;
    case 11: return step_vec_kernel<11, kFp32, kDevBias>;
    case 12: return step_vec_kernel<12, kFp32, kDevBias>;
    case 13: return step_vec_kernel<13, kFp32, kDevBias>;
    case 14: return step_vec_kernel<14, kFp32, kDevBias>;
    case 15: return step_vec_kernel<15, kFp32, kDevBias>;
    case 16: return step_vec_kernel<16, kFp32, kDevBias>;
    default: return nullptr;
  }
}

constexpr int kMaxDevices = 64;

constexpr int kMaxSmemKernels = 128;

struct DeviceInfo {
  int sms = 0;
  // [device-side bias][fp32 gradients][N]
  int vec_blocks_per_sm[2][2][kMaxRanks + 1] = {};
  int shift_blocks_per_sm[2][2][kMaxRanks + 1] = {};
  // Staged kernels whose dynamic shared memory limit is raised, and in which
  // CUDA context (a function attribute belongs to a context): a ring, an
  // evicted entry is simply set again.
  const void* smem_fn[kMaxSmemKernels] = {};
  unsigned long long smem_ctx[kMaxSmemKernels] = {};
  int smem_next = 0;
};

// Shared memory of one SM usable by CTAs, and what each CTA reserves.
constexpr long long kMaxSmemPerSm = 228 * 1024;
constexpr long long kSmemReservedPerCta = 1024;

std::mutex g_info_mutex;
DeviceInfo g_info[kMaxDevices];

// Raises `fn`'s dynamic shared memory limit to `bytes` once per CUDA context
// (the attribute belongs to the context: a second context on the same GPU
// needs its own call).  Without a context id the call is made every time.
// The record lives in this file's tables (internal linkage), not in statics
// of the launch templates: those would be one object process-wide, shared
// with any other copy of the library loaded alongside, which then would skip
// the call for its own kernels.
cudaError_t ensure_smem(int dev, const void* fn, uint32_t bytes) {
  unsigned long long cid = 0;
  const bool have_id = current_context_id(&cid);
  std::lock_guard<std::mutex> lock(g_info_mutex);
  DeviceInfo& d = g_info[dev];
  if (have_id) {
    for (int i = 0; i < kMaxSmemKernels; ++i)
      if (d.smem_fn[i] == fn && d.smem_ctx[i] == cid) return cudaSuccess;
  }
  const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e != cudaSuccess) return e;
  if (have_id) {
    d.smem_fn[d.smem_next] = fn;
    d.smem_ctx[d.smem_next] = cid;
    d.smem_next = (d.smem_next + 1) % kMaxSmemKernels;
  }
  return cudaSuccess;
}

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

unsigned int step_debug_failures() {
#ifdef ZFS_DEBUG_CHECKS
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_debug_failures, sizeof v) != cudaSuccess) return 0xFFFFFFFFu;
  return v;
#else
  return 0;
#endif
}

unsigned int step_timeouts() {
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_step_timeouts, sizeof v) != cudaSuccess) return 0xFFFFFFFFu;
  return v;
}

template <int N, bool kFp32, bool kDevBias>
cudaError_t launch_tma(const StepArgs& a, cudaStream_t stream) {
  constexpr uint32_t kSmem = TmaTile<N, kFp32>::kSmemBytes;
  static_assert(kSmem + 128 <= 227 * 1024, "staged tiles must fit one CTA's shared memory (227 KB)");
  const int dev = current_device();
  const cudaError_t e = ensure_smem(dev, reinterpret_cast<const void*>(step_tma_kernel<N, kFp32, kDevBias>), kSmem);
  if (e != cudaSuccess) return e;
  int per_sm = static_cast<int>(kMaxSmemPerSm / (kSmem + kSmemReservedPerCta));
  if (per_sm < 1) per_sm = 1;
  if (per_sm > kStepCtasPerSm) per_sm = kStepCtasPerSm;
  step_tma_kernel<N, kFp32, kDevBias>
      <<<static_cast<unsigned>(cached_sms(dev) * per_sm), kStepThreads, kSmem, stream>>>(a);
  return cudaGetLastError();
}

template <int N, bool kFp32, int kThreads, int kStages, int kCtasPerSm, bool kDevBias>
cudaError_t launch_pipe(const StepArgs& a, cudaStream_t stream) {
  constexpr uint32_t kSmem = Tma4Tile<N, kFp32, kThreads, kStages>::kSmemBytes;
  static_assert(kSmem + 128 <= 227 * 1024, "staged tiles must fit one CTA's shared memory (227 KB)");
  auto kernel = step_pipe_kernel<N, kFp32, kThreads, kStages, kDevBias>;
  const int dev = current_device();
  const cudaError_t e = ensure_smem(dev, reinterpret_cast<const void*>(kernel), kSmem);
  if (e != cudaSuccess) return e;
  int per_sm = static_cast<int>(kMaxSmemPerSm / (kSmem + kSmemReservedPerCta));
  if (per_sm < 1) per_sm = 1;
  if (per_sm > kCtasPerSm) per_sm = kCtasPerSm;
  kernel<<<static_cast<unsigned>(cached_sms(dev) * per_sm), kThreads, kSmem, stream>>>(a);
  return cudaGetLastError();
}

template <int N, bool kFp32, int kThreads, int kStages, int kCtasPerSm, bool kDevBias>
cudaError_t launch_tma4(const StepArgs& a, cudaStream_t stream) {
  constexpr uint32_t kSmem = Tma4Tile<N, kFp32, kThreads, kStages>::kSmemBytes;
  static_assert(kSmem + 128 <= 227 * 1024, "staged tiles must fit one CTA's shared memory (227 KB)");
  auto kernel = step_tma4_kernel<N, kFp32, kThreads, kStages, kDevBias>;
  const int dev = current_device();
  const cudaError_t e = ensure_smem(dev, reinterpret_cast<const void*>(kernel), kSmem);
  if (e != cudaSuccess) return e;
  int per_sm = static_cast<int>(kMaxSmemPerSm / (kSmem + kSmemReservedPerCta));
  if (per_sm < 1) per_sm = 1;
  if (per_sm > kCtasPerSm) per_sm = kCtasPerSm;
  kernel<<<static_cast<unsigned>(cached_sms(dev) * per_sm), kThreads, kSmem, stream>>>(a);
  return cudaGetLastError();
}

// fp32 replicas from N = 10: 256 threads (1,024-element tiles), three stages
// at N = 10, 11 and two from N = 12 (measured, see step_tma4_kernel).  At
// N = 7: 512 threads, two stages (100 M elements: 7038-7047 GB/s against
// 6661-6673 for the register-staged kernel and 6678 for step_tma_kernel; at
// N = 2, 4, 6 every staged shape tried was slower than the register-staged
// kernel).
template <int N, bool kDevBias>
cudaError_t launch_tma4_fp32(const StepArgs& a, cudaStream_t stream) {
  if constexpr (N < 10) {
    return launch_tma4<N, true, 2 * kStepThreads, 2, 1, kDevBias>(a, stream);
  } else {
    return launch_tma4<N, true, kStepThreads, (N <= 11 ? 3 : 2), 1, kDevBias>(a, stream);
  }
}

// bf16 replicas at N = 1..4.  Measured on GB300 over 100 M elements (GB/s):
// N = 1, 2 with 256 threads, two stages, two CTAs per SM: 6575-6623 and
// 6542-6557 against 6317-6344 for the register-staged kernel; N = 3, 4 with
// 512 threads, two stages, one CTA per SM: 6652-6680 and 6779-6807 against
// 6568-6581 and 6671-6724.  From N = 5 on the register-staged kernel is as
// fast or faster (N = 5: 6765 / 6778; N = 8: 6394-6599 / 6773).
template <int N, bool kDevBias>
cudaError_t launch_tma4_bf16(const StepArgs& a, cudaStream_t stream) {
  if constexpr (N <= 2) {
    return launch_tma4<N, false, kStepThreads, 2, 2, kDevBias>(a, stream);
  } else {
    return launch_tma4<N, false, 2 * kStepThreads, 2, 1, kDevBias>(a, stream);
  }
}

// A staged kernel where one measured faster than the register-staged kernel
// (launches of at least kTmaMinElems elements): bf16 N = 1..4 (4-element
// staged), N = 7..12 (barrier-free pipelined: four stages of 2,048-element
// tiles at N = 7, 8, where they fit, three from N = 9), N >= 13 (2,048-element
// staged); fp32 N >= 7.  Other rank counts return with *launched = false.
template <bool kDevBias>
cudaError_t try_launch_tma(const StepArgs& a, cudaStream_t stream, bool* launched) {
  *launched = true;
  if (!a.grad_fp32) {
    switch (a.n_ranks) {
      case 1: return launch_tma4_bf16<1, kDevBias>(a, stream);
      case 2: return launch_tma4_bf16<2, kDevBias>(a, stream);
      case 3: return launch_tma4_bf16<3, kDevBias>(a, stream);
      case 4: return launch_tma4_bf16<4, kDevBias>(a, stream);
      case 7: return launch_pipe<7, false, 512, 4, 1, kDevBias>(a, stream);
      case 8: return launch_pipe<8, false, 512, 4, 1, kDevBias>(a, stream);
      case 9: return launch_pipe<9, false, 512, 3, 1, kDevBias>(a, stream);
      case 10: return launch_pipe<10, false, 512, 3, 1, kDevBias>(a, stream);
      case 11: return launch_pipe<11, false, 512, 3, 1, kDevBias>(a, stream);
      case 12: return launch_pipe<12, false, 512, 3, 1, kDevBias>(a, stream);
      case 13: return launch_tma<13, false, kDevBias>(a, stream);
      case 14: return launch_tma<14, false, kDevBias>(a, stream);
      case 15: return launch_tma<15, false, kDevBias>(a, stream);
      case 16: return launch_tma<16, false, kDevBias>(a, stream);
      default: break;
    }
  } else {
    switch (a.n_ranks) {
      case 7: return launch_tma4_fp32<7, kDevBias>(a, stream);
      case 8: return launch_tma<8, true, kDevBias>(a, stream);
      case 9: return launch_tma<9, true, kDevBias>(a, stream);
      case 10: return launch_tma4_fp32<10, kDevBias>(a, stream);
      case 11: return launch_tma4_fp32<11, kDevBias>(a, stream);
      case 12: return launch_tma4_fp32<12, kDevBias>(a, stream);
      case 13: return launch_tma4_fp32<13, kDevBias>(a, stream);
      case 14: return launch_tma4_fp32<14, kDevBias>(a, stream);
      case 15: return launch_tma4_fp32<15, kDevBias>(a, stream);
      case 16: return launch_tma4_fp32<16, kDevBias>(a, stream);
      default: break;
    }
  }
  *launched = false;
  return cudaSuccess;
}

template <bool kDevBias>
cudaError_t launch_step_vec_t(const StepArgs& a, cudaStream_t stream) {
  if (a.total_elems >= kTmaMinElems) {
    bool launched = false;
    const cudaError_t e = try_launch_tma<kDevBias>(a, stream, &launched);
    if (launched) return e;
  }
  StepKernel k = a.grad_fp32 ? vec_kernel_for<true, kDevBias>(a.n_ranks) : vec_kernel_for<false, kDevBias>(a.n_ranks);
  if (!k) return cudaErrorInvalidValue;
  const int dev = current_device();
  const int sms = cached_sms(dev);
  int bps = resident_blocks(&g_info[dev].vec_blocks_per_sm[kDevBias ? 1 : 0][a.grad_fp32 ? 1 : 0][a.n_ranks],
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

template <bool kFp32, bool kDevBias>
StepKernel shift_kernel_for(int n) {
  switch (n) {
    case 1: return step_shift_kernel<1, kFp32, kDevBias>;
    case 2: return step_shift_kernel<2, kFp32, kDevBias>;
    case 3: return step_shift_kernel<3, kFp32, kDevBias>;
    case 4: return step_shift_kernel<4, kFp32, kDevBias>;
    case 5: return step_shift_kernel<5, kFp32, kDevBias>;
    case 6: return step_shift_kernel<6, kFp32, kDevBias>;
    case 7: return step_shift_kernel<7, kFp32, kDevBias>;
    case 8: return step_shift_kernel<8, kFp32, kDevBias>;
    case 9: return step_shift_kernel<9, kFp32, kDevBias>;
    case 10: return step_shift_kernel<10, kFp32, kDevBias>;
    case 11: return step_shift_kernel<11, kFp32, kDevBias>;
    case 12: return step_shift_kernel<12, kFp32, kDevBias>;
    case 13: return step_shift_kernel<13, kFp32, kDevBias>;
    case 14: return step_shift_kernel<14, kFp32, kDevBias>;
    case 15: return step_shift_kernel<15, kFp32, kDevBias>;
    case 16: return step_shift_kernel<16, kFp32, kDevBias>;
    default: return nullptr;
  }
}

template <bool kDevBias>
cudaError_t launch_step_shift_t(const StepArgs& a, cudaStream_t stream) {
  StepKernel k = a.grad_fp32 ? shift_kernel_for<true, kDevBias>(a.n_ranks) : shift_kernel_for<false, kDevBias>(a.n_ranks);
  if (!k) return cudaErrorInvalidValue;
  const int dev = current_device();
  const int sms = cached_sms(dev);
  int bps = resident_blocks(&g_info[dev].shift_blocks_per_sm[kDevBias ? 1 : 0][a.grad_fp32 ? 1 : 0][a.n_ranks],
                            reinterpret_cast<const void*>(k));
  if (bps > kStepCtasPerSm) bps = kStepCtasPerSm;  // as the register-staged kernel
  // enough threads for the heads and ragged ends: 16 per segment
  long long work = a.total_vec;
  if (work < static_cast<long long>(a.nseg) * 2 * kVec) work = static_cast<long long>(a.nseg) * 2 * kVec;
  const long long grid = grid_for(work, sms, bps);
  k<<<static_cast<unsigned>(grid), kStepThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_step_vec(const StepArgs& a, cudaStream_t stream) {
  return a.dev_t ? launch_step_vec_t<true>(a, stream) : launch_step_vec_t<false>(a, stream);
}

cudaError_t launch_step_shift(const StepArgs& a, cudaStream_t stream) {
  return a.dev_t ? launch_step_shift_t<true>(a, stream) : launch_step_shift_t<false>(a, stream);
}

cudaError_t launch_count_step(long long* t, cudaStream_t stream) {
  count_step_kernel<<<1, 1, 0, stream>>>(t);
  return cudaGetLastError();
}

}  // namespace zfs
