// Auxiliary sm_103a kernels of the ZeRO flat-parameter library: the
// gradient-norm pass of global-norm clipping, fp32 gradient accumulation,
// make_master's fills and copies, checkpoint copies and the ZeRO-3 gather.

#include <algorithm>
#include <utility>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "zero_device.cuh"
#include "zero_aux_internal.h"
#include "zero_internal.h"

namespace zfs {
namespace {

// ---------------------------------------------------------------------------
// Overlapped launches.  The norm pass, its finalize and the ZeRO-3 gathers
// are launched with programmatic stream serialization: their CTAs may become
// resident while the kernel before them on the stream is still finishing,
// and wait in await_previous_grid() — griddepcontrol.wait returns once every
// prerequisite grid has completed and its memory operations are visible —
// before their first load.  So such a kernel reads only what an ordinary
// launch would; what it gains is that its CTAs start the moment the previous
// kernel ends instead of being launched then.  Each CTA then lets the next
// kernel's CTAs be scheduled.  Measured on GB300: ten per-unit gathers of the
// Llama-2048 units at N = 8 6,285 -> 6,714 GB/s; the clip call (norm pass +
// finalize) over 73.4 M elements at N = 8 bf16 6,640 -> 6,721 GB/s of
// gradient reads, 268 M at N = 2 fp32 7,075 -> 7,142.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void await_previous_grid() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_overlapped(void (*kernel)(KArgs...), long long grid, int threads, cudaStream_t stream,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(static_cast<unsigned>(threads));
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Global gradient norm.
// ---------------------------------------------------------------------------
// Squares are accumulated per thread as an unevaluated fp32 pair (hi, lo):
// the product's rounding error comes exactly from one fma, the sum's from
// the two-sum identity, giving ~48-bit accuracy at fp32 throughput (fp64 is
// scarce on this part: a per-element fp64 operation would cap the pass far
// below HBM speed).
//
// The pair is exact as long as nothing overflows and no product error
// underflows.  Instead of testing every element (a range test per element
// cost a quarter of the pass's throughput at few replicas: measured on GB300
// over 2.03 B fp32 elements of two replicas, 5.58 TB/s of reads with the
// test, 7.45 without), a thread checks its result once: when the pair is not
// finite (an inf or NaN gradient, or an overflow) or the sum is below 2^-60
// (where product errors of tiny gradients may have been lost), the thread
// sums its elements again, in the same order, as fp64 squares (exact) with
// fp64 additions.  Which way a thread's sum goes is a function of its
// elements alone, so it is the same on every path.
struct SqAcc {
  float hi = 0.0f, lo = 0.0f;

  __device__ __forceinline__ void add(float g) {
    const float p = __fmul_rn(g, g);
    const float e = __fmaf_rn(g, g, -p);  // exact: g*g = p + e
    const float t = __fadd_rn(hi, p);
    const float bp = __fsub_rn(t, hi);
    const float err = __fadd_rn(__fsub_rn(hi, __fsub_rn(t, bp)), __fsub_rn(p, bp));  // hi + p = t + err
    hi = t;
    lo = __fadd_rn(lo, __fadd_rn(err, e));
  }
  __device__ __forceinline__ void add8(const float* g) {
#pragma unroll
    for (int e = 0; e < kVec; ++e) add(g[e]);
  }
  // The pair holds the sum to ~48 bits (see above).
  __device__ __forceinline__ bool exact() const { return isfinite(hi) && isfinite(lo) && hi >= 0x1p-60f; }
  __device__ __forceinline__ double total() const {
    return __dadd_rn(static_cast<double>(hi), static_cast<double>(lo));
  }
};

// Fixed-order sum of one double per thread across the CTA (warp tree, then
// warps in order).  Result valid in thread 0.
template <int kThreads>
__device__ __forceinline__ double block_sum(double d, double* smem) {
  for (int off = 16; off > 0; off >>= 1) d = __dadd_rn(d, __shfl_down_sync(0xffffffffu, d, off));
  const int warp = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) smem[warp] = d;
  __syncthreads();
  double total = 0.0;
  if (threadIdx.x == 0) {
    total = smem[0];
    for (int w = 1; w < kThreads / 32; ++w) total = __dadd_rn(total, smem[w]);
  }
  return total;
}

template <int N, bool kFp32>
__device__ __forceinline__ void reduced8(const NormArgs& a, const NormSeg& s, long long e0, float* g) {
  if constexpr (!kFp32) {
    uint4 raw[N];
#pragma unroll
    for (int r = 0; r < N; ++r) raw[r] = ld_stream(static_cast<const unsigned short*>(s.g[r]) + e0);
    g[0] = bf16_lo(raw[0].x); g[1] = bf16_hi(raw[0].x); g[2] = bf16_lo(raw[0].y); g[3] = bf16_hi(raw[0].y);
    g[4] = bf16_lo(raw[0].z); g[5] = bf16_hi(raw[0].z); g[6] = bf16_lo(raw[0].w); g[7] = bf16_hi(raw[0].w);
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
      const float* base = static_cast<const float*>(s.g[r]) + e0;
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
#pragma unroll
  for (int e = 0; e < kVec; ++e) g[e] = __fmul_rn(g[e], a.inv_n);
}

// reduced8 for a whole group of a unit whose gradients are not 16-byte
// aligned: replica r starts s.shift[r] elements past a boundary, so the
// group's elements lie in W + 1 aligned 16-byte words (W for phi == 0), all
// loaded before any is used; the word past the group starts inside it.  The
// last word is also the next thread's first: the duplicate request is served
// on chip (against taking it from the neighbouring lane by warp shuffle:
// N = 3 bf16 +11 %, elsewhere within 1 %).  Same values, same rank order as
// reduced8.
template <int N, bool kFp32>
__device__ __forceinline__ void shifted_reduced8(const NormArgs& a, const NormSeg& s, long long e0, float* g) {
  constexpr int W = kFp32 ? 2 : 1;  // 16-byte words of one group and replica
  uint4 w[N][W + 1];
#pragma unroll
  for (int r = 0; r < N; ++r) {
    const int phi = s.shift[r];
    const uint4* words = reinterpret_cast<const uint4*>(static_cast<const char*>(s.g[r]) - phi * (kFp32 ? 4 : 2)) +
                         (e0 / kVec) * W;
#pragma unroll
    for (int q = 0; q < W; ++q) w[r][q] = ld_stream(words + q);
    w[r][W] = phi != 0 ? ld_stream(words + W) : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int r = 0; r < N; ++r) {
    const int phi = s.shift[r];  // uniform over the launch
    float x[kVec];
    if constexpr (!kFp32) {
      const uint32_t u[8] = {w[r][0].x, w[r][0].y, w[r][0].z, w[r][0].w, w[r][1].x, w[r][1].y, w[r][1].z, w[r][1].w};
      const int k = phi >> 1;
      uint32_t t[6], v[5];
#pragma unroll
      for (int i = 0; i < 6; ++i) t[i] = (k & 2) ? u[i + 2] : u[i];
#pragma unroll
      for (int i = 0; i < 5; ++i) v[i] = (k & 1) ? t[i + 1] : t[i];
      const uint32_t sh = static_cast<uint32_t>(phi & 1) * 16;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t y = __funnelshift_r(v[i], v[i + 1], sh);
        x[2 * i] = bf16_lo(y);
        x[2 * i + 1] = bf16_hi(y);
      }
    } else {
      const uint32_t u[12] = {w[r][0].x, w[r][0].y, w[r][0].z, w[r][0].w, w[r][1].x, w[r][1].y,
                              w[r][1].z, w[r][1].w, w[r][2].x, w[r][2].y, w[r][2].z, w[r][2].w};
      uint32_t t[9];
#pragma unroll
      for (int i = 0; i < 9; ++i) t[i] = (phi & 2) ? u[i + 2] : u[i];
#pragma unroll
      for (int i = 0; i < kVec; ++i) x[i] = __uint_as_float((phi & 1) ? t[i + 1] : t[i]);
    }
    if (r == 0) {
#pragma unroll
      for (int e = 0; e < kVec; ++e) g[e] = x[e];
    } else {
#pragma unroll
      for (int e = 0; e < kVec; ++e) g[e] = __fadd_rn(g[e], x[e]);
    }
  }
#pragma unroll
  for (int e = 0; e < kVec; ++e) g[e] = __fmul_rn(g[e], a.inv_n);
}

// Same reduction as the step (rank order, then x 1/N) for one element of any alignment.
__device__ __forceinline__ float reduced1(const NormArgs& a, const NormSeg& s, long long k) {
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

// Stores 8 reduced gradients of a unit at unit-relative element e0.
__device__ __forceinline__ void keep8(const NormSeg& s, long long e0, const float* g) {
  float* p = s.keep + e0;
  if (s.keep_vec) {
    st_stream_f4(p, make_float4(g[0], g[1], g[2], g[3]));
    st_stream_f4(p + 4, make_float4(g[4], g[5], g[6], g[7]));
  } else {
    for (int e = 0; e < kVec; ++e) p[e] = g[e];
  }
}

// One CTA per chunk.  Thread t takes the chunk's 8-element groups t, t+256,
// ... in order and accumulates their elements in order; the vector and the
// element-wise paths visit elements in the same order, so the chunk's sum
// does not depend on the gradients' alignment.  Full groups are loaded two at a time before either is
// accumulated (more bytes in flight per thread; the loose register bound
// allows it), which does not change the order — except for fp32 gradients
// from kNormPairMaxRanksFp32 + 1 replicas on: two groups' loads then need
// more than 128 registers, which leaves one CTA per SM, so those instances
// load one group at a time at three CTAs per SM (measured on GB300 over
// 73.5 M elements, GB/s of gradient reads: N = 7 fp32 6988-7012 against
// 6328, N = 8 7054 against 6423, N = 16 7211-7228 against 7122; at N = 5, 6
// either way within 1 %; the norm bits are the same, as the order is).
constexpr int kNormPairMaxRanksFp32 = 6;

template <int N, bool kFp32>
struct NormShape {
  static constexpr bool kPairs = !kFp32 || N <= kNormPairMaxRanksFp32;
  static constexpr int kMinBlocks = kPairs ? 1 : 3;
};

// A thread's elements of one chunk again, in the same order, as exact fp64
// squares summed in fp64: the rare path of SqAcc::exact() == false.
__device__ __noinline__ double exact_thread_sum(const NormArgs& a, const NormSeg& s, long long c0, long long len) {
  double w = 0.0;
  for (long long grp = threadIdx.x; grp * kVec < len; grp += kStepThreads) {
    for (int e = 0; e < kVec; ++e) {
      if (grp * kVec + e < len) {
        const double d = static_cast<double>(reduced1(a, s, c0 + grp * kVec + e));
        w = __dadd_rn(w, __dmul_rn(d, d));
      }
    }
  }
  return w;
}

// kShifted instances take the launches of units whose gradients are not
// 16-byte aligned (whole groups through shifted aligned words, one group at a
// time, every register they need); the others take aligned units, so their
// code and register budget are those of the aligned path alone.
template <int N, bool kFp32, bool kShifted>
__global__ void __launch_bounds__(kStepThreads, kShifted ? 1 : NormShape<N, kFp32>::kMinBlocks)
    grad_sq_kernel(const __grid_constant__ NormArgs a) {
  await_previous_grid();
  constexpr bool kPairs = NormShape<N, kFp32>::kPairs;
  __shared__ double smem[kStepThreads / 32];
  const long long b = blockIdx.x;
  int si = 0;
  while (si + 1 < a.nseg && b >= a.seg[si + 1].chunk_start) ++si;
  const NormSeg& s = a.seg[si];
  const long long k = b - s.chunk_start;
  const long long c0 = k * kClipChunk;
  const long long c1 = (k == s.n_chunks - 1) ? s.len : c0 + kClipChunk;
  // (CTA-uniform: a failed check empties the chunk, the block sum still runs)
  const long long len = ZFS_CHECK(k >= 0 && k < s.n_chunks && c1 <= s.len) ? c1 - c0 : 0;
  SqAcc acc;
  long long grp = threadIdx.x;
  if constexpr (kShifted) {
    // Unaligned gradients: whole groups through shifted aligned words, in the
    // same order; a thread leaves at its first group that is not whole, which
    // the loop below takes element by element.
    for (; grp * kVec + kVec <= len; grp += kStepThreads) {
      float g[kVec];
      shifted_reduced8<N, kFp32>(a, s, c0 + grp * kVec, g);
      if (s.keep) keep8(s, c0 + grp * kVec, g);
      acc.add8(g);
    }
  }
  for (; kPairs && s.vec_ok && (grp + kStepThreads) * kVec + kVec <= len; grp += 2 * kStepThreads) {
    float g0[kVec], g1[kVec];
    reduced8<N, kFp32>(a, s, c0 + grp * kVec, g0);
    reduced8<N, kFp32>(a, s, c0 + (grp + kStepThreads) * kVec, g1);
    if (s.keep) {
      keep8(s, c0 + grp * kVec, g0);
      keep8(s, c0 + (grp + kStepThreads) * kVec, g1);
    }
    acc.add8(g0);
    acc.add8(g1);
  }
  for (; grp * kVec < len; grp += kStepThreads) {
    const long long e0 = c0 + grp * kVec;
    if (s.vec_ok && grp * kVec + kVec <= len) {
      float g[kVec];
      reduced8<N, kFp32>(a, s, e0, g);
      if (s.keep) keep8(s, e0, g);
      acc.add8(g);
    } else {
      for (int e = 0; e < kVec; ++e) {
        if (grp * kVec + e < len) {
          const float g = reduced1(a, s, e0 + e);
          if (s.keep) s.keep[e0 + e] = g;
          acc.add(g);
        }
      }
    }
  }
  const double mine = acc.exact() ? acc.total() : exact_thread_sum(a, s, c0, len);
  const double total = block_sum<kStepThreads>(mine, smem);
  if (threadIdx.x == 0) a.partials[s.out_start + k] = total;
}

__global__ void __launch_bounds__(kFinalizeThreads) clip_finalize_kernel(char* ws, long long n, float max_norm) {
  await_previous_grid();
  __shared__ double smem[kFinalizeThreads / 32];
  const double* partials = reinterpret_cast<const double*>(ws + kClipHeaderBytes);
  double d = 0.0;
  for (long long i = threadIdx.x; i < n; i += kFinalizeThreads) d = __dadd_rn(d, partials[i]);
  const double sum_sq = block_sum<kFinalizeThreads>(d, smem);
  if (threadIdx.x == 0) {
    const double norm = __dsqrt_rn(sum_sq);
    const double coef = __ddiv_rn(static_cast<double>(max_norm), __dadd_rn(norm, 1e-6));
    *reinterpret_cast<double*>(ws) = norm;
    // the cap at 1 keeps a NaN: a NaN norm makes every clipped gradient NaN
    *reinterpret_cast<float*>(ws + 8) = isnan(coef) ? __int_as_float(0x7fc00000) : (coef < 1.0 ? __double2float_rn(coef) : 1.0f);
  }
}

// ---------------------------------------------------------------------------
// fp32 gradient accumulation (one micro-step).  The replicas' buffers form
// one concatenated index space for the grid-stride loop; 8 elements per
// vector: one 16-byte bf16 load, two 16-byte fp32 loads (none on the first
// micro-step) and two 16-byte fp32 stores.  A thread loads kIlp vectors
// before adding any.  Measured on GB300 (2 CTAs/SM): 2 vectors give 6741 GB/s
// on later micro-steps (4 gave 5861, 8 gave 6314); the write-heavy first
// micro-step does best with 8 (6245 GB/s; 2 gave 5833).
// ---------------------------------------------------------------------------
constexpr int kAccumIlpFirst = 8;
constexpr int kAccumIlpLater = 2;

__device__ __forceinline__ void accumulate8(const uint4 raw, const float4 x0, const float4 x1, bool first, float* p) {
  float g[kVec] = {bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y),
                   bf16_lo(raw.z), bf16_hi(raw.z), bf16_lo(raw.w), bf16_hi(raw.w)};
  if (!first) {
    g[0] = __fadd_rn(x0.x, g[0]); g[1] = __fadd_rn(x0.y, g[1]);
    g[2] = __fadd_rn(x0.z, g[2]); g[3] = __fadd_rn(x0.w, g[3]);
    g[4] = __fadd_rn(x1.x, g[4]); g[5] = __fadd_rn(x1.y, g[5]);
    g[6] = __fadd_rn(x1.z, g[6]); g[7] = __fadd_rn(x1.w, g[7]);
  }
  st_stream_f4(p, make_float4(g[0], g[1], g[2], g[3]));
  st_stream_f4(p + 4, make_float4(g[4], g[5], g[6], g[7]));
}

// kFirst is a template flag, not a runtime one: the first micro-step's
// instance holds no registers for accumulator loads it never makes.  That
// micro-step writes twice the bytes it reads (bf16 in, fp32 out), and it
// runs one CTA per SM: measured over 2 x 256 M elements, 6321-6347 GB/s
// against 5131-5154 with two CTAs per SM and 5429-5498 with 16 or 4 vectors
// in flight per thread (fewer concurrent write streams suit the DRAM).
template <int kAccumIlp, bool kFirst>
__global__ void __launch_bounds__(kStepThreads, 1) accumulate_vec_kernel(const __grid_constant__ AccumArgs a) {
  const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  const long long nvec = a.n / kVec;
  for (int r = 0; r < a.n_ranks; ++r) {
    const uint4* micro = reinterpret_cast<const uint4*>(a.micro[r]);
    float* acc = a.acc[r];
    long long vi = first_index(tid, static_cast<long long>(r) * nvec, stride);
    for (; vi + (kAccumIlp - 1) * stride < nvec; vi += kAccumIlp * stride) {
      uint4 raw[kAccumIlp];
      float4 x[kAccumIlp][2];
#pragma unroll
      for (int u = 0; u < kAccumIlp; ++u) {
        raw[u] = ld_stream(micro + vi + u * stride);
        if constexpr (!kFirst) {
          const float* p = acc + (vi + u * stride) * kVec;
          x[u][0] = ld_stream_f4(p);
          x[u][1] = ld_stream_f4(p + 4);
        } else {
          x[u][0] = x[u][1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int u = 0; u < kAccumIlp; ++u) accumulate8(raw[u], x[u][0], x[u][1], kFirst, acc + (vi + u * stride) * kVec);
    }
    for (; vi < nvec; vi += stride) {
      float* p = acc + vi * kVec;
      const uint4 raw = ld_stream(micro + vi);
      float4 x0 = make_float4(0.f, 0.f, 0.f, 0.f), x1 = x0;
      if constexpr (!kFirst) {
        x0 = ld_stream_f4(p);
        x1 = ld_stream_f4(p + 4);
      }
      accumulate8(raw, x0, x1, kFirst, p);
    }
    // ragged end of this replica (fewer than 8 elements)
    const long long k = nvec * kVec + (tid - static_cast<long long>(r) * kVec);
    if (tid >= static_cast<long long>(r) * kVec && tid < static_cast<long long>(r + 1) * kVec && k < a.n) {
      const float g = __uint_as_float(static_cast<uint32_t>(a.micro[r][k]) << 16);
      acc[k] = kFirst ? g : __fadd_rn(acc[k], g);
    }
  }
}

__global__ void __launch_bounds__(kStepThreads) accumulate_scalar_kernel(const __grid_constant__ AccumArgs a) {
  const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (int r = 0; r < a.n_ranks; ++r) {
    for (long long k = first_index(tid, static_cast<long long>(r) * a.n, stride); k < a.n; k += stride) {
      const float g = __uint_as_float(static_cast<uint32_t>(a.micro[r][k]) << 16);
      a.acc[r][k] = a.first ? g : __fadd_rn(a.acc[r][k], g);
    }
  }
}

// ---------------------------------------------------------------------------
// make_master and gather.
// ---------------------------------------------------------------------------
__global__ void zero_fill_kernel(float* __restrict__ master, float* __restrict__ m, float* __restrict__ v,
                                 uint16_t* __restrict__ p16, long long n) {
  const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  const long long n8 = n / 8;
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  for (long long i = tid; i < n8; i += stride) {
    reinterpret_cast<uint4*>(master)[2 * i] = z;
    reinterpret_cast<uint4*>(master)[2 * i + 1] = z;
    reinterpret_cast<uint4*>(m)[2 * i] = z;
    reinterpret_cast<uint4*>(m)[2 * i + 1] = z;
    reinterpret_cast<uint4*>(v)[2 * i] = z;
    reinterpret_cast<uint4*>(v)[2 * i + 1] = z;
    reinterpret_cast<uint4*>(p16)[i] = z;
  }
  for (long long k = n8 * 8 + tid; k < n; k += stride) {
    master[k] = 0.0f;
    m[k] = 0.0f;
    v[k] = 0.0f;
    p16[k] = 0;
  }
}

__global__ void copy_param_kernel(const float* __restrict__ src, float* __restrict__ master,
                                  uint16_t* __restrict__ p16, long long offset, long long n) {
  const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long k = tid; k < n; k += stride) {
    const float x = src[k];
    if (master) master[offset + k] = x;  // no device master in an offload context
    p16[offset + k] = to_bf16_bits(x);
  }
}

__global__ void copy_f32_kernel(const float* __restrict__ src, float* __restrict__ dst, long long n) {
  const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long k = tid; k < n; k += stride) dst[k] = src[k];
}

// One 16-byte vector per thread over a grid covering the unit (no grid-
// stride loop) with plain loads and stores: measured as the fastest of the
// copy variants tried — on 800 MB 6566 GB/s against 6353-6404 for a
// persistent 8-CTA-per-SM grid with streaming hints (cudaMemcpyAsync: 6621).
__device__ __forceinline__ void gather_vec_body(const uint4* __restrict__ src, uint4* __restrict__ dst, long long n16,
                                                long long i) {
  if (i < n16) dst[i] = src[i];
}

// Units that are not 16-byte aligned on both sides, or not a whole number
// of vectors (a unit's flat base is not a multiple of 8 when padding to a
// multiple of N moved it, CMU 15-779 Lecture 13 notes §3.6): the first
// `head` elements are copied one by one so that the destination is aligned
// from there on; thread i then writes destination vector i, built from the
// two aligned source words that hold its elements, shifted by phi elements
// (the second word starts inside the unit: its first phi elements are the
// vector's last).  The second word is also the next thread's first: the
// duplicate request is served on chip (measured 3-4 % faster than passing
// it between lanes by warp shuffle).  The threads after the last vector
// copy the head and the ragged tail.
__device__ __forceinline__ void gather_shift_body(const uint16_t* __restrict__ src, uint16_t* __restrict__ dst,
                                                  long long n, int head, int phi, long long nvec, long long i) {
  const bool active = i < nvec;
  const uint4* words = reinterpret_cast<const uint4*>(src + head - phi);  // 16-byte aligned
  uint4 w0 = make_uint4(0u, 0u, 0u, 0u), w1 = make_uint4(0u, 0u, 0u, 0u);
  if (active && ZFS_CHECK(head + 8 * i + 8 <= n)) {
    w0 = words[i];
    if (phi != 0) w1 = words[i + 1];
  }
  if (active && ZFS_CHECK(head + 8 * i + 8 <= n)) {
    uint4 out = w0;
    if (phi != 0) {
      const uint32_t u[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
      const int k = phi >> 1;
      uint32_t t[6], v[5];
#pragma unroll
      for (int q = 0; q < 6; ++q) t[q] = (k & 2) ? u[q + 2] : u[q];
#pragma unroll
      for (int q = 0; q < 5; ++q) v[q] = (k & 1) ? t[q + 1] : t[q];
      const uint32_t sh = static_cast<uint32_t>(phi & 1) * 16;
      out = make_uint4(__funnelshift_r(v[0], v[1], sh), __funnelshift_r(v[1], v[2], sh),
                       __funnelshift_r(v[2], v[3], sh), __funnelshift_r(v[3], v[4], sh));
    }
    reinterpret_cast<uint4*>(dst + head)[i] = out;
  }
  const long long q = i - nvec;  // head and tail: at most 7 + 7 elements
  if (q >= 0 && q < 16) {
    const long long k = q < head ? q : head + 8 * nvec + (q - head);
    if ((q < head || q - head < 8) && k < n) dst[k] = src[k];
  }
}

// The gathers are overlapped launches (see await_previous_grid).
__global__ void gather_vec_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, long long n16) {
  await_previous_grid();
  gather_vec_body(src, dst, n16, static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x);
}

__global__ void gather_shift_kernel(const uint16_t* __restrict__ src, uint16_t* __restrict__ dst, long long n,
                                    int head, int phi, long long nvec) {
  await_previous_grid();
  gather_shift_body(src, dst, n, head, phi, nvec, static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x);
}

// Several units in one launch (a prefetch of the next units, the way ZeRO-3
// implementations gather more than one module's parameters ahead of use):
// unit u owns CTAs [cta_begin[u], cta_begin[u+1]), so every CTA stays within
// one unit (its branch between the bodies is uniform); aligned units take
// the vector body, the others the shifted one.  One launch instead of one per unit spares the
// ramp and drain between consecutive copies.
__global__ void __launch_bounds__(kStepThreads) gather_units_kernel(const __grid_constant__ GatherBatch b) {
  await_previous_grid();
  const long long blk = blockIdx.x;
  int lo = 0, hi = b.count - 1;  // the last unit with cta_begin <= blk
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (b.cta_begin[mid] <= blk) lo = mid; else hi = mid - 1;
  }
  const GatherUnit& g = b.unit[lo];
  const long long i = (blk - b.cta_begin[lo]) * blockDim.x + threadIdx.x;
  if (g.shifted) {
    gather_shift_body(g.src, g.dst, g.n, g.head, g.phi, g.nvec, i);
  } else {
    gather_vec_body(reinterpret_cast<const uint4*>(g.src), reinterpret_cast<uint4*>(g.dst), g.nvec, i);
  }
}

// ---------------------------------------------------------------------------
// ZeRO-Offload: reduced gradient of one chunk, written for the host.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float reduce_one(const ReduceArgs& a, const ReduceSeg& s, long long k) {
  float acc;
  if (a.grad_fp32) {
    acc = __ldcs(static_cast<const float*>(s.g[0]) + k);
    for (int r = 1; r < a.n_ranks; ++r) acc = __fadd_rn(acc, __ldcs(static_cast<const float*>(s.g[r]) + k));
  } else {
    acc = __uint_as_float(static_cast<uint32_t>(__ldcs(static_cast<const unsigned short*>(s.g[0]) + k)) << 16);
    for (int r = 1; r < a.n_ranks; ++r) {
      acc = __fadd_rn(acc, __uint_as_float(static_cast<uint32_t>(__ldcs(static_cast<const unsigned short*>(s.g[r]) + k)) << 16));
    }
  }
  return acc;
}

__global__ void __launch_bounds__(kStepThreads) reduce_out_kernel(const __grid_constant__ ReduceArgs a) {
  const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  const float clip = a.clip ? *a.clip : 1.0f;
  unsigned nf = 0;  // non-finite reduced gradients seen by this thread
  int s = 0;
  for (long long q = tid; q < a.total_groups; q += stride) {
    while (s + 1 < a.nseg && q >= a.seg[s + 1].group_start) ++s;
    const ReduceSeg& sg = a.seg[s];
    const long long k = (q - sg.group_start) * kVec;
    float* out = a.out + sg.out_off + k;
    if (!ZFS_CHECK(k >= 0 && k < sg.len && sg.out_off + (k + kVec < sg.len ? k + kVec : sg.len) <= a.out_len)) {
      continue;
    }
    if (sg.vec_ok && k + kVec <= sg.len) {
      float acc[kVec];
      for (int r = 0; r < a.n_ranks; ++r) {
        float x[kVec];
        if (a.grad_fp32) {
          const float* gp = static_cast<const float*>(sg.g[r]) + k;
          const float4 lo = ld_stream_f4(gp), hi = ld_stream_f4(gp + 4);
          x[0] = lo.x; x[1] = lo.y; x[2] = lo.z; x[3] = lo.w;
          x[4] = hi.x; x[5] = hi.y; x[6] = hi.z; x[7] = hi.w;
        } else {
          const uint4 h = ld_stream(static_cast<const uint16_t*>(sg.g[r]) + k);
          x[0] = bf16_lo(h.x); x[1] = bf16_hi(h.x); x[2] = bf16_lo(h.y); x[3] = bf16_hi(h.y);
          x[4] = bf16_lo(h.z); x[5] = bf16_hi(h.z); x[6] = bf16_lo(h.w); x[7] = bf16_hi(h.w);
        }
#pragma unroll
        for (int e = 0; e < kVec; ++e) acc[e] = r == 0 ? x[e] : __fadd_rn(acc[e], x[e]);
      }
      nf += tally_nonfinite<kVec>(acc);
#pragma unroll
      for (int e = 0; e < kVec; ++e) acc[e] = __fmul_rn(__fmul_rn(acc[e], a.inv_n), clip);
      st_stream_f4(out, make_float4(acc[0], acc[1], acc[2], acc[3]));
      st_stream_f4(out + 4, make_float4(acc[4], acc[5], acc[6], acc[7]));
    } else {
      const long long end = k + kVec < sg.len ? k + kVec : sg.len;
      for (long long e = k; e < end; ++e) {
        const float r = reduce_one(a, sg, e);
        nf += tally_nonfinite<1>(&r);
        out[e - k] = __fmul_rn(__fmul_rn(r, a.inv_n), clip);
      }
    }
  }
  flush_nonfinite(a.nonfinite, nf);
}

}  // namespace

unsigned int aux_debug_failures() {
#ifdef ZFS_DEBUG_CHECKS
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_debug_failures, sizeof v) != cudaSuccess) return 0xFFFFFFFFu;
  return v;
#else
  return 0;
#endif
}

cudaError_t launch_reduce_out(const ReduceArgs& a, cudaStream_t stream) {
  if (a.total_groups <= 0 || a.nseg <= 0) return cudaSuccess;
  const long long grid = grid_for(a.total_groups, sm_count(), 8);
  reduce_out_kernel<<<static_cast<unsigned>(grid), kStepThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

using NormKernel = void (*)(NormArgs);

template <bool kFp32, bool kShifted>
NormKernel norm_kernel_for(int n) {
  switch (n) {
    case 1: return grad_sq_kernel<1, kFp32, kShifted>;
    case 2: return grad_sq_kernel<2, kFp32, kShifted>;
    case 3: return grad_sq_kernel<3, kFp32, kShifted>;
    case 4: return grad_sq_kernel<4, kFp32, kShifted>;
    case 5: return grad_sq_kernel<5, kFp32, kShifted>;
    case 6: return grad_sq_kernel<6, kFp32, kShifted>;
    case 7: return grad_sq_kernel<7, kFp32, kShifted>;
    case 8: return grad_sq_kernel<8, kFp32, kShifted>;
    case 9: return grad_sq_kernel<9, kFp32, kShifted>;
    case 10: return grad_sq_kernel<10, kFp32, kShifted>;
    case 11: return grad_sq_kernel<11, kFp32, kShifted>;
    case 12: return grad_sq_kernel<12, kFp32, kShifted>;
    case 13: return grad_sq_kernel<13, kFp32, kShifted>;
    case 14: return grad_sq_kernel<14, kFp32, kShifted>;
    case 15: return grad_sq_kernel<15, kFp32, kShifted>;
    case 16: return grad_sq_kernel<16, kFp32, kShifted>;
    default: return nullptr;
  }
}

cudaError_t launch_grad_sq(const NormArgs& a, long long chunks, bool shifted, cudaStream_t stream) {
  if (chunks <= 0) return cudaSuccess;
  NormKernel k = shifted ? (a.grad_fp32 ? norm_kernel_for<true, true>(a.n_ranks) : norm_kernel_for<false, true>(a.n_ranks))
                         : (a.grad_fp32 ? norm_kernel_for<true, false>(a.n_ranks) : norm_kernel_for<false, false>(a.n_ranks));
  if (!k) return cudaErrorInvalidValue;
  return launch_overlapped(k, chunks, kStepThreads, stream, a);
}

cudaError_t launch_clip_finalize(void* workspace, long long n_partials, float max_norm, cudaStream_t stream) {
  return launch_overlapped(clip_finalize_kernel, 1, kFinalizeThreads, stream, static_cast<char*>(workspace),
                           n_partials, max_norm);
}

cudaError_t launch_accumulate(const AccumArgs& a, bool vec, cudaStream_t stream) {
  if (a.n <= 0 || a.n_ranks <= 0) return cudaSuccess;
  const int sms = sm_count();
  if (vec) {
    long long work = (a.n / kVec) * a.n_ranks;
    if (work < static_cast<long long>(a.n_ranks) * kVec) work = static_cast<long long>(a.n_ranks) * kVec;
    const long long grid = grid_for(work, sms, kStepCtasPerSm);
    if (a.first) {
      const long long grid1 = grid_for(work, sms, 1);
      accumulate_vec_kernel<kAccumIlpFirst, true><<<static_cast<unsigned>(grid1), kStepThreads, 0, stream>>>(a);
    } else {
      accumulate_vec_kernel<kAccumIlpLater, false><<<static_cast<unsigned>(grid), kStepThreads, 0, stream>>>(a);
    }
  } else {
    const long long grid = grid_for(a.n * a.n_ranks, sms, 8);
    accumulate_scalar_kernel<<<static_cast<unsigned>(grid), kStepThreads, 0, stream>>>(a);
  }
  return cudaGetLastError();
}

cudaError_t launch_zero_fill(float* master, float* m, float* v, uint16_t* p16, long long n,
                             cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  const long long grid = grid_for(n / 8 + 1, sm_count(), 8);
  zero_fill_kernel<<<static_cast<unsigned>(grid), kStepThreads, 0, stream>>>(master, m, v, p16, n);
  return cudaGetLastError();
}

cudaError_t launch_copy_param(const float* src, float* master, uint16_t* p16, long long offset,
                              long long n, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  const long long grid = grid_for(n, sm_count(), 8);
  copy_param_kernel<<<static_cast<unsigned>(grid), kStepThreads, 0, stream>>>(src, master, p16, offset, n);
  return cudaGetLastError();
}

cudaError_t launch_copy_f32(const float* src, float* dst, long long n, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  const long long grid = grid_for(n, sm_count(), 8);
  copy_f32_kernel<<<static_cast<unsigned>(grid), kStepThreads, 0, stream>>>(src, dst, n);
  return cudaGetLastError();
}

namespace {

// How one unit is copied: the vector body when source and destination are
// 16-byte aligned and the unit is whole vectors, else the shifted body.
GatherUnit plan_gather(const uint16_t* src, uint16_t* dst, long long n) {
  GatherUnit g{};
  g.src = src;
  g.dst = dst;
  g.n = n;
  const bool aligned = (reinterpret_cast<uintptr_t>(src) % 16 == 0) && (reinterpret_cast<uintptr_t>(dst) % 16 == 0);
  if (aligned && n % 8 == 0) {
    g.nvec = n / 8;
    g.threads = g.nvec;
  } else {
    // the destination aligned after `head` elements; the source's offset
    // from a 16-byte boundary there, in elements
    const long long head =
        std::min<long long>(n, (8 - static_cast<long long>(reinterpret_cast<uintptr_t>(dst) / 2 % 8)) % 8);
    g.shifted = 1;
    g.head = static_cast<int>(head);
    g.phi = static_cast<int>(reinterpret_cast<uintptr_t>(src + head) / 2 % 8);
    g.nvec = (n - head) / 8;
    g.threads = g.nvec + 2 * kVec;  // the head and tail threads after the vectors
  }
  return g;
}

}  // namespace

cudaError_t launch_gather(const uint16_t* src, uint16_t* dst, long long n, cudaStream_t stream, int* launches) {
  if (n <= 0) return cudaSuccess;
  const GatherUnit g = plan_gather(src, dst, n);
  // one thread per vector: under 2^31 blocks for any unit a device can hold
  const long long grid = (g.threads + kStepThreads - 1) / kStepThreads;
  const cudaError_t e =
      !g.shifted ? launch_overlapped(gather_vec_kernel, grid, kStepThreads, stream, reinterpret_cast<const uint4*>(src),
                                     reinterpret_cast<uint4*>(dst), g.nvec)
                 : launch_overlapped(gather_shift_kernel, grid, kStepThreads, stream, src, dst, n, g.head, g.phi,
                                     g.nvec);
  if (e == cudaSuccess) ++*launches;
  return e;
}

cudaError_t launch_gather_units(const uint16_t* const* src, uint16_t* const* dst, const long long* n, int count,
                                cudaStream_t stream, int* launches) {
  GatherBatch b{};
  auto flush = [&]() -> cudaError_t {
    if (b.count == 0) return cudaSuccess;
    const long long grid = b.cta_begin[b.count];
    const cudaError_t e = launch_overlapped(gather_units_kernel, grid, kStepThreads, stream, b);
    if (e == cudaSuccess) ++*launches;
    b = GatherBatch{};
    return e;
  };
  for (int k = 0; k < count; ++k) {
    if (n[k] <= 0) continue;
    const GatherUnit g = plan_gather(src[k], dst[k], n[k]);
    const long long ctas = (g.threads + kStepThreads - 1) / kStepThreads;
    if (b.count == kMaxGatherUnits || b.cta_begin[b.count] + ctas > kMaxGatherCtas) {
      const cudaError_t e = flush();
      if (e != cudaSuccess) return e;
    }
    b.unit[b.count] = g;
    b.cta_begin[b.count + 1] = b.cta_begin[b.count] + ctas;
    ++b.count;
  }
  return flush();
}

}  // namespace zfs
