// Internal interface between the host runtime (zero_runtime.cpp) and the
// sm_103a kernels (zero_step_kernels.cu, zero_aux_kernels.cu).  Not part of
// the public ABI.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

namespace zfs {

constexpr int kMaxRanks = 16;     // N simulated data-parallel replicas
constexpr int kMaxSegs = 48;      // gradient segments per step launch
constexpr int kVec = 8;           // elements per thread-iteration (16 B of bf16)
constexpr int kStepThreads = 256; // threads per CTA of the step kernels
constexpr int kStepCtasPerSm = 2; // resident CTAs per SM of the vector step kernel

// A run of consecutive flat elements whose N replica gradients are
// contiguous buffers: element base + k reads g[r][k].
struct Seg {
  long long base;        // flat element offset
  long long len;         // elements
  long long vec_start;   // index of this segment's first vector in the
                         // concatenated vector space of the launch
  const void* g[kMaxRanks];
};

// Everything one step launch needs, passed by value as a __grid_constant__
// kernel parameter (no device-side tables, nothing to allocate).
struct StepArgs {
  float* master;
  float* m;
  float* v;
  uint16_t* p16;         // bf16 bit patterns
  float inv_n;           // 1 / N
  float lr;
  float beta1;
  float beta2;
  float omb1;            // 1 - beta1
  float omb2;            // 1 - beta2
  float eps;
  float bc1;             // 1 - beta1^t
  float bc2;             // 1 - beta2^t
  float decay;           // 1 - lr * wd  (exactly 1 for plain Adam)
  int n_ranks;
  int grad_fp32;         // 0 = bf16 grads, 1 = fp32 grads
  int nseg;
  long long total_vec;   // vectors over all segments (vector kernel)
  long long total_elems; // elements over all segments (scalar kernel)
  const float* clip;     // device clip coefficient, or nullptr (no clipping)
  Seg seg[kMaxSegs];
};

// Global-norm clipping.  The squared norm of the reduced gradient is summed
// over fixed unit-relative chunks of kClipChunk elements (the last chunk of a
// unit also takes the unit's zero pads), each chunk in a fixed order, then
// the chunk sums in chunk order: the result does not depend on the stage
// (padding) or on how the grid is scheduled.
constexpr long long kClipChunk = 16384;
constexpr int kFinalizeThreads = 1024;

// Workspace layout: [0] double norm, [8] float coefficient, [32..] double chunk partials.
constexpr long long kClipHeaderBytes = 32;

struct NormSeg {
  long long len;          // padded unit length (elements)
  long long n_chunks;     // chunks of this unit
  long long chunk_start;  // first chunk's index within this launch
  long long out_start;    // first chunk's index in the workspace partials
  int vec_ok;             // 16-byte aligned gradients: vector loads allowed
  const void* g[kMaxRanks];
};

struct NormArgs {
  int n_ranks;
  int grad_fp32;
  float inv_n;
  int nseg;
  double* partials;
  NormSeg seg[kMaxSegs];
};

// Norm pass: one CTA per chunk; writes one partial per chunk.
cudaError_t launch_grad_sq(const NormArgs& a, long long chunks, cudaStream_t stream);
// Sums n partials in a fixed order and writes the norm and the clip
// coefficient min(1, max_norm / (norm + 1e-6)) into the workspace header.
cudaError_t launch_clip_finalize(void* workspace, long long n_partials, float max_norm, cudaStream_t stream);

// Launchers.  Each returns the cudaError_t of its launch.
// Vector kernel: every segment has base % kVec == 0 and 16-byte aligned
// gradient pointers; the last kVec-1 elements of a segment may be ragged.
cudaError_t launch_step_vec(const StepArgs& a, cudaStream_t stream);
// Scalar kernel: any alignment (used for segments the vector kernel cannot take).
cudaError_t launch_step_scalar(const StepArgs& a, cudaStream_t stream);

// make_master pieces.
cudaError_t launch_zero_fill(float* master, float* m, float* v, uint16_t* p16, long long n,
                             cudaStream_t stream);
cudaError_t launch_copy_param(const float* src, float* master, uint16_t* p16, long long offset,
                              long long n, cudaStream_t stream);
// Plain fp32 copy of n elements (checkpoint export/import).
cudaError_t launch_copy_f32(const float* src, float* dst, long long n, cudaStream_t stream);

// fp32 gradient accumulation of one micro-step: for every replica r,
// acc[r][j] = (first ? 0 : acc[r][j]) + widen(micro[r][j]), j < n.
struct AccumArgs {
  int n_ranks;
  int first;
  long long n;
  const uint16_t* micro[kMaxRanks];
  float* acc[kMaxRanks];
};
cudaError_t launch_accumulate(const AccumArgs& a, bool vec, cudaStream_t stream);

// ZeRO-3 unit gather: copy n bf16 elements; *launches counts the kernels enqueued.
cudaError_t launch_gather(const uint16_t* src, uint16_t* dst, long long n, cudaStream_t stream, int* launches);

// Multiprocessor count of the current device (cached per device).
int sm_count();

// CTAs for a grid-stride launch of kStepThreads-thread CTAs over work_items
// items: enough to cover them, at most blocks_per_sm per SM.
long long grid_for(long long work_items, int sms, int blocks_per_sm);

}  // namespace zfs

struct zero_ctx;
// Records `message` as the context's last error (or the calling thread's when
// ctx is NULL) and returns `status`.  Defined by the host runtime.
int zfs_report_error(zero_ctx* ctx, int status, const char* message);
