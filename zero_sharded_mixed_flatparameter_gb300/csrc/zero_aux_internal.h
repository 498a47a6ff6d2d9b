// Internal interface of the auxiliary kernels (zero_aux_kernels.cu): the
// clip norm pass, fp32 gradient accumulation, make_master / checkpoint
// copies and the ZeRO-3 gather.  Not part of the public ABI.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

#include "zero_internal.h"

namespace zfs {

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
  // Otherwise replica r's gradient starts shift[r] elements past a 16-byte
  // boundary: vector loads of aligned words, shifted into place.
  unsigned char shift[kMaxRanks];
  float* keep;            // where to store this unit's reduced gradient, or nullptr
  int keep_vec;           // keep is 16-byte aligned: vector stores allowed
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

// Norm pass: one CTA per chunk; writes one partial per chunk.  `shifted`:
// every segment of the launch has vec_ok == 0 (unaligned gradients; the
// instances with shifted loads); otherwise every segment has vec_ok == 1.
cudaError_t launch_grad_sq(const NormArgs& a, long long chunks, bool shifted, cudaStream_t stream);
// Sums n partials in a fixed order and writes the norm and the clip
// coefficient min(1, max_norm / (norm + 1e-6)) into the workspace header (NaN
// when the norm is NaN).
cudaError_t launch_clip_finalize(void* workspace, long long n_partials, float max_norm, cudaStream_t stream);

// make_master pieces.
cudaError_t launch_zero_fill(float* master, float* m, float* v, uint16_t* p16, long long n,
                             cudaStream_t stream);
// master[offset + k] = src[k] (skipped when master is nullptr) and
// p16[offset + k] = bf16(src[k]), k < n.
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

// ZeRO-Offload: the reduced gradient of one chunk of the flat buffer,
// out[out_off + k] = ((G_0 + G_1) + ... + G_{N-1})[k] * fp32(1/N) * clip for
// k < len of every segment (clip = 1 without a pending clip), for the host
// Adam to read.  Segments are walked as one index space of 8-element groups.
struct ReduceSeg {
  long long out_off;      // element offset of this segment in out
  long long len;          // elements
  long long group_start;  // first 8-element group of this segment in the launch
  int vec_ok;             // gradients and out + out_off 16-byte aligned
  const void* g[kMaxRanks];
};

struct ReduceArgs {
  unsigned long long* nonfinite;  // caller's overflow counter, or nullptr
  float* out;
  long long out_len;  // elements of out (debug bounds checks)
  const float* clip;  // device clip coefficient, or nullptr
  float inv_n;
  int n_ranks;
  int grad_fp32;
  int nseg;
  long long total_groups;
  ReduceSeg seg[kMaxSegs];
};
cudaError_t launch_reduce_out(const ReduceArgs& a, cudaStream_t stream);

// Failed index checks of a debug build in zero_aux_kernels.cu (0xFFFFFFFF if
// the counter cannot be read; always 0 in a release build).
unsigned int aux_debug_failures();

// ZeRO-3 unit gather: copy n bf16 elements; *launches counts the kernels enqueued.
cudaError_t launch_gather(const uint16_t* src, uint16_t* dst, long long n, cudaStream_t stream, int* launches);

// Several unit gathers in as few launches as the batch limits allow.
constexpr int kMaxGatherUnits = 32;
constexpr long long kMaxGatherCtas = 0x7fffffffLL;  // grid.x limit
struct GatherUnit {
  const uint16_t* src;
  uint16_t* dst;
  long long n;        // elements
  long long nvec;     // 16-byte destination vectors (after the head when shifted)
  long long threads;  // threads the unit's CTAs cover
  int shifted;        // 0: aligned vector copy; 1: head + shifted vectors + tail
  int head;           // shifted: elements before the destination is aligned
  int phi;            // shifted: source offset from a 16-byte boundary there, in elements
};
struct GatherBatch {
  int count;
  long long cta_begin[kMaxGatherUnits + 1];
  GatherUnit unit[kMaxGatherUnits];
};
cudaError_t launch_gather_units(const uint16_t* const* src, uint16_t* const* dst, const long long* n, int count,
                                cudaStream_t stream, int* launches);

}  // namespace zfs
