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
// Tile-staged (TMA bulk copy) step kernels: used for launches of at least
// kTmaMinElems elements with bf16 replicas N = 1..4 or N >= 7 and fp32
// replicas N >= 7 (the rank counts where they measured faster).
constexpr long long kTmaMinElems = 1LL << 23;
constexpr long long kTmaTile = 2048; // elements per tile (one 8-element vector per thread)
constexpr int kTmaStages = 2;        // tiles in flight per CTA

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
  long long total_padded;  // elements of master / m / v / p16 (debug bounds checks)
  // Capturable steps (dev_t != nullptr): the step count before this step is
  // *dev_t, and bc1 / bc2 of step t are dev_bias[2(t-1)], dev_bias[2(t-1)+1]
  // for t <= dev_steps (instead of the bc1 / bc2 above).
  const long long* dev_t;
  const float* dev_bias;
  long long dev_steps;
  unsigned long long* nonfinite;  // caller's counter of non-finite reduced
                                  // gradients, or nullptr (not counted)
  int inject_missing_copy; // test hook: the tile-staged kernel announces the
                           // launch's first tile but issues none of its copies
  Seg seg[kMaxSegs];
  // Shifted-gradient kernel only: segment s's body starts at seg[s].base (a
  // multiple of kVec), its head[s] < kVec elements before it are the body's
  // elements -head[s] .. -1, and replica r's gradient at the body's start
  // lies gshift[s][r] elements past a 16-byte boundary.
  unsigned char head[kMaxSegs];
  unsigned char gshift[kMaxSegs][kMaxRanks];
};

// Launchers.  Each returns the cudaError_t of its launch.
// Vector kernel: every segment has base % kVec == 0 and 16-byte aligned
// gradient pointers; the last kVec-1 elements of a segment may be ragged.
cudaError_t launch_step_vec(const StepArgs& a, cudaStream_t stream);
// Shifted-gradient kernel: segments of any alignment, described by their
// aligned body, head and per-replica gradient shift (see StepArgs).
cudaError_t launch_step_shift(const StepArgs& a, cudaStream_t stream);

// Multiprocessor count of the current device (cached per device).
int sm_count();

// The unique id of the calling thread's current CUDA context, which the
// driver never reuses within a process; false when no context is current or
// the driver cannot say.  State that belongs to a context rather than to a
// device (a kernel's raised shared-memory limit, the address of a __device__
// object) is cached under it.
bool current_context_id(unsigned long long* id);

// Bounded waits of the tile-staged step kernel that gave up on the current
// device since the library was loaded (0xFFFFFFFF if it cannot be read).
unsigned int step_timeouts();
// Capturable steps: *t += 1 on the stream (one thread).
cudaError_t launch_count_step(long long* t, cudaStream_t stream);
// Failed index checks of a debug build in zero_step_kernels.cu (0xFFFFFFFF
// if the counter cannot be read; always 0 in a release build).
unsigned int step_debug_failures();

// CTAs for a grid-stride launch of kStepThreads-thread CTAs over work_items
// items: enough to cover them, at most blocks_per_sm per SM.
long long grid_for(long long work_items, int sms, int blocks_per_sm);

}  // namespace zfs

struct zero_ctx;
// Records `message` as the context's last error (or the calling thread's when
// ctx is NULL) and returns `status`.  Defined by the host runtime.
int zfs_report_error(zero_ctx* ctx, int status, const char* message);
