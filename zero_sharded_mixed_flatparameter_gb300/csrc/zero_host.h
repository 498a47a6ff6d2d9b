// Internal interface of the host side of ZeRO-Offload (zero_host_adam.cpp):
// the CPU Adam over host-resident fp32 state and the worker pool that runs
// it.  Not part of the public ABI.
#pragma once

#include <cstdint>
#include <functional>

namespace zfs_host {

// The fp32 scalars of one Adam / AdamW step, computed on the host exactly as
// for the device step (bias corrections in double, rounded once to fp32).
struct AdamScalars {
  float lr, beta1, beta2, omb1, omb2, eps, bc1, bc2, decay;
};

// Adam / AdamW on n consecutive elements: g is the reduced (and clipped)
// fp32 gradient; w, m, v are updated in place and p16 receives bf16(w)
// rounded to nearest even.  Every operation is one IEEE fp32 operation in
// the device step's order (no contraction), so the results equal the
// device step's bit for bit.
void adam_range(const AdamScalars& s, const float* g, float* w, float* m, float* v, uint16_t* p16, int64_t n);

// A fixed set of worker threads.  run() splits [0, n) into one contiguous,
// 64-element-aligned part per thread (the calling thread takes the first)
// and returns when every part is done.  One run() at a time per pool.
class Pool;
Pool* pool_create(int threads);  // nullptr if the threads cannot be started
void pool_destroy(Pool* pool);
int pool_threads(const Pool* pool);
void pool_run(Pool* pool, int64_t n, const std::function<void(int64_t, int64_t)>& fn);

}  // namespace zfs_host
