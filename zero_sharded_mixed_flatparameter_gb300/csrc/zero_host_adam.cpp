// Host side of ZeRO-Offload: the CPU Adam that updates host-resident fp32
// master / m / v chunk by chunk while the GPU reduces the next chunk's
// gradients.  CMU 15-779 Lecture 13 notes, §7.1-7.2: in ZeRO-Offload's
// partition only the 16-bit parameters stay on the GPU; gradients go down to
// the host, a SIMD + multi-threaded CPU Adam updates the fp32 state, and the
// new 16-bit parameters go back up in chunks, pipelined with the update of
// the next chunk.
//
// Built with -O3 -ffp-contract=off -fno-math-errno and no fast-math: the
// loop vectorizes (division and square root stay correctly rounded IEEE
// operations on every SIMD unit), nothing is fused, so each element gets
// exactly the device step's sequence of rounded fp32 operations.  Portable
// C++ only: no intrinsics, the same source builds for x86-64 and aarch64.

#include "zero_host.h"

#include <cmath>
#include <condition_variable>
#include <cstring>
#include <mutex>
#include <new>
#include <thread>
#include <vector>

namespace zfs_host {

namespace {

// bf16 bits of x, rounded to nearest even; a NaN stays a (quiet) NaN.
inline uint16_t bf16_bits(float x) {
  uint32_t u;
  std::memcpy(&u, &x, sizeof u);
  const uint32_t rounded = (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
  const uint32_t nan = (u >> 16) | 0x0040u;
  return static_cast<uint16_t>((u & 0x7FFFFFFFu) > 0x7F800000u ? nan : rounded);
}

}  // namespace

void adam_range(const AdamScalars& s, const float* __restrict g, float* __restrict w, float* __restrict m,
                float* __restrict v, uint16_t* __restrict p16, int64_t n) {
  const float lr = s.lr, beta1 = s.beta1, beta2 = s.beta2, omb1 = s.omb1, omb2 = s.omb2;
  const float eps = s.eps, bc1 = s.bc1, bc2 = s.bc2, decay = s.decay;
  for (int64_t j = 0; j < n; ++j) {
    const float gj = g[j];
    const float wd = w[j] * decay;
    const float mj = beta1 * m[j] + omb1 * gj;
    const float vj = beta2 * v[j] + omb2 * (gj * gj);
    const float m_hat = mj / bc1;
    const float v_hat = vj / bc2;
    const float denom = std::sqrt(v_hat) + eps;
    const float wj = wd - lr * (m_hat / denom);
    w[j] = wj;
    m[j] = mj;
    v[j] = vj;
    p16[j] = bf16_bits(wj);
  }
}

class Pool {
 public:
  explicit Pool(int threads) : threads_(threads < 1 ? 1 : threads) {}

  bool start() {
    try {
      for (int i = 1; i < threads_; ++i) workers_.emplace_back([this, i] { loop(i); });
    } catch (...) {
      stop();
      return false;
    }
    return true;
  }

  ~Pool() { stop(); }

  int threads() const { return threads_; }

  void run(int64_t n, const std::function<void(int64_t, int64_t)>& fn) {
    if (n <= 0) return;
    {
      std::lock_guard<std::mutex> lock(mu_);
      fn_ = &fn;
      n_ = n;
      pending_ = static_cast<int>(workers_.size());
      ++generation_;
    }
    wake_.notify_all();
    part(0);
    std::unique_lock<std::mutex> lock(mu_);
    done_.wait(lock, [this] { return pending_ == 0; });
    fn_ = nullptr;
  }

 private:
  void part(int i) const {
    // 64-element (256 B of fp32) aligned parts: no two threads share a cache line.
    const int64_t per = ((n_ + threads_ - 1) / threads_ + 63) / 64 * 64;
    const int64_t lo = per * i;
    const int64_t hi = lo + per < n_ ? lo + per : n_;
    if (lo < hi) (*fn_)(lo, hi);
  }

  void loop(int i) {
    uint64_t seen = 0;
    for (;;) {
      {
        std::unique_lock<std::mutex> lock(mu_);
        wake_.wait(lock, [&] { return generation_ != seen || stopping_; });
        if (stopping_) return;
        seen = generation_;
      }
      part(i);
      {
        std::lock_guard<std::mutex> lock(mu_);
        if (--pending_ == 0) done_.notify_one();
      }
    }
  }

  void stop() {
    {
      std::lock_guard<std::mutex> lock(mu_);
      stopping_ = true;
    }
    wake_.notify_all();
    for (std::thread& t : workers_) t.join();
    workers_.clear();
  }

  const int threads_;
  std::vector<std::thread> workers_;
  std::mutex mu_;
  std::condition_variable wake_, done_;
  const std::function<void(int64_t, int64_t)>* fn_ = nullptr;
  int64_t n_ = 0;
  int pending_ = 0;
  uint64_t generation_ = 0;
  bool stopping_ = false;
};

Pool* pool_create(int threads) {
  Pool* p = new (std::nothrow) Pool(threads);
  if (p && !p->start()) {
    delete p;
    return nullptr;
  }
  return p;
}

void pool_destroy(Pool* pool) { delete pool; }

int pool_threads(const Pool* pool) { return pool ? pool->threads() : 0; }

void pool_run(Pool* pool, int64_t n, const std::function<void(int64_t, int64_t)>& fn) { pool->run(n, fn); }

}  // namespace zfs_host
