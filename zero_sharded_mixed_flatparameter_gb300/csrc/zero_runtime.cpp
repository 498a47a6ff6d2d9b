// Host runtime of the ZeRO flat-parameter library: the C ABI declared in
// include/zero_flatstep.h.  It owns only host metadata — the FlatParameter
// layout, the registered gradient pointers, the step count and error text,
// and an offload context's worker threads — and enqueues the sm_103a kernels
// (zero_step_kernels.cu, zero_aux_kernels.cu) on the caller's stream.
//
// Protocol: Femtotron dev log #6 (ShardingStrategy: make_master /
// reduce_grads / gather_weights / post_step).  Layout: CMU 15-779 Lecture 13
// notes §0.4 and §5.2 (flatten, concatenate, right-pad to a multiple of F,
// split evenly).  Ledger: same notes §2.3, §3.5, §9 item 2, §11 Exercise 5.
// ZeRO-Offload (host-resident fp32 state, CPU Adam): same notes §7.1-7.2.
//
// Sections, in order: context and helpers; planning and make_master (also
// the offload variant); registration; the step; the offload step and the
// stateless CPU Adam; clipping; gather / post_step; checkpoints; queries,
// test hooks and capturable mode.

#include <algorithm>
#include <cmath>
#include <functional>
#include <memory>
#include <mutex>
#include <thread>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>

#include "zero_flatstep.h"
#include "zero_aux_internal.h"
#include "zero_host.h"
#include "zero_internal.h"

namespace {

thread_local std::string g_thread_error;

enum class Phase { kPlanned, kReady, kStepped };

}  // namespace

struct zero_ctx {
  zero_config cfg{};
  int32_t n_units = 0;
  int32_t n_params = 0;
  int64_t shards = 1;  // F
  std::vector<int64_t> unit_numel, unit_padded, unit_shard, unit_base, param_offset;
  int64_t padded_total = 0;
  int64_t numel_total = 0;

  Phase phase = Phase::kPlanned;
  zero_buffers bufs{};
  int device = -1;
  int64_t t = 0;
  int32_t last_launches = 0;

  // Registered replica gradient pointers, n_units x kMaxRanks.
  std::vector<const void*> grads;
  std::vector<uint8_t> registered;

  // Clipping: workspace of the clip pending for the next step (cleared by
  // post_step) and of the last clip run (for zero_grad_norm).
  char* clip_ws = nullptr;
  char* last_clip_ws = nullptr;
  // With ZERO_CLIP_KEEP_REDUCED: the reduced fp32 gradient (padded_total
  // elements) the pending step reads instead of the replicas.
  float* clip_keep = nullptr;

  // ZeRO-Offload: master / m / v are host memory, the step runs through
  // zero_offload_step with this worker pool (created on first use).
  bool offload = false;
  zfs_host::Pool* pool = nullptr;

  // Caller's device counter of non-finite reduced gradients (zero_count_nonfinite), or nullptr.
  unsigned long long* nonfinite = nullptr;

  // Test hook armed by zero_debug_inject for the next step's first launch.
  int32_t inject = 0;

  // Capturable mode: the device step count and the table of bias
  // corrections in the caller's workspace (nullptr when off).
  long long* cap_t = nullptr;
  float* cap_bias = nullptr;
  int64_t cap_steps = 0;

  std::string error;

  ~zero_ctx() { zfs_host::pool_destroy(pool); }
};

namespace {

zero_status fail(zero_ctx* ctx, zero_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  if (ctx) {
    ctx->error = buf;
  } else {
    g_thread_error = buf;
  }
  return st;
}

zero_status fail_cuda(zero_ctx* ctx, const char* what, cudaError_t e) {
  return fail(ctx, ZERO_ECUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t grad_bytes(const zero_config& c) { return c.grad_dtype == ZERO_GRAD_FP32 ? 4 : 2; }

zero_status check_config(const zero_config* cfg, zero_ctx* errctx) {
  if (!cfg) return fail(errctx, ZERO_EINVAL, "config is NULL");
  if (cfg->stage < 0 || cfg->stage > 3) return fail(errctx, ZERO_EINVAL, "stage %d not in 0..3", cfg->stage);
  if (cfg->n_ranks < 1 || cfg->n_ranks > zfs::kMaxRanks)
    return fail(errctx, ZERO_EINVAL, "n_ranks %d not in 1..%d", cfg->n_ranks, zfs::kMaxRanks);
  if (cfg->grad_dtype != ZERO_GRAD_BF16 && cfg->grad_dtype != ZERO_GRAD_FP32)
    return fail(errctx, ZERO_EINVAL, "grad_dtype %d is neither bf16 (0) nor fp32 (1)", cfg->grad_dtype);
  if (cfg->adamw != 0 && cfg->adamw != 1) return fail(errctx, ZERO_EINVAL, "adamw must be 0 or 1");
  if (!std::isfinite(cfg->lr)) return fail(errctx, ZERO_EINVAL, "lr is not finite");
  if (!(cfg->beta1 >= 0.0f && cfg->beta1 < 1.0f)) return fail(errctx, ZERO_EINVAL, "beta1 not in [0, 1)");
  if (!(cfg->beta2 >= 0.0f && cfg->beta2 < 1.0f)) return fail(errctx, ZERO_EINVAL, "beta2 not in [0, 1)");
  if (!(cfg->eps >= 0.0f) || !std::isfinite(cfg->eps)) return fail(errctx, ZERO_EINVAL, "eps must be finite and >= 0");
  if (!std::isfinite(cfg->weight_decay) || cfg->weight_decay < 0.0f)
    return fail(errctx, ZERO_EINVAL, "weight_decay must be finite and >= 0");
  if (!cfg->adamw && cfg->weight_decay != 0.0f)
    return fail(errctx, ZERO_EINVAL, "weight_decay needs adamw = 1 (only decoupled decay is provided)");
  return ZERO_OK;
}

// FlatParameter layout: per unit, numel = sum of its params; padded = the
// smallest multiple of F not below numel; shard = padded / F; base = running
// sum of padded sizes.  Params sit back to back in caller order.
zero_status plan_layout(zero_ctx* ctx, const int64_t* param_numel, const int32_t* param_unit, int32_t n_params) {
  if (n_params < 0) return fail(nullptr, ZERO_EINVAL, "n_params is negative");
  if (n_params > 0 && (!param_numel || !param_unit))
    return fail(nullptr, ZERO_EINVAL, "param_numel / param_unit is NULL");
  int32_t last = 0;
  for (int32_t p = 0; p < n_params; ++p) {
    if (param_numel[p] < 0) return fail(nullptr, ZERO_EINVAL, "param %d has negative numel", p);
    if (param_unit[p] < last) return fail(nullptr, ZERO_EINVAL, "param_unit decreases at param %d", p);
    last = param_unit[p];
  }
  if (n_params > 0 && param_unit[0] < 0) return fail(nullptr, ZERO_EINVAL, "param_unit is negative");
  const int32_t n_units = n_params > 0 ? param_unit[n_params - 1] + 1 : 0;
  const int64_t F = ctx->cfg.stage == 0 ? 1 : ctx->cfg.n_ranks;
  ctx->shards = F;
  ctx->n_units = n_units;
  ctx->n_params = n_params;
  ctx->unit_numel.assign(n_units, 0);
  ctx->unit_padded.assign(n_units, 0);
  ctx->unit_shard.assign(n_units, 0);
  ctx->unit_base.assign(n_units, 0);
  ctx->param_offset.assign(n_params, 0);
  for (int32_t p = 0; p < n_params; ++p) {
    const int64_t before = ctx->unit_numel[param_unit[p]];
    if (before > INT64_MAX / 4 - param_numel[p]) return fail(nullptr, ZERO_EINVAL, "parameter sizes overflow");
    ctx->unit_numel[param_unit[p]] = before + param_numel[p];
  }
  int64_t base = 0, numel = 0;
  for (int32_t i = 0; i < n_units; ++i) {
    const int64_t rem = ctx->unit_numel[i] % F;
    ctx->unit_padded[i] = ctx->unit_numel[i] + (rem ? F - rem : 0);
    ctx->unit_shard[i] = ctx->unit_padded[i] / F;
    ctx->unit_base[i] = base;
    if (base > INT64_MAX / 16 - ctx->unit_padded[i]) return fail(nullptr, ZERO_EINVAL, "parameter sizes overflow");
    base += ctx->unit_padded[i];
    numel += ctx->unit_numel[i];
  }
  ctx->padded_total = base;
  ctx->numel_total = numel;
  int32_t cur = -1;
  int64_t cursor = 0;
  for (int32_t p = 0; p < n_params; ++p) {
    if (param_unit[p] != cur) {
      cur = param_unit[p];
      cursor = ctx->unit_base[cur];
    }
    ctx->param_offset[p] = cursor;
    cursor += param_numel[p];
  }
  ctx->grads.assign(static_cast<size_t>(n_units) * zfs::kMaxRanks, nullptr);
  ctx->registered.assign(n_units, 0);
  return ZERO_OK;
}

bool is_device_pointer(const void* p, int* device) {
  cudaPointerAttributes attr{};
  const cudaError_t e = cudaPointerGetAttributes(&attr, p);
  if (e != cudaSuccess) {
    cudaGetLastError();  // clear the sticky-free error state of this query
    return false;
  }
  if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged) return false;
  if (device) *device = attr.device;
  return true;
}

zero_status check_current_device(zero_ctx* ctx) {
  int dev = -1;
  const cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(ctx, "cudaGetDevice", e);
  if (dev != ctx->device)
    return fail(ctx, ZERO_ESTATE, "current device %d is not the context's device %d", dev, ctx->device);
  return ZERO_OK;
}

zero_status require_bound(zero_ctx* ctx) {
  if (ctx->phase == Phase::kPlanned) return fail(ctx, ZERO_ESTATE, "no buffers bound (context from zero_plan)");
  return check_current_device(ctx);
}

// Scalars of step t, each from its definition (evaluated in double where the
// definition has a power or a product of hyper-parameters, rounded once).
zfs_host::AdamScalars adam_scalars(const zero_config& c, int64_t t) {
  zfs_host::AdamScalars s;
  s.lr = c.lr;
  s.beta1 = c.beta1;
  s.beta2 = c.beta2;
  s.omb1 = 1.0f - c.beta1;
  s.omb2 = 1.0f - c.beta2;
  s.eps = c.eps;
  s.bc1 = static_cast<float>(1.0 - std::pow(static_cast<double>(c.beta1), static_cast<double>(t)));
  s.bc2 = static_cast<float>(1.0 - std::pow(static_cast<double>(c.beta2), static_cast<double>(t)));
  s.decay = c.adamw ? static_cast<float>(1.0 - static_cast<double>(c.lr) * static_cast<double>(c.weight_decay))
                    : 1.0f;
  return s;
}

void fill_scalars(const zero_ctx* ctx, int64_t t, zfs::StepArgs* a) {
  const zero_config& c = ctx->cfg;
  const zfs_host::AdamScalars s = adam_scalars(c, t);
  a->inv_n = 1.0f / static_cast<float>(c.n_ranks);
  a->lr = s.lr;
  a->beta1 = s.beta1;
  a->beta2 = s.beta2;
  a->omb1 = s.omb1;
  a->omb2 = s.omb2;
  a->eps = s.eps;
  a->bc1 = s.bc1;
  a->bc2 = s.bc2;
  a->decay = s.decay;
  a->n_ranks = c.n_ranks;
  a->grad_fp32 = c.grad_dtype == ZERO_GRAD_FP32 ? 1 : 0;
}

struct PlannedSeg {
  int64_t base, len;
  const void* g[zfs::kMaxRanks];
  // Segments for the shifted-gradient kernel: base, len and g describe the
  // aligned body; head elements precede it; shift[r] is replica r's gradient
  // offset from a 16-byte boundary at the body's start, in elements.
  int head = 0;
  unsigned char shift[zfs::kMaxRanks] = {};
};

// One segment per non-empty unit, merged with the previous one when every
// replica's buffer continues exactly where the previous unit's ended (a
// whole-buffer registration becomes a single segment).
std::vector<PlannedSeg> build_segments(const zero_ctx* ctx) {
  const int N = ctx->cfg.n_ranks;
  const size_t esz = grad_bytes(ctx->cfg);
  std::vector<PlannedSeg> out;
  for (int32_t i = 0; i < ctx->n_units; ++i) {
    if (ctx->unit_padded[i] == 0) continue;
    const void* const* g = &ctx->grads[static_cast<size_t>(i) * zfs::kMaxRanks];
    if (!out.empty()) {
      PlannedSeg& prev = out.back();
      bool contiguous = prev.base + prev.len == ctx->unit_base[i];
      for (int r = 0; r < N && contiguous; ++r) {
        contiguous = static_cast<const char*>(prev.g[r]) + prev.len * esz == static_cast<const char*>(g[r]);
      }
      if (contiguous) {
        prev.len += ctx->unit_padded[i];
        continue;
      }
    }
    PlannedSeg s{};
    s.base = ctx->unit_base[i];
    s.len = ctx->unit_padded[i];
    for (int r = 0; r < N; ++r) s.g[r] = g[r];
    out.push_back(s);
  }
  return out;
}

bool vector_ok(const PlannedSeg& s, int N) {
  if (s.base % zfs::kVec != 0) return false;
  for (int r = 0; r < N; ++r)
    if (!aligned(s.g[r], 16)) return false;
  return true;
}

// A segment the aligned kernels cannot take, as the shifted-gradient kernel
// takes it: the first (kVec - base % kVec) % kVec elements become the head,
// so that the body's state arrays are aligned, and each replica's gradient
// offset from a 16-byte boundary at the body's start is recorded.
PlannedSeg peel(const PlannedSeg& s, int N, size_t esz) {
  PlannedSeg out = s;
  const int64_t h = std::min<int64_t>(s.len, (zfs::kVec - s.base % zfs::kVec) % zfs::kVec);
  out.head = static_cast<int>(h);
  out.base = s.base + h;
  out.len = s.len - h;
  for (int r = 0; r < N; ++r) {
    out.g[r] = static_cast<const char*>(s.g[r]) + h * static_cast<int64_t>(esz);
    out.shift[r] = static_cast<unsigned char>((reinterpret_cast<uintptr_t>(out.g[r]) % 16) / esz);
  }
  return out;
}

// Launch one kernel per batch of up to kMaxSegs segments of one kind.
zero_status launch_batches(zero_ctx* ctx, const std::vector<PlannedSeg>& segs, bool vec, int64_t t,
                           cudaStream_t stream, int32_t* launches) {
  const int N = ctx->cfg.n_ranks;
  size_t i = 0;
  while (i < segs.size()) {
    zfs::StepArgs a;
    std::memset(&a, 0, sizeof a);
    a.master = ctx->bufs.master;
    a.m = ctx->bufs.exp_avg;
    a.v = ctx->bufs.exp_avg_sq;
    a.p16 = static_cast<uint16_t*>(ctx->bufs.param16);
    a.clip = ctx->clip_ws ? reinterpret_cast<const float*>(ctx->clip_ws + 8) : nullptr;
    a.nonfinite = ctx->nonfinite;
    fill_scalars(ctx, t, &a);
    a.total_padded = ctx->padded_total;
    a.dev_t = ctx->cap_t;
    a.dev_bias = ctx->cap_bias;
    a.dev_steps = ctx->cap_steps;
    if (ctx->inject == ZERO_INJECT_MISSING_COPY && vec) {
      a.inject_missing_copy = 1;
      ctx->inject = 0;
    }
    if (ctx->inject == ZERO_INJECT_SHORT_BOUNDS) a.total_padded = ctx->padded_total - zfs::kVec;
    long long vecs = 0, elems = 0;
    int n = 0;
    for (; i < segs.size() && n < zfs::kMaxSegs; ++i, ++n) {
      zfs::Seg& s = a.seg[n];
      s.base = segs[i].base;
      s.len = segs[i].len;
      s.vec_start = vecs;
      for (int r = 0; r < N; ++r) s.g[r] = segs[i].g[r];
      a.head[n] = static_cast<unsigned char>(segs[i].head);
      for (int r = 0; r < N; ++r) a.gshift[n][r] = segs[i].shift[r];
      vecs += s.len / zfs::kVec;
      elems += s.len + segs[i].head;
    }
    a.nseg = n;
    a.total_vec = vecs;
    a.total_elems = elems;
    const cudaError_t e = vec ? zfs::launch_step_vec(a, stream) : zfs::launch_step_shift(a, stream);
    if (e != cudaSuccess) return fail_cuda(ctx, "step kernel launch", e);
    ++*launches;
  }
  return ZERO_OK;
}

// Norm chunks of unit i: ceil(numel / C) chunks over the real elements; the
// last one also covers the unit's pads, so the chunking (and the sum) is the
// same with or without padding.
int64_t unit_chunks(const zero_ctx* ctx, int32_t i) {
  if (ctx->unit_padded[i] == 0) return 0;
  const int64_t n = (ctx->unit_numel[i] + zfs::kClipChunk - 1) / zfs::kClipChunk;
  return n > 0 ? n : 1;
}

int64_t total_chunks(const zero_ctx* ctx) {
  int64_t n = 0;
  for (int32_t i = 0; i < ctx->n_units; ++i) n += unit_chunks(ctx, i);
  return n;
}

bool all_registered(const zero_ctx* ctx, int32_t* missing) {
  for (int32_t i = 0; i < ctx->n_units; ++i) {
    if (!ctx->registered[i]) {
      if (missing) *missing = i;
      return false;
    }
  }
  return true;
}

// Length of unit i padded as stage `stage` pads it with this context's N:
// stage 0 (plain data parallelism) does not pad, stages 1-3 pad to a
// multiple of N (CMU 15-779 Lecture 13 notes §3.6).  The ledger of a stage is
// that of this layout run as that stage, whatever the context's own stage.
int64_t padded_as_stage(const zero_ctx* ctx, int32_t i, int32_t stage) {
  const int64_t F = stage == 0 ? 1 : ctx->cfg.n_ranks;
  return (ctx->unit_numel[i] + F - 1) / F * F;
}

}  // namespace

namespace zfs {
namespace {

// Driver calls reached through the runtime's entry-point query, so that the
// library needs no link-time dependency on the driver library.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
std::once_flag g_driver_once;
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;

void load_driver_calls() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
  if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess && fn) {
    g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(fn);
  }
  fn = nullptr;
  q = cudaDriverEntryPointSymbolNotFound;
  if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess && fn) {
    g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(fn);
  }
}

}  // namespace

bool current_context_id(unsigned long long* id) {
  std::call_once(g_driver_once, load_driver_calls);
  if (!g_ctx_get_current || !g_ctx_get_id) return false;
  CUcontext ctx = nullptr;
  if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
  return g_ctx_get_id(ctx, id) == CUDA_SUCCESS;
}

}  // namespace zfs

int zfs_report_error(zero_ctx* ctx, int status, const char* message) {
  return fail(ctx, static_cast<zero_status>(status), "%s", message);
}

extern "C" {

zero_status zero_plan(const zero_config* cfg, const int64_t* param_numel, const int32_t* param_unit,
                      int32_t n_params, zero_ctx** out) {
  if (!out) return fail(nullptr, ZERO_EINVAL, "out is NULL");
  *out = nullptr;
  zero_status st = check_config(cfg, nullptr);
  if (st != ZERO_OK) return st;
  zero_ctx* ctx = new (std::nothrow) zero_ctx;
  if (!ctx) return fail(nullptr, ZERO_ENOMEM, "cannot allocate context");
  ctx->cfg = *cfg;
  try {
    st = plan_layout(ctx, param_numel, param_unit, n_params);
  } catch (const std::bad_alloc&) {
    st = fail(nullptr, ZERO_ENOMEM, "cannot allocate layout tables");
  }
  if (st != ZERO_OK) {
    delete ctx;
    return st;
  }
  *out = ctx;
  return ZERO_OK;
}

zero_status zero_make_master(const zero_config* cfg, const int64_t* param_numel, const int32_t* param_unit,
                             int32_t n_params, const float* const* init_params, const zero_buffers* bufs,
                             void* stream, zero_ctx** out) {
  if (!out) return fail(nullptr, ZERO_EINVAL, "out is NULL");
  *out = nullptr;
  if (!bufs) return fail(nullptr, ZERO_EINVAL, "bufs is NULL");
  zero_ctx* ctx = nullptr;
  zero_status st = zero_plan(cfg, param_numel, param_unit, n_params, &ctx);
  if (st != ZERO_OK) return st;
  auto bail = [&](zero_status s) {
    g_thread_error = ctx->error;
    delete ctx;
    return s;
  };
  const void* need[4] = {bufs->master, bufs->exp_avg, bufs->exp_avg_sq, bufs->param16};
  const char* names[4] = {"master", "exp_avg", "exp_avg_sq", "param16"};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return bail(fail(ctx, ZERO_ECUDA, "no CUDA device"));
  for (int k = 0; k < 4; ++k) {
    if (!need[k]) return bail(fail(ctx, ZERO_EINVAL, "buffer %s is NULL", names[k]));
    if (!aligned(need[k], 16)) return bail(fail(ctx, ZERO_EINVAL, "buffer %s is not 16-byte aligned", names[k]));
    int pdev = -1;
    if (!is_device_pointer(need[k], &pdev))
      return bail(fail(ctx, ZERO_EINVAL, "buffer %s is not CUDA device memory", names[k]));
    if (pdev != dev) return bail(fail(ctx, ZERO_EINVAL, "buffer %s is on device %d, current is %d", names[k], pdev, dev));
  }
  for (int32_t p = 0; p < n_params; ++p) {
    if (param_numel[p] == 0) continue;
    if (!init_params || !init_params[p]) return bail(fail(ctx, ZERO_EINVAL, "init param %d is NULL", p));
    if (!aligned(init_params[p], 4)) return bail(fail(ctx, ZERO_EINVAL, "init param %d is not 4-byte aligned", p));
    if (!is_device_pointer(init_params[p], nullptr))
      return bail(fail(ctx, ZERO_EINVAL, "init param %d is not CUDA device memory", p));
  }
  ctx->bufs = *bufs;
  ctx->device = dev;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint16_t* p16 = static_cast<uint16_t*>(bufs->param16);
  cudaError_t e = zfs::launch_zero_fill(bufs->master, bufs->exp_avg, bufs->exp_avg_sq, p16, ctx->padded_total, s);
  if (e != cudaSuccess) return bail(fail_cuda(ctx, "make_master zero fill", e));
  for (int32_t p = 0; p < n_params; ++p) {
    e = zfs::launch_copy_param(init_params ? init_params[p] : nullptr, bufs->master, p16, ctx->param_offset[p],
                               param_numel[p], s);
    if (e != cudaSuccess) return bail(fail_cuda(ctx, "make_master copy", e));
  }
  ctx->phase = Phase::kReady;
  ctx->t = 0;
  *out = ctx;
  return ZERO_OK;
}

zero_status zero_make_master_offload(const zero_config* cfg, const int64_t* param_numel, const int32_t* param_unit,
                                     int32_t n_params, const float* const* init_params, const zero_buffers* bufs,
                                     void* stream, zero_ctx** out) {
  if (!out) return fail(nullptr, ZERO_EINVAL, "out is NULL");
  *out = nullptr;
  if (!bufs) return fail(nullptr, ZERO_EINVAL, "bufs is NULL");
  zero_ctx* ctx = nullptr;
  zero_status st = zero_plan(cfg, param_numel, param_unit, n_params, &ctx);
  if (st != ZERO_OK) return st;
  auto bail = [&](zero_status s) {
    g_thread_error = ctx->error;
    delete ctx;
    return s;
  };
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return bail(fail(ctx, ZERO_ECUDA, "no CUDA device"));
  float* host[3] = {bufs->master, bufs->exp_avg, bufs->exp_avg_sq};
  const char* names[3] = {"master", "exp_avg", "exp_avg_sq"};
  for (int k = 0; k < 3; ++k) {
    if (!host[k]) return bail(fail(ctx, ZERO_EINVAL, "buffer %s is NULL", names[k]));
    if (!aligned(host[k], 16)) return bail(fail(ctx, ZERO_EINVAL, "buffer %s is not 16-byte aligned", names[k]));
    if (is_device_pointer(host[k], nullptr))
      return bail(fail(ctx, ZERO_EINVAL, "buffer %s must be host memory in an offload context", names[k]));
  }
  int pdev = -1;
  if (!bufs->param16) return bail(fail(ctx, ZERO_EINVAL, "buffer param16 is NULL"));
  if (!aligned(bufs->param16, 16)) return bail(fail(ctx, ZERO_EINVAL, "buffer param16 is not 16-byte aligned"));
  if (!is_device_pointer(bufs->param16, &pdev)) return bail(fail(ctx, ZERO_EINVAL, "buffer param16 is not CUDA device memory"));
  if (pdev != dev) return bail(fail(ctx, ZERO_EINVAL, "buffer param16 is on device %d, current is %d", pdev, dev));
  for (int32_t p = 0; p < n_params; ++p) {
    if (param_numel[p] == 0) continue;
    if (!init_params || !init_params[p]) return bail(fail(ctx, ZERO_EINVAL, "init param %d is NULL", p));
    if (!aligned(init_params[p], 4)) return bail(fail(ctx, ZERO_EINVAL, "init param %d is not 4-byte aligned", p));
    if (!is_device_pointer(init_params[p], nullptr))
      return bail(fail(ctx, ZERO_EINVAL, "init param %d is not CUDA device memory", p));
  }
  ctx->bufs = *bufs;
  ctx->device = dev;
  ctx->offload = true;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint16_t* p16 = static_cast<uint16_t*>(bufs->param16);
  // Host master = init params at their offsets, pads / m / v = 0; device
  // param16 = bf16(init params), pads 0.
  cudaError_t e = cudaStreamSynchronize(s);
  for (int k = 0; k < 3 && e == cudaSuccess; ++k)
    std::memset(host[k], 0, static_cast<size_t>(ctx->padded_total) * sizeof(float));
  if (e == cudaSuccess && ctx->padded_total > 0) e = cudaMemsetAsync(p16, 0, static_cast<size_t>(ctx->padded_total) * 2, s);
  for (int32_t p = 0; p < n_params && e == cudaSuccess; ++p) {
    if (param_numel[p] == 0) continue;
    e = cudaMemcpyAsync(host[0] + ctx->param_offset[p], init_params[p], param_numel[p] * sizeof(float),
                        cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = zfs::launch_copy_param(init_params[p], nullptr, p16, ctx->param_offset[p], param_numel[p], s);
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return bail(fail_cuda(ctx, "make_master_offload", e));
  ctx->phase = Phase::kReady;
  ctx->t = 0;
  *out = ctx;
  return ZERO_OK;
}

zero_status zero_num_units(const zero_ctx* ctx, int32_t* n_units) {
  if (!ctx || !n_units) return fail(nullptr, ZERO_EINVAL, "NULL argument");
  *n_units = ctx->n_units;
  return ZERO_OK;
}

zero_status zero_padded_numel(const zero_ctx* ctx, int64_t* padded, int64_t* numel) {
  if (!ctx) return fail(nullptr, ZERO_EINVAL, "ctx is NULL");
  if (padded) *padded = ctx->padded_total;
  if (numel) *numel = ctx->numel_total;
  return ZERO_OK;
}

zero_status zero_layout(const zero_ctx* ctx, int32_t unit, int64_t* numel, int64_t* padded, int64_t* shard,
                        int64_t* base) {
  if (!ctx) return fail(nullptr, ZERO_EINVAL, "ctx is NULL");
  zero_ctx* c = const_cast<zero_ctx*>(ctx);
  if (unit < 0 || unit >= ctx->n_units) return fail(c, ZERO_EINVAL, "unit %d out of range [0, %d)", unit, ctx->n_units);
  if (numel) *numel = ctx->unit_numel[unit];
  if (padded) *padded = ctx->unit_padded[unit];
  if (shard) *shard = ctx->unit_shard[unit];
  if (base) *base = ctx->unit_base[unit];
  return ZERO_OK;
}

zero_status zero_param_offset(const zero_ctx* ctx, int32_t param, int64_t* offset) {
  if (!ctx || !offset) return fail(nullptr, ZERO_EINVAL, "NULL argument");
  zero_ctx* c = const_cast<zero_ctx*>(ctx);
  if (param < 0 || param >= ctx->n_params) return fail(c, ZERO_EINVAL, "param %d out of range", param);
  *offset = ctx->param_offset[param];
  return ZERO_OK;
}

zero_status zero_state_bytes(const zero_ctx* ctx, int32_t stage, int64_t* per_rank_bytes) {
  if (!ctx || !per_rank_bytes) return fail(nullptr, ZERO_EINVAL, "NULL argument");
  zero_ctx* c = const_cast<zero_ctx*>(ctx);
  if (stage < 0 || stage > 3) return fail(c, ZERO_EINVAL, "stage %d not in 0..3", stage);
  const int64_t N = ctx->cfg.n_ranks;
  int64_t P = 0, S = 0;
  for (int32_t i = 0; i < ctx->n_units; ++i) {
    const int64_t padded = padded_as_stage(ctx, i, stage);
    P += padded;
    S += padded / N;
  }
  int64_t bytes;
  switch (stage) {
    case 0: bytes = 16 * P; break;
    case 1: bytes = 4 * P + 12 * S; break;
    case 2: bytes = 2 * P + 14 * S; break;
    default: bytes = 16 * S; break;
  }
  for (int64_t r = 0; r < N; ++r) per_rank_bytes[r] = bytes;
  return ZERO_OK;
}

zero_status zero_stage3_peak_bytes(const zero_ctx* ctx, int64_t* peak_bytes, int32_t* peak_unit) {
  if (!ctx || !peak_bytes) return fail(nullptr, ZERO_EINVAL, "NULL argument");
  const int64_t N = ctx->cfg.n_ranks;
  int64_t S = 0;
  for (int32_t i = 0; i < ctx->n_units; ++i) S += padded_as_stage(ctx, i, 3) / N;
  const int64_t resident = 14 * S;  // bf16 param shard 2 + fp32 master/m/v 12
  int64_t best = resident, reduced = 0;
  int32_t where = -1;
  for (int32_t k = ctx->n_units - 1; k >= 0; --k) {
    const int64_t padded = padded_as_stage(ctx, k, 3);
    const int64_t at = resident + reduced + 4 * padded;
    if (at > best) {
      best = at;
      where = k;
    }
    reduced += 2 * (padded / N);
  }
  *peak_bytes = best;
  if (peak_unit) *peak_unit = where;
  return ZERO_OK;
}

zero_status zero_reduce_grads(zero_ctx* ctx, int32_t unit, const void* const* replica_grads, void* stream) {
  (void)stream;  // the reduction is fused into zero_step; nothing is enqueued here
  if (!ctx) return fail(nullptr, ZERO_EINVAL, "ctx is NULL");
  zero_status st = require_bound(ctx);
  if (st != ZERO_OK) return st;
  if (ctx->phase == Phase::kStepped) return fail(ctx, ZERO_ESTATE, "reduce_grads after step: call post_step first");
  if (ctx->clip_ws)
    return fail(ctx, ZERO_ESTATE, "reduce_grads after zero_clip_grad_norm: the clip was computed from the "
                                  "gradients registered before it; register all units, then clip");
  if (unit < -1 || unit >= ctx->n_units) return fail(ctx, ZERO_EINVAL, "unit %d out of range", unit);
  if (!replica_grads) return fail(ctx, ZERO_EINVAL, "replica_grads is NULL");
  const int N = ctx->cfg.n_ranks;
  const size_t esz = grad_bytes(ctx->cfg);
  const int64_t len = unit < 0 ? ctx->padded_total : ctx->unit_padded[unit];
  for (int r = 0; r < N; ++r) {
    if (len > 0 && !replica_grads[r]) return fail(ctx, ZERO_EINVAL, "replica %d gradient is NULL", r);
    if (!aligned(replica_grads[r], esz))
      return fail(ctx, ZERO_EINVAL, "replica %d gradient is not %zu-byte aligned", r, esz);
  }
  if (unit >= 0) {
    for (int r = 0; r < N; ++r) ctx->grads[static_cast<size_t>(unit) * zfs::kMaxRanks + r] = replica_grads[r];
    ctx->registered[unit] = 1;
  } else {
    for (int32_t i = 0; i < ctx->n_units; ++i) {
      for (int r = 0; r < N; ++r) {
        const char* b = static_cast<const char*>(replica_grads[r]);
        ctx->grads[static_cast<size_t>(i) * zfs::kMaxRanks + r] = b ? b + ctx->unit_base[i] * esz : nullptr;
      }
      ctx->registered[i] = 1;
    }
  }
  return ZERO_OK;
}

zero_status zero_accumulate_grads(zero_ctx* ctx, int32_t unit, const void* const* micro_grads_bf16,
                                  float* const* accumulators, int32_t first, void* stream) {
  if (!ctx) return fail(nullptr, ZERO_EINVAL, "ctx is NULL");
  zero_status st = require_bound(ctx);
  if (st != ZERO_OK) return st;
  if (ctx->cfg.grad_dtype != ZERO_GRAD_FP32)
    return fail(ctx, ZERO_EINVAL, "accumulation needs a context with grad_dtype fp32 (the accumulators it steps on)");
  if (unit < -1 || unit >= ctx->n_units) return fail(ctx, ZERO_EINVAL, "unit %d out of range", unit);
  if (!micro_grads_bf16 || !accumulators) return fail(ctx, ZERO_EINVAL, "pointer arrays are NULL");
  const int N = ctx->cfg.n_ranks;
  const int64_t len = unit < 0 ? ctx->padded_total : ctx->unit_padded[unit];
  zfs::AccumArgs a;
  std::memset(&a, 0, sizeof a);
  a.n_ranks = N;
  a.first = first ? 1 : 0;
  a.n = len;
  bool vec = true;
  for (int r = 0; r < N; ++r) {
    if (len > 0 && (!micro_grads_bf16[r] || !accumulators[r]))
      return fail(ctx, ZERO_EINVAL, "replica %d buffer is NULL", r);
    if (!aligned(micro_grads_bf16[r], 2) || !aligned(accumulators[r], 4))
      return fail(ctx, ZERO_EINVAL, "replica %d buffer is misaligned for its element type", r);
    if (!aligned(micro_grads_bf16[r], 16) || !aligned(accumulators[r], 16)) vec = false;
    a.micro[r] = static_cast<const uint16_t*>(micro_grads_bf16[r]);
    a.acc[r] = accumulators[r];
  }
  if (len == 0) {
    ctx->last_launches = 0;
    return ZERO_OK;
  }
  const cudaError_t e = zfs::launch_accumulate(a, vec, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(ctx, "accumulate kernel launch", e);
  ctx->last_launches = 1;
  return ZERO_OK;
}

zero_status zero_step(zero_ctx* ctx, void* stream) {
  if (!ctx) return fail(nullptr, ZERO_EINVAL, "ctx is NULL");
  zero_status st = require_bound(ctx);
  if (st != ZERO_OK) return st;
  if (ctx->offload) return fail(ctx, ZERO_ESTATE, "offload context: its step is zero_offload_step");
  if (ctx->phase == Phase::kStepped) return fail(ctx, ZERO_ESTATE, "step already taken: call post_step first");
  for (int32_t i = 0; i < ctx->n_units; ++i) {
    if (!ctx->registered[i]) return fail(ctx, ZERO_ESTATE, "unit %d has no registered gradients", i);
  }
  const int64_t t = ctx->t + 1;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t launches = 0;
  if (ctx->clip_keep) {
    // The clip kept the reduced gradient: one fp32 "replica" over the whole
    // padded buffer, already scaled by 1/N (x 1 below is exact).
    if (ctx->padded_total > 0) {
      zfs::StepArgs a;
      std::memset(&a, 0, sizeof a);
      a.master = ctx->bufs.master;
      a.m = ctx->bufs.exp_avg;
      a.v = ctx->bufs.exp_avg_sq;
      a.p16 = static_cast<uint16_t*>(ctx->bufs.param16);
      a.clip = reinterpret_cast<const float*>(ctx->clip_ws + 8);
      a.nonfinite = ctx->nonfinite;
      fill_scalars(ctx, t, &a);
      a.total_padded = ctx->padded_total - (ctx->inject == ZERO_INJECT_SHORT_BOUNDS ? zfs::kVec : 0);
      a.dev_t = ctx->cap_t;
      a.dev_bias = ctx->cap_bias;
      a.dev_steps = ctx->cap_steps;
      a.inv_n = 1.0f;
      a.n_ranks = 1;
      a.grad_fp32 = 1;
      a.nseg = 1;
      a.seg[0].base = 0;
      a.seg[0].len = ctx->padded_total;
      a.seg[0].vec_start = 0;
      a.seg[0].g[0] = ctx->clip_keep;
      a.total_vec = ctx->padded_total / zfs::kVec;
      a.total_elems = ctx->padded_total;
      const cudaError_t e = zfs::launch_step_vec(a, s);
      if (e != cudaSuccess) return fail_cuda(ctx, "step kernel launch", e);
      launches = 1;
    }
  } else {
    std::vector<PlannedSeg> vec_segs, shift_segs;
    try {
      for (const PlannedSeg& sg : build_segments(ctx)) {
        if (vector_ok(sg, ctx->cfg.n_ranks)) {
          vec_segs.push_back(sg);
        } else {
          shift_segs.push_back(peel(sg, ctx->cfg.n_ranks, grad_bytes(ctx->cfg)));
        }
      }
    } catch (const std::bad_alloc&) {
      return fail(ctx, ZERO_ENOMEM, "cannot allocate segment list");
    }
    st = launch_batches(ctx, vec_segs, true, t, s, &launches);
    if (st != ZERO_OK) return st;
    st = launch_batches(ctx, shift_segs, false, t, s, &launches);
    if (st != ZERO_OK) return st;
  }
  if (ctx->inject == ZERO_INJECT_SHORT_BOUNDS) ctx->inject = 0;
  if (ctx->cap_t) {
    const cudaError_t e = zfs::launch_count_step(ctx->cap_t, s);
    if (e != cudaSuccess) return fail_cuda(ctx, "step count launch", e);
    ++launches;
  }
  ctx->last_launches = launches;
  ctx->t = t;
  ctx->phase = Phase::kStepped;
  return ZERO_OK;
}

// ---------------------------------------------------------------------------
// ZeRO-Offload step.
// ---------------------------------------------------------------------------
namespace {

constexpr int kOffloadRing = 3;  // chunks in flight between the GPU and the host

int64_t offload_slot_elems(const zero_ctx* ctx, int64_t chunk) {
  const int64_t c = std::min<int64_t>(chunk, std::max<int64_t>(ctx->padded_total, 1));
  return (c + 63) / 64 * 64;
}

// One chunk of host Adam work; the pool's callback captures only a
// reference to it (small enough for std::function to store without allocating).
struct HostAdamJob {
  zfs_host::AdamScalars sc;
  const float* g;
  float* w;
  float* m;
  float* v;
  uint16_t* p16;
  void operator()(int64_t lo, int64_t hi) const {
    zfs_host::adam_range(sc, g + lo, w + lo, m + lo, v + lo, p16 + lo, hi - lo);
  }
};

struct EventSet {
  std::vector<cudaEvent_t> ev;
  ~EventSet() {
    for (cudaEvent_t e : ev) cudaEventDestroy(e);
  }
  cudaError_t make(int n) {
    for (int i = 0; i < n; ++i) {
      cudaEvent_t e = nullptr;
      const cudaError_t r = cudaEventCreateWithFlags(&e, cudaEventDisableTiming);
      if (r != cudaSuccess) return r;
      ev.push_back(e);
    }
    return cudaSuccess;
  }
};

// Launches of the reduced gradient of [c0, c1) into out (slot of the device
// workspace): the registered segments intersected with the chunk.
cudaError_t enqueue_chunk_reduce(const zero_ctx* ctx, const std::vector<PlannedSeg>& segs, int64_t c0, int64_t c1,
                                 float* out, const float* clip, cudaStream_t s, int32_t* launches) {
  const int N = ctx->cfg.n_ranks;
  const size_t esz = grad_bytes(ctx->cfg);
  zfs::ReduceArgs a;
  std::memset(&a, 0, sizeof a);
  a.out = out;
  a.out_len = c1 - c0;
  a.clip = clip;
  a.nonfinite = ctx->nonfinite;
  a.inv_n = 1.0f / static_cast<float>(N);
  a.n_ranks = N;
  a.grad_fp32 = ctx->cfg.grad_dtype == ZERO_GRAD_FP32 ? 1 : 0;
  auto flush = [&]() -> cudaError_t {
    if (a.nseg == 0) return cudaSuccess;
    const cudaError_t e = zfs::launch_reduce_out(a, s);
    if (e == cudaSuccess) ++*launches;
    a.nseg = 0;
    a.total_groups = 0;
    return e;
  };
  for (const PlannedSeg& sg : segs) {
    const int64_t lo = std::max(sg.base, c0), hi = std::min(sg.base + sg.len, c1);
    if (lo >= hi) continue;
    if (a.nseg == zfs::kMaxSegs) {
      const cudaError_t e = flush();
      if (e != cudaSuccess) return e;
    }
    zfs::ReduceSeg& r = a.seg[a.nseg++];
    r.out_off = lo - c0;
    r.len = hi - lo;
    r.group_start = a.total_groups;
    bool vec = r.out_off % 4 == 0;
    for (int k = 0; k < N; ++k) {
      r.g[k] = static_cast<const char*>(sg.g[k]) + (lo - sg.base) * esz;
      vec = vec && aligned(r.g[k], 16);
    }
    r.vec_ok = vec ? 1 : 0;
    a.total_groups += (r.len + zfs::kVec - 1) / zfs::kVec;
  }
  return flush();
}

}  // namespace

zero_status zero_offload_workspace_bytes(const zero_ctx* ctx, int64_t chunk, int64_t* host_bytes,
                                         int64_t* device_bytes) {
  if (!ctx || !host_bytes || !device_bytes) return fail(nullptr, ZERO_EINVAL, "NULL argument");
  if (chunk < 1) return fail(const_cast<zero_ctx*>(ctx), ZERO_EINVAL, "chunk must be >= 1 element");
  const int64_t slot = offload_slot_elems(ctx, chunk);
  *host_bytes = kOffloadRing * slot * (4 + 2);
  *device_bytes = kOffloadRing * slot * 4;
  return ZERO_OK;
}

zero_status zero_offload_step(zero_ctx* ctx, int64_t chunk, void* host_workspace, int64_t host_bytes,
                              void* device_workspace, int64_t device_bytes, int32_t n_threads, void* stream,
                              void* copy_stream) {
  if (!ctx) return fail(nullptr, ZERO_EINVAL, "ctx is NULL");
  zero_status st = require_bound(ctx);
  if (st != ZERO_OK) return st;
  if (!ctx->offload) return fail(ctx, ZERO_ESTATE, "not an offload context (see zero_make_master_offload)");
  if (ctx->phase == Phase::kStepped) return fail(ctx, ZERO_ESTATE, "step already taken: call post_step first");
  int32_t missing = -1;
  if (!all_registered(ctx, &missing)) return fail(ctx, ZERO_ESTATE, "unit %d has no registered gradients", missing);
  if (chunk < 1) return fail(ctx, ZERO_EINVAL, "chunk must be >= 1 element");
  if (n_threads < 0 || n_threads > 1024) return fail(ctx, ZERO_EINVAL, "n_threads %d not in 0..1024", n_threads);
  const int64_t slot = offload_slot_elems(ctx, chunk);
  if (host_bytes < kOffloadRing * slot * 6) return fail(ctx, ZERO_EINVAL, "host workspace too small");
  if (device_bytes < kOffloadRing * slot * 4) return fail(ctx, ZERO_EINVAL, "device workspace too small");
  if (!host_workspace || !aligned(host_workspace, 16)) return fail(ctx, ZERO_EINVAL, "host workspace NULL or not 16-byte aligned");
  if (!device_workspace || !aligned(device_workspace, 16))
    return fail(ctx, ZERO_EINVAL, "device workspace NULL or not 16-byte aligned");
  {
    cudaPointerAttributes attr{};
    if (cudaPointerGetAttributes(&attr, host_workspace) != cudaSuccess || attr.type != cudaMemoryTypeHost) {
      cudaGetLastError();
      return fail(ctx, ZERO_EINVAL, "host workspace is not page-locked (pinned) host memory");
    }
    int wdev = -1;
    if (!is_device_pointer(device_workspace, &wdev) || wdev != ctx->device)
      return fail(ctx, ZERO_EINVAL, "device workspace is not memory of the context's device");
  }
  int threads = n_threads > 0 ? n_threads : static_cast<int>(std::thread::hardware_concurrency());
  if (threads < 1) threads = 1;
  if (!ctx->pool || zfs_host::pool_threads(ctx->pool) != threads) {
    zfs_host::pool_destroy(ctx->pool);
    ctx->pool = zfs_host::pool_create(threads);
    if (!ctx->pool) return fail(ctx, ZERO_ENOMEM, "cannot start %d host threads", threads);
  }
  std::vector<PlannedSeg> segs;
  try {
    segs = build_segments(ctx);
  } catch (const std::bad_alloc&) {
    return fail(ctx, ZERO_ENOMEM, "cannot allocate segment list");
  }
  const int64_t t = ctx->t + 1;
  const zfs_host::AdamScalars sc = adam_scalars(ctx->cfg, t);
  const float* clip = ctx->clip_ws ? reinterpret_cast<const float*>(ctx->clip_ws + 8) : nullptr;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaStream_t cs = copy_stream ? static_cast<cudaStream_t>(copy_stream) : s;
  float* dev_g = static_cast<float*>(device_workspace);
  float* host_g = static_cast<float*>(host_workspace);
  uint16_t* host_p = reinterpret_cast<uint16_t*>(host_g + kOffloadRing * slot);
  uint16_t* p16 = static_cast<uint16_t*>(ctx->bufs.param16);
  const int64_t P = ctx->padded_total;
  const int64_t n_chunks = (P + chunk - 1) / chunk;

  // Events: [0, R) gradients of a slot on the host, [R, 2R) a slot's
  // parameters on the device, 2R: start of the step on `stream`, 2R+1: end.
  EventSet evs;
  cudaError_t e = evs.make(2 * kOffloadRing + 2);
  if (e != cudaSuccess) return fail_cuda(ctx, "offload events", e);
  cudaEvent_t* ev_g = evs.ev.data();
  cudaEvent_t* ev_p = evs.ev.data() + kOffloadRing;
  int32_t launches = 0;
  // param16 is rewritten on the copy stream: only after the caller's earlier work on `stream`.
  e = cudaEventRecord(evs.ev[2 * kOffloadRing], s);
  if (e == cudaSuccess && cs != s) e = cudaStreamWaitEvent(cs, evs.ev[2 * kOffloadRing], 0);
  auto enqueue = [&](int64_t c) -> cudaError_t {
    const int k = static_cast<int>(c % kOffloadRing);
    const int64_t c0 = c * chunk, c1 = std::min(P, c0 + chunk);
    cudaError_t r = enqueue_chunk_reduce(ctx, segs, c0, c1, dev_g + k * slot, clip, s, &launches);
    if (r == cudaSuccess)
      r = cudaMemcpyAsync(host_g + k * slot, dev_g + k * slot, (c1 - c0) * sizeof(float), cudaMemcpyDeviceToHost, s);
    if (r == cudaSuccess) r = cudaEventRecord(ev_g[k], s);
    return r;
  };
  for (int64_t c = 0; c < std::min<int64_t>(kOffloadRing, n_chunks) && e == cudaSuccess; ++c) e = enqueue(c);
  for (int64_t c = 0; c < n_chunks && e == cudaSuccess; ++c) {
    const int k = static_cast<int>(c % kOffloadRing);
    const int64_t c0 = c * chunk, c1 = std::min(P, c0 + chunk);
    e = cudaEventSynchronize(ev_g[k]);                       // this chunk's gradients are on the host
    if (e == cudaSuccess && c >= kOffloadRing) e = cudaEventSynchronize(ev_p[k]);  // slot's last upload done
    if (e != cudaSuccess) break;
    const HostAdamJob job{sc, host_g + k * slot, ctx->bufs.master + c0, ctx->bufs.exp_avg + c0,
                          ctx->bufs.exp_avg_sq + c0, host_p + k * slot};
    zfs_host::pool_run(ctx->pool, c1 - c0, [&job](int64_t lo, int64_t hi) { job(lo, hi); });
    e = cudaMemcpyAsync(p16 + c0, job.p16, (c1 - c0) * 2, cudaMemcpyHostToDevice, cs);
    if (e == cudaSuccess) e = cudaEventRecord(ev_p[k], cs);
    if (e == cudaSuccess && c + kOffloadRing < n_chunks) e = enqueue(c + kOffloadRing);
  }
  // Later work on `stream` sees the new param16.
  if (e == cudaSuccess && cs != s) e = cudaEventRecord(evs.ev[2 * kOffloadRing + 1], cs);
  if (e == cudaSuccess && cs != s) e = cudaStreamWaitEvent(s, evs.ev[2 * kOffloadRing + 1], 0);
  if (e != cudaSuccess) {
    // Chunks already updated on the host stay updated: the state is partial.
    cudaStreamSynchronize(cs);
    cudaStreamSynchronize(s);
    return fail_cuda(ctx, "offload step (state partially updated)", e);
  }
  ctx->last_launches = launches;
  ctx->t = t;
  ctx->phase = Phase::kStepped;
  return ZERO_OK;
}

zero_status zero_cpu_adam(const zero_config* cfg, int64_t t, const float* grad, float* master, float* exp_avg,
                          float* exp_avg_sq, uint16_t* param16, int64_t n, int32_t n_threads) {
  zero_status st = check_config(cfg, nullptr);
  if (st != ZERO_OK) return st;
  if (t < 1) return fail(nullptr, ZERO_EINVAL, "t must be >= 1");
  if (n < 0) return fail(nullptr, ZERO_EINVAL, "n is negative");
  if (n_threads < 0 || n_threads > 1024) return fail(nullptr, ZERO_EINVAL, "n_threads %d not in 0..1024", n_threads);
  if (n == 0) return ZERO_OK;
  const void* ptrs[5] = {grad, master, exp_avg, exp_avg_sq, param16};
  const char* names[5] = {"grad", "master", "exp_avg", "exp_avg_sq", "param16"};
  for (int k = 0; k < 5; ++k) {
    if (!ptrs[k]) return fail(nullptr, ZERO_EINVAL, "%s is NULL", names[k]);
    if (!aligned(ptrs[k], k == 4 ? 2 : 4)) return fail(nullptr, ZERO_EINVAL, "%s is misaligned", names[k]);
  }
  int threads = n_threads > 0 ? n_threads : static_cast<int>(std::thread::hardware_concurrency());
  if (threads < 1) threads = 1;
  const zfs_host::AdamScalars sc = adam_scalars(*cfg, t);
  // One process-wide pool for these context-free calls (kept between calls:
  // starting the threads costs about as much as updating a few million
  // elements); concurrent callers take turns.
  static std::mutex pool_mutex;
  static std::unique_ptr<zfs_host::Pool, void (*)(zfs_host::Pool*)> pool(nullptr, zfs_host::pool_destroy);
  std::lock_guard<std::mutex> lock(pool_mutex);
  if (!pool || zfs_host::pool_threads(pool.get()) != threads) {
    pool.reset();
    pool.reset(zfs_host::pool_create(threads));
    if (!pool) return fail(nullptr, ZERO_ENOMEM, "cannot start %d host threads", threads);
  }
  const HostAdamJob job{sc, grad, master, exp_avg, exp_avg_sq, param16};
  zfs_host::pool_run(pool.get(), n, [&job](int64_t lo, int64_t hi) { job(lo, hi); });
  return ZERO_OK;
}

namespace {

int64_t clip_partials_end(const zero_ctx* ctx) { return zfs::kClipHeaderBytes + 8 * total_chunks(ctx); }

// Byte offset of the kept reduced gradient inside the workspace.
int64_t clip_keep_offset(const zero_ctx* ctx) { return (clip_partials_end(ctx) + 255) / 256 * 256; }

int64_t clip_bytes(const zero_ctx* ctx, int32_t flags) {
  return (flags & ZERO_CLIP_KEEP_REDUCED) ? clip_keep_offset(ctx) + 4 * ctx->padded_total : clip_partials_end(ctx);
}

}  // namespace

zero_status zero_clip_workspace_bytes(const zero_ctx* ctx, int64_t* bytes) {
  return zero_clip_workspace_bytes_ex(ctx, 0, bytes);
}

zero_status zero_clip_workspace_bytes_ex(const zero_ctx* ctx, int32_t flags, int64_t* bytes) {
  if (!ctx || !bytes) return fail(nullptr, ZERO_EINVAL, "NULL argument");
  if (flags & ~ZERO_CLIP_KEEP_REDUCED) return fail(const_cast<zero_ctx*>(ctx), ZERO_EINVAL, "unknown clip flags");
  *bytes = clip_bytes(ctx, flags);
  return ZERO_OK;
}

zero_status zero_clip_grad_norm(zero_ctx* ctx, float max_norm, void* workspace, int64_t workspace_bytes,
                                void* stream) {
  return zero_clip_grad_norm_ex(ctx, max_norm, 0, workspace, workspace_bytes, stream);
}

zero_status zero_clip_grad_norm_ex(zero_ctx* ctx, float max_norm, int32_t flags, void* workspace,
                                   int64_t workspace_bytes, void* stream) {
  if (!ctx) return fail(nullptr, ZERO_EINVAL, "ctx is NULL");
  if (flags & ~ZERO_CLIP_KEEP_REDUCED) return fail(ctx, ZERO_EINVAL, "unknown clip flags");
  const bool keep = (flags & ZERO_CLIP_KEEP_REDUCED) != 0;
  zero_status st = require_bound(ctx);
  if (st != ZERO_OK) return st;
  if (keep && ctx->offload)
    return fail(ctx, ZERO_ENOTSUP, "ZERO_CLIP_KEEP_REDUCED is not available in an offload context");
  if (ctx->phase == Phase::kStepped) return fail(ctx, ZERO_ESTATE, "clip after step: call post_step first");
  int32_t missing = -1;
  if (!all_registered(ctx, &missing)) return fail(ctx, ZERO_ESTATE, "unit %d has no registered gradients", missing);
  if (!(max_norm > 0.0f) || !std::isfinite(max_norm)) return fail(ctx, ZERO_EINVAL, "max_norm must be finite and > 0");
  const int64_t need = clip_bytes(ctx, flags);
  if (!workspace) return fail(ctx, ZERO_EINVAL, "workspace is NULL");
  if (!aligned(workspace, 16)) return fail(ctx, ZERO_EINVAL, "workspace is not 16-byte aligned");
  if (workspace_bytes < need)
    return fail(ctx, ZERO_EINVAL, "workspace has %lld bytes, %lld needed", static_cast<long long>(workspace_bytes),
                static_cast<long long>(need));
  if (!is_device_pointer(workspace, nullptr)) return fail(ctx, ZERO_EINVAL, "workspace is not CUDA device memory");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  double* partials = reinterpret_cast<double*>(ws + zfs::kClipHeaderBytes);
  float* keep_base = keep ? reinterpret_cast<float*>(ws + clip_keep_offset(ctx)) : nullptr;
  const int N = ctx->cfg.n_ranks;
  int32_t launches = 0;
  int64_t out = 0;
  // Units with 16-byte-aligned gradients and units without go to separate
  // launches (the instances with shifted loads take the latter); partials
  // keep their unit-order places whatever launch writes them.
  zfs::NormArgs batch[2];
  long long batch_chunks[2] = {0, 0};
  for (int b = 0; b < 2; ++b) {
    std::memset(&batch[b], 0, sizeof batch[b]);
    batch[b].n_ranks = N;
    batch[b].grad_fp32 = ctx->cfg.grad_dtype == ZERO_GRAD_FP32 ? 1 : 0;
    batch[b].inv_n = 1.0f / static_cast<float>(N);
    batch[b].partials = partials;
  }
  auto flush = [&](int b) -> cudaError_t {
    if (batch[b].nseg == 0) return cudaSuccess;
    const cudaError_t e = zfs::launch_grad_sq(batch[b], batch_chunks[b], b == 1, s);
    if (e == cudaSuccess) ++launches;
    batch[b].nseg = 0;
    batch_chunks[b] = 0;
    return e;
  };
  for (int32_t i = 0; i < ctx->n_units; ++i) {
    const int64_t c = unit_chunks(ctx, i);
    if (c == 0) continue;
    zfs::NormSeg g{};
    g.len = ctx->unit_padded[i];
    g.n_chunks = c;
    g.out_start = out;
    g.vec_ok = 1;
    g.keep = keep ? keep_base + ctx->unit_base[i] : nullptr;
    g.keep_vec = keep && aligned(g.keep, 16) ? 1 : 0;
    for (int r = 0; r < N; ++r) {
      g.g[r] = ctx->grads[static_cast<size_t>(i) * zfs::kMaxRanks + r];
      if (!aligned(g.g[r], 16)) g.vec_ok = 0;
      g.shift[r] = static_cast<unsigned char>((reinterpret_cast<uintptr_t>(g.g[r]) % 16) / grad_bytes(ctx->cfg));
    }
    const int b = g.vec_ok ? 0 : 1;
    if (batch[b].nseg == zfs::kMaxSegs) {
      const cudaError_t e = flush(b);
      if (e != cudaSuccess) return fail_cuda(ctx, "norm kernel launch", e);
    }
    g.chunk_start = batch_chunks[b];
    batch[b].seg[batch[b].nseg++] = g;
    batch_chunks[b] += c;
    out += c;
  }
  for (int b = 0; b < 2; ++b) {
    const cudaError_t e = flush(b);
    if (e != cudaSuccess) return fail_cuda(ctx, "norm kernel launch", e);
  }
  const cudaError_t e = zfs::launch_clip_finalize(ws, out, max_norm, s);
  if (e != cudaSuccess) return fail_cuda(ctx, "clip finalize launch", e);
  ctx->last_launches = launches + 1;
  ctx->clip_ws = ws;
  ctx->last_clip_ws = ws;
  ctx->clip_keep = keep_base;
  return ZERO_OK;
}

zero_status zero_grad_norm(zero_ctx* ctx, double* norm, void* stream) {
  if (!ctx || !norm) return fail(nullptr, ZERO_EINVAL, "NULL argument");
  zero_status st = require_bound(ctx);
  if (st != ZERO_OK) return st;
  if (!ctx->last_clip_ws) return fail(ctx, ZERO_ESTATE, "no zero_clip_grad_norm has run on this context");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  double host = 0.0;
  cudaError_t e = cudaMemcpyAsync(&host, ctx->last_clip_ws, sizeof host, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail_cuda(ctx, "reading the norm", e);
  *norm = host;
  return ZERO_OK;
}

zero_status zero_gather_weights(zero_ctx* ctx, int32_t unit, void* unit_buf, void* stream) {
  if (!ctx) return fail(nullptr, ZERO_EINVAL, "ctx is NULL");
  zero_status st = require_bound(ctx);
  if (st != ZERO_OK) return st;
  if (unit < -1 || unit >= ctx->n_units) return fail(ctx, ZERO_EINVAL, "unit %d out of range", unit);
  if (ctx->cfg.stage != 3) {  // the fused step already wrote every replica's full copy
    ctx->last_launches = 0;
    return ZERO_OK;
  }
  const int64_t base = unit < 0 ? 0 : ctx->unit_base[unit];
  const int64_t len = unit < 0 ? ctx->padded_total : ctx->unit_padded[unit];
  if (len == 0) {
    ctx->last_launches = 0;
    return ZERO_OK;
  }
  if (!unit_buf) return fail(ctx, ZERO_EINVAL, "unit_buf is NULL");
  if (!aligned(unit_buf, 2)) return fail(ctx, ZERO_EINVAL, "unit_buf is not 2-byte aligned");
  const uint16_t* src = static_cast<const uint16_t*>(ctx->bufs.param16) + base;
  int32_t launches = 0;
  const cudaError_t e = zfs::launch_gather(src, static_cast<uint16_t*>(unit_buf), len,
                                           static_cast<cudaStream_t>(stream), &launches);
  if (e != cudaSuccess) return fail_cuda(ctx, "gather kernel launch", e);
  ctx->last_launches = launches;
  return ZERO_OK;
}

zero_status zero_gather_units(zero_ctx* ctx, int32_t first_unit, int32_t count, void* const* unit_bufs,
                              void* stream) {
  if (!ctx) return fail(nullptr, ZERO_EINVAL, "ctx is NULL");
  zero_status st = require_bound(ctx);
  if (st != ZERO_OK) return st;
  if (count < 0) return fail(ctx, ZERO_EINVAL, "count %d is negative", count);
  if (first_unit < 0 || first_unit > ctx->n_units || count > ctx->n_units - first_unit) {
    return fail(ctx, ZERO_EINVAL, "units [%d, %d + %d) out of range (%d units)", first_unit, first_unit, count,
                ctx->n_units);
  }
  ctx->last_launches = 0;
  if (ctx->cfg.stage != 3 || count == 0) return ZERO_OK;  // stages 0-2: the step wrote every full copy
  if (!unit_bufs) return fail(ctx, ZERO_EINVAL, "unit_bufs is NULL");
  std::vector<const uint16_t*> src;
  std::vector<uint16_t*> dst;
  std::vector<long long> len;
  for (int32_t k = 0; k < count; ++k) {
    const int32_t u = first_unit + k;
    if (ctx->unit_padded[u] == 0) continue;
    void* buf = unit_bufs[k];
    if (!buf) return fail(ctx, ZERO_EINVAL, "unit_bufs[%d] (unit %d) is NULL", k, u);
    if (!aligned(buf, 2)) return fail(ctx, ZERO_EINVAL, "unit_bufs[%d] (unit %d) is not 2-byte aligned", k, u);
    src.push_back(static_cast<const uint16_t*>(ctx->bufs.param16) + ctx->unit_base[u]);
    dst.push_back(static_cast<uint16_t*>(buf));
    len.push_back(ctx->unit_padded[u]);
  }
  int32_t launches = 0;
  const cudaError_t e = zfs::launch_gather_units(src.data(), dst.data(), len.data(), static_cast<int>(src.size()),
                                                 static_cast<cudaStream_t>(stream), &launches);
  if (e != cudaSuccess) return fail_cuda(ctx, "gather kernel launch", e);
  ctx->last_launches = launches;
  return ZERO_OK;
}

zero_status zero_post_step(zero_ctx* ctx, void* stream) {
  (void)stream;
  if (!ctx) return fail(nullptr, ZERO_EINVAL, "ctx is NULL");
  if (ctx->phase != Phase::kStepped) return fail(ctx, ZERO_ESTATE, "post_step without a step since the last post_step");
  std::fill(ctx->registered.begin(), ctx->registered.end(), 0);
  std::fill(ctx->grads.begin(), ctx->grads.end(), nullptr);
  ctx->clip_ws = nullptr;
  ctx->clip_keep = nullptr;
  ctx->phase = Phase::kReady;
  return ZERO_OK;
}

namespace {

zero_status check_state_buffers(zero_ctx* ctx, const void* const* ptrs, const char* const* names) {
  if (ctx->numel_total == 0) return ZERO_OK;
  for (int k = 0; k < 3; ++k) {
    if (!ptrs[k]) return fail(ctx, ZERO_EINVAL, "%s is NULL", names[k]);
    if (!aligned(ptrs[k], 4)) return fail(ctx, ZERO_EINVAL, "%s is not 4-byte aligned", names[k]);
    if (!is_device_pointer(ptrs[k], nullptr)) return fail(ctx, ZERO_EINVAL, "%s is not CUDA device memory", names[k]);
  }
  return ZERO_OK;
}

// Offload import: host state zeroed (pads), each unit's real elements copied
// down, param16 = bf16(master) on the device; synchronizes the stream.
zero_status import_offload(zero_ctx* ctx, const float* master_in, const float* exp_avg_in,
                           const float* exp_avg_sq_in, int64_t t, cudaStream_t s) {
  uint16_t* p16 = static_cast<uint16_t*>(ctx->bufs.param16);
  float* dst[3] = {ctx->bufs.master, ctx->bufs.exp_avg, ctx->bufs.exp_avg_sq};
  const float* src[3] = {master_in, exp_avg_in, exp_avg_sq_in};
  cudaError_t e = cudaStreamSynchronize(s);  // no earlier work still reading the host state
  if (e != cudaSuccess) return fail_cuda(ctx, "import synchronize", e);
  for (int k = 0; k < 3; ++k) std::memset(dst[k], 0, static_cast<size_t>(ctx->padded_total) * sizeof(float));
  if (ctx->padded_total > 0) e = cudaMemsetAsync(p16, 0, static_cast<size_t>(ctx->padded_total) * 2, s);
  int64_t in = 0;
  for (int32_t i = 0; i < ctx->n_units && e == cudaSuccess; ++i) {
    const int64_t n = ctx->unit_numel[i], base = ctx->unit_base[i];
    for (int k = 0; k < 3 && e == cudaSuccess && n > 0; ++k) {
      e = cudaMemcpyAsync(dst[k] + base, src[k] + in, n * sizeof(float), cudaMemcpyDeviceToHost, s);
    }
    if (e == cudaSuccess) e = zfs::launch_copy_param(master_in + in, nullptr, p16, base, n, s);
    in += n;
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail_cuda(ctx, "import copy", e);
  ctx->t = t;
  return ZERO_OK;
}

}  // namespace

zero_status zero_export_state(zero_ctx* ctx, float* master_out, float* exp_avg_out, float* exp_avg_sq_out,
                              int64_t* t, void* stream) {
  if (!ctx) return fail(nullptr, ZERO_EINVAL, "ctx is NULL");
  zero_status st = require_bound(ctx);
  if (st != ZERO_OK) return st;
  if (ctx->cap_t) return fail(ctx, ZERO_ESTATE, "capturable mode: call zero_disable_capturable first");
  const void* ptrs[3] = {master_out, exp_avg_out, exp_avg_sq_out};
  const char* names[3] = {"master_out", "exp_avg_out", "exp_avg_sq_out"};
  st = check_state_buffers(ctx, ptrs, names);
  if (st != ZERO_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const float* src[3] = {ctx->bufs.master, ctx->bufs.exp_avg, ctx->bufs.exp_avg_sq};
  float* dst[3] = {master_out, exp_avg_out, exp_avg_sq_out};
  int32_t launches = 0;
  int64_t out = 0;
  for (int32_t i = 0; i < ctx->n_units; ++i) {
    for (int k = 0; k < 3; ++k) {
      const int64_t n = ctx->unit_numel[i];
      const float* from = src[k] + ctx->unit_base[i];
      // Offload: the state is host memory, copied up in the same order.
      const cudaError_t e = ctx->offload
          ? (n > 0 ? cudaMemcpyAsync(dst[k] + out, from, n * sizeof(float), cudaMemcpyHostToDevice, s) : cudaSuccess)
          : zfs::launch_copy_f32(from, dst[k] + out, n, s);
      if (e != cudaSuccess) return fail_cuda(ctx, "export copy", e);
      if (n > 0 && !ctx->offload) ++launches;
    }
    out += ctx->unit_numel[i];
  }
  ctx->last_launches = launches;
  if (t) *t = ctx->t;
  return ZERO_OK;
}

zero_status zero_import_state(zero_ctx* ctx, const float* master_in, const float* exp_avg_in,
                              const float* exp_avg_sq_in, int64_t t, void* stream) {
  if (!ctx) return fail(nullptr, ZERO_EINVAL, "ctx is NULL");
  zero_status st = require_bound(ctx);
  if (st != ZERO_OK) return st;
  if (ctx->phase == Phase::kStepped) return fail(ctx, ZERO_ESTATE, "import while a step awaits post_step");
  if (ctx->cap_t) return fail(ctx, ZERO_ESTATE, "capturable mode: call zero_disable_capturable first");
  if (t < 0) return fail(ctx, ZERO_EINVAL, "t is negative");
  const void* ptrs[3] = {master_in, exp_avg_in, exp_avg_sq_in};
  const char* names[3] = {"master_in", "exp_avg_in", "exp_avg_sq_in"};
  st = check_state_buffers(ctx, ptrs, names);
  if (st != ZERO_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint16_t* p16 = static_cast<uint16_t*>(ctx->bufs.param16);
  if (ctx->offload) return import_offload(ctx, master_in, exp_avg_in, exp_avg_sq_in, t, s);
  cudaError_t e = zfs::launch_zero_fill(ctx->bufs.master, ctx->bufs.exp_avg, ctx->bufs.exp_avg_sq, p16,
                                        ctx->padded_total, s);
  if (e != cudaSuccess) return fail_cuda(ctx, "import zero fill", e);
  int64_t in = 0;
  for (int32_t i = 0; i < ctx->n_units; ++i) {
    const int64_t n = ctx->unit_numel[i], base = ctx->unit_base[i];
    e = zfs::launch_copy_param(master_in + in, ctx->bufs.master, p16, base, n, s);
    if (e == cudaSuccess) e = zfs::launch_copy_f32(exp_avg_in + in, ctx->bufs.exp_avg + base, n, s);
    if (e == cudaSuccess) e = zfs::launch_copy_f32(exp_avg_sq_in + in, ctx->bufs.exp_avg_sq + base, n, s);
    if (e != cudaSuccess) return fail_cuda(ctx, "import copy", e);
    in += n;
  }
  ctx->t = t;
  return ZERO_OK;
}

zero_status zero_debug_check_failures(uint32_t* count) {
  if (!count) return fail(nullptr, ZERO_EINVAL, "count is NULL");
#ifdef ZFS_DEBUG_CHECKS
  const unsigned int a = zfs::step_debug_failures(), b = zfs::aux_debug_failures();
  if (a == 0xFFFFFFFFu || b == 0xFFFFFFFFu) return fail(nullptr, ZERO_ECUDA, "cannot read the check counters");
  *count = a + b;
  return ZERO_OK;
#else
  *count = 0;
  return fail(nullptr, ZERO_ENOTSUP, "library built without ZFS_DEBUG_CHECKS");
#endif
}

zero_status zero_debug_inject(zero_ctx* ctx, int32_t what) {
  if (!ctx) return fail(nullptr, ZERO_EINVAL, "ctx is NULL");
  if (what != 0 && what != ZERO_INJECT_MISSING_COPY && what != ZERO_INJECT_SHORT_BOUNDS)
    return fail(ctx, ZERO_EINVAL, "unknown injection %d", what);
  ctx->inject = what;
  return ZERO_OK;
}

zero_status zero_count_nonfinite(zero_ctx* ctx, uint64_t* counter) {
  if (!ctx) return fail(nullptr, ZERO_EINVAL, "ctx is NULL");
  if (counter) {
    if (!aligned(counter, 8)) return fail(ctx, ZERO_EINVAL, "counter is not 8-byte aligned");
    int pdev = -1;
    if (!is_device_pointer(counter, &pdev)) return fail(ctx, ZERO_EINVAL, "counter is not CUDA device memory");
    if (ctx->device >= 0 && pdev != ctx->device)
      return fail(ctx, ZERO_EINVAL, "counter is on device %d, the context's buffers on %d", pdev, ctx->device);
  }
  ctx->nonfinite = reinterpret_cast<unsigned long long*>(counter);
  return ZERO_OK;
}

zero_status zero_read_nonfinite(zero_ctx* ctx, uint64_t* count, void* stream) {
  if (!ctx || !count) return fail(ctx, ZERO_EINVAL, "NULL argument");
  if (!ctx->nonfinite) return fail(ctx, ZERO_ESTATE, "no counter: call zero_count_nonfinite first");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned long long v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, ctx->nonfinite, sizeof v, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail_cuda(ctx, "reading the non-finite counter", e);
  *count = v;
  return ZERO_OK;
}

zero_status zero_kernel_timeouts(const zero_ctx* ctx, uint32_t* count) {
  if (!count) return fail(const_cast<zero_ctx*>(ctx), ZERO_EINVAL, "count is NULL");
  const unsigned int v = zfs::step_timeouts();
  if (v == 0xFFFFFFFFu) return fail(const_cast<zero_ctx*>(ctx), ZERO_ECUDA, "cannot read the timeout counter");
  *count = v;
  return ZERO_OK;
}

zero_status zero_capturable_workspace_bytes(const zero_ctx* ctx, int64_t max_steps, int64_t* bytes) {
  if (!ctx || !bytes) return fail(nullptr, ZERO_EINVAL, "NULL argument");
  if (max_steps < 1) return fail(const_cast<zero_ctx*>(ctx), ZERO_EINVAL, "max_steps must be >= 1");
  *bytes = 16 + 8 * max_steps;  // the step count, then bc1, bc2 per step
  return ZERO_OK;
}

zero_status zero_enable_capturable(zero_ctx* ctx, void* workspace, int64_t workspace_bytes, int64_t max_steps,
                                   void* stream) {
  if (!ctx) return fail(nullptr, ZERO_EINVAL, "ctx is NULL");
  zero_status st = require_bound(ctx);
  if (st != ZERO_OK) return st;
  if (ctx->offload) return fail(ctx, ZERO_ENOTSUP, "the offload step is not capturable (it runs on host threads)");
  if (ctx->phase == Phase::kStepped) return fail(ctx, ZERO_ESTATE, "a step awaits post_step");
  if (max_steps < 1) return fail(ctx, ZERO_EINVAL, "max_steps must be >= 1");
  if (max_steps <= ctx->t) return fail(ctx, ZERO_EINVAL, "max_steps %lld does not exceed the steps taken (%lld)",
                                       static_cast<long long>(max_steps), static_cast<long long>(ctx->t));
  if (!workspace || !aligned(workspace, 16)) return fail(ctx, ZERO_EINVAL, "workspace NULL or not 16-byte aligned");
  if (workspace_bytes < 16 + 8 * max_steps) return fail(ctx, ZERO_EINVAL, "workspace too small");
  int wdev = -1;
  if (!is_device_pointer(workspace, &wdev) || wdev != ctx->device)
    return fail(ctx, ZERO_EINVAL, "workspace is not memory of the context's device");
  std::vector<float> table;
  try {
    table.resize(static_cast<size_t>(2 * max_steps));
  } catch (const std::bad_alloc&) {
    return fail(ctx, ZERO_ENOMEM, "cannot allocate the host table");
  }
  for (int64_t t = 1; t <= max_steps; ++t) {  // the same scalars zero_step would pass
    const zfs_host::AdamScalars sc = adam_scalars(ctx->cfg, t);
    table[2 * (t - 1)] = sc.bc1;
    table[2 * (t - 1) + 1] = sc.bc2;
  }
  long long* cap_t = static_cast<long long*>(workspace);
  float* cap_bias = reinterpret_cast<float*>(static_cast<char*>(workspace) + 16);
  const long long t_now = ctx->t;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(cap_t, &t_now, sizeof t_now, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(cap_bias, table.data(), table.size() * sizeof(float), cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);  // the host sources leave scope here
  if (e != cudaSuccess) return fail_cuda(ctx, "capturable upload", e);
  ctx->cap_t = cap_t;
  ctx->cap_bias = cap_bias;
  ctx->cap_steps = max_steps;
  return ZERO_OK;
}

namespace {

// The device step count of a capturable context (synchronizes the stream).
zero_status read_device_count(zero_ctx* ctx, void* stream, long long* t) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(t, ctx->cap_t, sizeof *t, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail_cuda(ctx, "reading the step count", e);
  return ZERO_OK;
}

}  // namespace

zero_status zero_disable_capturable(zero_ctx* ctx, void* stream) {
  if (!ctx) return fail(nullptr, ZERO_EINVAL, "ctx is NULL");
  if (!ctx->cap_t) return fail(ctx, ZERO_ESTATE, "capturable mode is not on");
  long long t = 0;
  zero_status st = read_device_count(ctx, stream, &t);
  if (st != ZERO_OK) return st;
  // Steps past the table were skipped: they changed nothing.
  ctx->t = t < ctx->cap_steps ? t : ctx->cap_steps;
  ctx->cap_t = nullptr;
  ctx->cap_bias = nullptr;
  ctx->cap_steps = 0;
  return ZERO_OK;
}

zero_status zero_step_count(const zero_ctx* ctx, int64_t* t) {
  if (!ctx || !t) return fail(nullptr, ZERO_EINVAL, "NULL argument");
  if (ctx->cap_t) {
    zero_ctx* c = const_cast<zero_ctx*>(ctx);
    long long d = 0;
    zero_status st = read_device_count(c, nullptr, &d);
    if (st != ZERO_OK) return st;
    if (d > ctx->cap_steps) {
      *t = ctx->cap_steps;
      return fail(c, ZERO_ESTATE, "capturable table of %lld steps exhausted: %lld later step(s) were skipped",
                  static_cast<long long>(ctx->cap_steps), d - static_cast<long long>(ctx->cap_steps));
    }
    *t = d;
    return ZERO_OK;
  }
  *t = ctx->t;
  return ZERO_OK;
}

zero_status zero_last_launches(const zero_ctx* ctx, int32_t* launches) {
  if (!ctx || !launches) return fail(nullptr, ZERO_EINVAL, "NULL argument");
  *launches = ctx->last_launches;
  return ZERO_OK;
}

zero_status zero_set_lr(zero_ctx* ctx, float lr) {
  if (!ctx) return fail(nullptr, ZERO_EINVAL, "ctx is NULL");
  if (!std::isfinite(lr)) return fail(ctx, ZERO_EINVAL, "lr is not finite");
  ctx->cfg.lr = lr;
  return ZERO_OK;
}

zero_status zero_destroy(zero_ctx* ctx) {
  delete ctx;
  return ZERO_OK;
}

const char* zero_last_error(const zero_ctx* ctx) {
  return ctx ? ctx->error.c_str() : g_thread_error.c_str();
}

const char* zero_status_string(zero_status status) {
  switch (status) {
    case ZERO_OK: return "ZERO_OK";
    case ZERO_EINVAL: return "ZERO_EINVAL";
    case ZERO_ENOMEM: return "ZERO_ENOMEM";
    case ZERO_ECUDA: return "ZERO_ECUDA";
    case ZERO_ESTATE: return "ZERO_ESTATE";
    case ZERO_ENOTSUP: return "ZERO_ENOTSUP";
  }
  return "ZERO_UNKNOWN";
}

}  // extern "C"
