// ORACLE — test infrastructure only.
//
// A plain, slow, single-threaded CPU restatement of the ZeRO-1/2/3 optimizer
// step over a flattened, padded FlatParameter.  Only the tests, the smoke
// check and the benchmark's CPU-baseline leg may load this file's library.
// It shares no code, header, table or helper with the CUDA library; neither
// includes or links the other.
//
// Sources (all statements below are restated, not copied):
//  * CMU 15-779 Lecture 13 notes "Zero Redundancy and PyTorch FSDP"
//    (semidirectx.com): §0.4 (zero.py: per-layer FlatParameter, zero-padded to a
//    multiple of the device count, device d owns segment d), §2.1 (Adam),
//    §2.2 (fp32 master weights), §2.3 (16 bytes per parameter, K = 12),
//    §3.1-3.3 (the three stages), §3.4 (bit-identity with data parallelism
//    when the summation order is fixed), §3.5-3.6 (memory ledger, padding),
//    §4.3 (the missing post-update all-gather), §5.2 (FlatParameter:
//    flatten, concatenate, right-pad to a multiple of F, split evenly),
//    §9 item 2 and Exercise 5 (ledger formulas, ZeRO-3 peak).
//  * Femtotron dev log #6 "ZeRO-1 and ZeRO-2" (koas-w.github.io): the
//    ShardingStrategy protocol (make_master / reduce_grads / gather_weights /
//    post_step) and the 1-D (not by-shape) master sharding.
//  * Femtotron dev log #7 (ZeRO-2 hook: flatten the grad, zero-pad to
//    shard_size * N, reduce-scatter with AVG, keep the shard).
//  * Femtotron dev logs #4/#5 (mixed-precision step order: bf16 grad -> fp32,
//    AdamW on the fp32 master, master -> bf16 compute copy).
//
// Readings taken where the pages are silent:
//  * Reduce: each replica's gradient is widened exactly to fp32 and summed in
//    rank order 0..N-1 starting from replica 0's value, then multiplied by
//    fp32(1/N) (= 1.0f / N).  Never rounded back to bf16.
//  * Bias corrections: bc1 = 1 - beta1^t, bc2 = 1 - beta2^t evaluated in
//    double from the fp32 betas and rounded once to fp32; t = 1 on the first
//    step.  m_hat = m / bc1, v_hat = v / bc2 (fp32 divisions).
//  * (1 - beta) is the fp32 difference 1.0f - beta (exact for beta in [0.5,1]).
//  * epsilon is added outside the square root; the update is
//    w <- w - lr * (m_hat / (sqrt(v_hat) + eps)).
//  * Decoupled weight decay (AdamW) multiplies the pre-update weight by
//    fp32(1 - lr * wd) (evaluated in double, rounded once) before the Adam
//    update.
//  * Every fp32 operation is rounded on its own (built with
//    -ffp-contract=off); sqrt and division are IEEE correctly rounded.
//  * bf16 cast: round to nearest, ties to even, from the IEEE bit patterns;
//    NaN stays a (quiet) NaN of the same sign; overflow rounds to infinity.
//  * Gradient accumulation over micro-steps (Femtotron #5: no_sync micro-steps
//    accumulate into the gradient before the one reduce; the source guide's
//    Megatron main_grad: fp32 accumulation, 18 B/param): per replica and
//    element, acc = widen(micro) on the first micro-step, else
//    acc = acc + widen(micro), one fp32 addition per micro-step in micro-step
//    order.  No scaling: the pages scale the loss by 1/accum_steps instead.
//  * Gradient clipping (Femtotron #4/#5: ClipGradNorm on the fp32 gradient,
//    before AdamW; the source guide's --clip-grad / gradient_clipping): the
//    global L2 norm of the reduced gradient, sqrt(sum_j g_j^2).  Each square
//    is exact in fp64; the sum uses Neumaier's compensated summation (an
//    improved Kahan-Babuska sum), so the oracle's own rounding error stays
//    near one fp64 ulp instead of the n * 2^-53 bound of a plain running sum.
//    Coefficient min(1, max_norm / (norm + 1e-6)) evaluated in fp64 and
//    rounded once to fp32; the reduced gradient is multiplied by it (one fp32
//    multiply) before Adam.  The cap at 1 keeps a NaN (torch's
//    clip_grad_norm_ clamps the coefficient with torch.clamp, which passes
//    NaN through): a NaN norm makes every clipped gradient NaN.
//
// Parity pins: every function here is pinned by a "not gpu" test against
// values printed on the pages, closed forms, invariants or brute force.

#include <cmath>
#include <limits>
#include <cstdint>
#include <cstdlib>
#include <cstring>

namespace {

// ---------------------------------------------------------------------------
// bf16 <-> fp32 from the IEEE-754 binary32 / bfloat16 bit layouts.
// bfloat16 keeps the upper 16 bits of a binary32 value (sign, 8-bit exponent,
// 7-bit fraction).  Widening is exact: append 16 zero bits.
// ---------------------------------------------------------------------------
float widen_bf16(uint16_t h) {
  uint32_t bits = static_cast<uint32_t>(h) << 16;
  float f;
  std::memcpy(&f, &bits, sizeof f);
  return f;
}

// Round-to-nearest-even narrowing.  Let hi be the upper 16 bits (the value
// truncated toward zero in magnitude) and lo the 16 discarded bits.  If lo is
// above half an ulp of bf16 (0x8000) the magnitude rounds up; if exactly half,
// it rounds up only when hi is odd; otherwise it is kept.  Rounding up is an
// increment of the 16-bit magnitude pattern, which carries into the exponent
// and reaches the infinity pattern on overflow, as IEEE rounding requires.
uint16_t narrow_bf16(float x) {
  uint32_t bits;
  std::memcpy(&bits, &x, sizeof bits);
  const uint32_t exponent = (bits >> 23) & 0xFFu;
  const uint32_t fraction = bits & 0x7FFFFFu;
  if (exponent == 0xFFu && fraction != 0u) {
    // NaN: keep sign and the top fraction bits, force the quiet bit.
    return static_cast<uint16_t>((bits >> 16) | 0x0040u);
  }
  uint16_t hi = static_cast<uint16_t>(bits >> 16);
  const uint32_t lo = bits & 0xFFFFu;
  bool round_up;
  if (lo > 0x8000u) {
    round_up = true;
  } else if (lo == 0x8000u) {
    round_up = (hi & 1u) != 0u;
  } else {
    round_up = false;
  }
  if (round_up) hi = static_cast<uint16_t>(hi + 1u);
  return hi;
}

struct Hyper {
  float lr, beta1, beta2, eps, weight_decay;
  int adamw;
  int n_ranks;
  int grad_dtype;  // 0 = bf16, 1 = fp32
};

// Scalars of step t, each evaluated from its definition.
struct StepScalars {
  float one_minus_beta1;  // 1 - beta1  (fp32)
  float one_minus_beta2;  // 1 - beta2  (fp32)
  float bc1;              // 1 - beta1^t
  float bc2;              // 1 - beta2^t
  float decay;            // 1 - lr * wd  (AdamW)
  float inv_n;            // 1 / N
};

StepScalars step_scalars(const Hyper& h, int64_t t) {
  StepScalars s;
  s.one_minus_beta1 = 1.0f - h.beta1;
  s.one_minus_beta2 = 1.0f - h.beta2;
  s.bc1 = static_cast<float>(1.0 - std::pow(static_cast<double>(h.beta1), static_cast<double>(t)));
  s.bc2 = static_cast<float>(1.0 - std::pow(static_cast<double>(h.beta2), static_cast<double>(t)));
  s.decay = static_cast<float>(1.0 - static_cast<double>(h.lr) * static_cast<double>(h.weight_decay));
  s.inv_n = 1.0f / static_cast<float>(h.n_ranks);
  return s;
}

// Replica r's gradient at flat index j, widened to fp32.
float replica_grad(const Hyper& h, const void* const* grads, int r, int64_t j) {
  if (h.grad_dtype == 0) {
    return widen_bf16(static_cast<const uint16_t*>(grads[r])[j]);
  }
  return static_cast<const float*>(grads[r])[j];
}

// Reduce-scatter stand-in for one element: the N replica gradients summed in
// fp32 in fixed rank order 0, 1, ..., N-1, then scaled by 1/N (the AVG of the
// Femtotron ZeRO-2 hook, summed in the order the bit-identity argument of the
// lecture notes §3.4 requires).
float reduce_element(const Hyper& h, const StepScalars& s, const void* const* grads, int64_t j) {
  float acc = replica_grad(h, grads, 0, j);
  for (int r = 1; r < h.n_ranks; ++r) {
    acc = acc + replica_grad(h, grads, r, j);
  }
  return acc * s.inv_n;
}

// Adam (lecture notes §2.1) on one fp32 master element, with the optional
// decoupled weight decay of AdamW (Femtotron #4/#5 runs AdamW on the fp32
// master):
//   m <- beta1 m + (1 - beta1) g
//   v <- beta2 v + (1 - beta2) g^2
//   w <- w - lr * m_hat / (sqrt(v_hat) + eps),  m_hat = m / bc1, v_hat = v / bc2
void adam_element(const Hyper& h, const StepScalars& s, float g, float* w, float* m, float* v) {
  float weight = *w;
  if (h.adamw) {
    weight = weight * s.decay;
  }
  const float m_new = h.beta1 * (*m) + s.one_minus_beta1 * g;
  const float g_squared = g * g;
  const float v_new = h.beta2 * (*v) + s.one_minus_beta2 * g_squared;
  const float m_hat = m_new / s.bc1;
  const float v_hat = v_new / s.bc2;
  const float denom = std::sqrt(v_hat) + h.eps;
  const float ratio = m_hat / denom;
  weight = weight - h.lr * ratio;
  *w = weight;
  *m = m_new;
  *v = v_new;
}

// Compensated running sum (Neumaier): sum holds the rounded total and comp
// the rounding errors lost by each addition, recovered exactly.
// Neumaier's compensated sum of the finite terms; non-finite terms (an
// infinite or NaN square) go to a plain sum of their own, so the result is
// what the exact sum is under IEEE arithmetic: +inf if some term is +inf and
// none is NaN, NaN if some term is NaN.  (Fed to the compensation, an
// infinite term would turn into inf - inf = NaN.)
struct CompensatedSum {
  double sum = 0.0;
  double comp = 0.0;
  double special = 0.0;
  void add(double x) {
    if (!std::isfinite(x)) {
      special = special + x;
      return;
    }
    const double t = sum + x;
    if (std::fabs(sum) >= std::fabs(x)) {
      comp = comp + ((sum - t) + x);
    } else {
      comp = comp + ((x - t) + sum);
    }
    sum = t;
  }
  double value() const { return special != 0.0 ? special : sum + comp; }  // NaN != 0 holds too
};

// Global L2 norm of the reduced gradient over flat elements [0, n); every
// square is exact in fp64.
double grad_norm(const Hyper& h, const StepScalars& s, const void* const* grads, int64_t n) {
  CompensatedSum sum_sq;
  for (int64_t j = 0; j < n; ++j) {
    const double g = static_cast<double>(reduce_element(h, s, grads, j));
    sum_sq.add(g * g);
  }
  return std::sqrt(sum_sq.value());
}

// Clip coefficient: scale the gradient down to max_norm when its norm is
// larger; 1 otherwise; NaN when the norm is NaN.
float clip_coefficient(double norm, float max_norm) {
  const double coef = static_cast<double>(max_norm) / (norm + 1e-6);
  if (std::isnan(coef)) return std::numeric_limits<float>::quiet_NaN();
  return coef < 1.0 ? static_cast<float>(coef) : 1.0f;
}

Hyper hyper_from(const float* f, const int32_t* i) {
  Hyper h;
  h.lr = f[0];
  h.beta1 = f[1];
  h.beta2 = f[2];
  h.eps = f[3];
  h.weight_decay = f[4];
  h.adamw = i[0];
  h.n_ranks = i[1];
  h.grad_dtype = i[2];
  return h;
}

}  // namespace

extern "C" {

// ---------------------------------------------------------------------------
// bf16 conversions exposed for pinning.
// ---------------------------------------------------------------------------
uint16_t oracle_bf16_round(float x) { return narrow_bf16(x); }
float oracle_bf16_widen(uint16_t h) { return widen_bf16(h); }

void oracle_bf16_round_array(int64_t n, const float* x, uint16_t* out) {
  for (int64_t k = 0; k < n; ++k) out[k] = narrow_bf16(x[k]);
}

// ---------------------------------------------------------------------------
// FlatParameter layout (lecture notes §0.4, §5.2; Femtotron #6, #7).
// Params are taken in caller order; param p belongs to unit param_unit[p]
// (nondecreasing, units numbered 0..n_units-1).  For unit i:
//   numel_i  = sum of its params' numel
//   padded_i = numel_i right-padded with zeros to a multiple of F
//   shard_i  = padded_i / F          (rank d owns [d*shard_i, (d+1)*shard_i))
//   base_i   = sum over k < i of padded_k
// F is the number of shards: N for stages 1-3, 1 for stage 0 (plain data
// parallelism keeps everything on every rank and needs no padding).
// Returns 0 on success, -1 on invalid input.
// ---------------------------------------------------------------------------
int oracle_layout(int32_t n_params, const int64_t* param_numel, const int32_t* param_unit,
                  int32_t n_ranks, int32_t stage, int32_t n_units,
                  int64_t* unit_numel, int64_t* unit_padded, int64_t* unit_shard,
                  int64_t* unit_base, int64_t* param_offset, int64_t* total_padded) {
  if (n_ranks < 1 || n_units < 0 || n_params < 0) return -1;
  const int64_t F = (stage == 0) ? 1 : n_ranks;
  for (int32_t i = 0; i < n_units; ++i) unit_numel[i] = 0;
  int32_t previous_unit = 0;
  for (int32_t p = 0; p < n_params; ++p) {
    const int32_t u = param_unit[p];
    if (u < 0 || u >= n_units || u < previous_unit || param_numel[p] < 0) return -1;
    previous_unit = u;
    unit_numel[u] += param_numel[p];
  }
  int64_t base = 0;
  for (int32_t i = 0; i < n_units; ++i) {
    // Smallest multiple of F that is >= numel_i.
    const int64_t remainder = unit_numel[i] % F;
    const int64_t pad = (remainder == 0) ? 0 : (F - remainder);
    unit_padded[i] = unit_numel[i] + pad;
    unit_shard[i] = unit_padded[i] / F;
    unit_base[i] = base;
    base += unit_padded[i];
  }
  *total_padded = base;
  // Params sit back to back inside their unit, in caller order.
  int64_t cursor = 0;
  int32_t current = -1;
  for (int32_t p = 0; p < n_params; ++p) {
    const int32_t u = param_unit[p];
    if (u != current) {
      current = u;
      cursor = unit_base[u];
    }
    param_offset[p] = cursor;
    cursor += param_numel[p];
  }
  return 0;
}

// ---------------------------------------------------------------------------
// Model-state ledger, bytes per rank (lecture notes §2.3, §9 item 2):
// bf16 params 2, bf16 grads 2, optimizer state K = 12 (fp32 master, m, v).
//   stage 0 (DP):   2 P + 2 P + 12 P          = 16 P
//   stage 1 (P_os): 2 P + 2 P + 12 S          = 4 P + 12 P/N
//   stage 2 (+g):   2 P + 2 S + 12 S          = 2 P + 14 P/N
//   stage 3 (+p):   2 S + 2 S + 12 S          = 16 P/N
// with P the padded total and S the sum of the per-unit shard lengths
// (every rank holds exactly S elements of each sharded state).
// ---------------------------------------------------------------------------
void oracle_state_bytes(int32_t n_units, const int64_t* unit_padded, int32_t n_ranks,
                        int32_t stage, int64_t* per_rank_bytes) {
  int64_t P = 0;
  int64_t S = 0;
  for (int32_t i = 0; i < n_units; ++i) {
    P += unit_padded[i];
    S += unit_padded[i] / n_ranks;
  }
  int64_t bytes = 0;
  if (stage == 0) {
    bytes = 2 * P + 2 * P + 12 * P;
  } else if (stage == 1) {
    bytes = 2 * P + 2 * P + 12 * S;
  } else if (stage == 2) {
    bytes = 2 * P + 2 * S + 12 * S;
  } else {
    bytes = 2 * S + 2 * S + 12 * S;
  }
  for (int32_t r = 0; r < n_ranks; ++r) per_rank_bytes[r] = bytes;
}

// ZeRO-3 model-state peak on one rank during backward (lecture notes §3.5 and
// Exercise 5): units are processed from the last to the first.  While unit k
// is processed a rank holds its resident shards (bf16 params 2 S + fp32
// states 12 S), the bf16 grad shards of the units already reduce-scattered
// (k+1 .. last), and the full bf16 params and full bf16 grads of unit k.
// Returns the maximum over k and writes the unit where it occurs.
int64_t oracle_zero3_backward_peak(int32_t n_units, const int64_t* unit_padded, int32_t n_ranks,
                                   int32_t* peak_unit) {
  int64_t S = 0;
  for (int32_t i = 0; i < n_units; ++i) S += unit_padded[i] / n_ranks;
  const int64_t resident = 2 * S + 12 * S;
  int64_t best = resident;
  int32_t best_unit = -1;
  for (int32_t k = n_units - 1; k >= 0; --k) {
    int64_t reduced_grad_shards = 0;
    for (int32_t i = k + 1; i < n_units; ++i) reduced_grad_shards += 2 * (unit_padded[i] / n_ranks);
    const int64_t full_unit = 2 * unit_padded[k] + 2 * unit_padded[k];
    const int64_t at_k = resident + reduced_grad_shards + full_unit;
    if (at_k > best) {
      best = at_k;
      best_unit = k;
    }
  }
  if (peak_unit) *peak_unit = best_unit;
  return best;
}

// ---------------------------------------------------------------------------
// make_master: the fp32 master is the caller's params flattened in order into
// the padded layout; pads are zero; Adam moments start at zero; the bf16
// compute copy is the bf16 cast of the master.
// ---------------------------------------------------------------------------
void oracle_make_master(int32_t n_params, const int64_t* param_numel, const int64_t* param_offset,
                        const float* const* init_params, int64_t total_padded,
                        float* master, float* m, float* v, uint16_t* param16) {
  for (int64_t j = 0; j < total_padded; ++j) {
    master[j] = 0.0f;
    m[j] = 0.0f;
    v[j] = 0.0f;
  }
  for (int32_t p = 0; p < n_params; ++p) {
    for (int64_t e = 0; e < param_numel[p]; ++e) {
      master[param_offset[p] + e] = init_params[p][e];
    }
  }
  for (int64_t j = 0; j < total_padded; ++j) param16[j] = narrow_bf16(master[j]);
}

// Reduce one flat index j over the N replicas (exposed for pinning).
// hyper_f = {lr, beta1, beta2, eps, weight_decay}, hyper_i = {adamw, N, grad_dtype}.
float oracle_reduce(const float* hyper_f, const int32_t* hyper_i, const void* const* grads, int64_t j) {
  const Hyper h = hyper_from(hyper_f, hyper_i);
  const StepScalars s = step_scalars(h, 1);
  return reduce_element(h, s, grads, j);
}

// Global L2 norm of the reduced gradient of n flat elements (exposed for pinning).
double oracle_grad_norm(const float* hyper_f, const int32_t* hyper_i, int64_t n, const void* const* grads) {
  const Hyper h = hyper_from(hyper_f, hyper_i);
  const StepScalars s = step_scalars(h, 1);
  return grad_norm(h, s, grads, n);
}

float oracle_clip_coef(double norm, float max_norm) { return clip_coefficient(norm, max_norm); }

// How many flat elements j in [0, n) have a reduced gradient (the rank-order
// fp32 sum times 1/N, before any clipping) that is not finite: a replica
// holds an inf or a NaN there, or the fp32 sum of the replicas overflows.
// This is what the overflow check at the start of DeepSpeed's ZeRO step
// looks for (source guide §4.3: step() checks for overflow, then clips).
int64_t oracle_nonfinite_count(const float* hyper_f, const int32_t* hyper_i, int64_t n, const void* const* grads) {
  const Hyper h = hyper_from(hyper_f, hyper_i);
  const StepScalars s = step_scalars(h, 1);
  int64_t count = 0;
  for (int64_t j = 0; j < n; ++j) {
    if (!std::isfinite(reduce_element(h, s, grads, j))) ++count;
  }
  return count;
}

// The fp32 scalars of step t (exposed for pinning):
// out = {1-beta1, 1-beta2, bc1, bc2, decay, 1/N}.
void oracle_step_scalars(const float* hyper_f, const int32_t* hyper_i, int64_t t, float* out) {
  const Hyper h = hyper_from(hyper_f, hyper_i);
  const StepScalars s = step_scalars(h, t);
  out[0] = s.one_minus_beta1;
  out[1] = s.one_minus_beta2;
  out[2] = s.bc1;
  out[3] = s.bc2;
  out[4] = s.decay;
  out[5] = s.inv_n;
}

// ---------------------------------------------------------------------------
// The ZeRO step, literally, over N simulated ranks (lecture notes §3.1-3.3,
// Femtotron #6/#7), for step number t (1 on the first step):
//   1. reduce-scatter: rank d obtains, for its shard of every unit, the
//      fixed-order fp32 average of the N replicas' gradients;
//   2. rank d runs Adam on its fp32 master / m / v shard;
//   3. rank d casts its updated master shard to bf16;
//   4. all-gather (stages 1-2): every rank's bf16 shard is copied into every
//      rank's full bf16 parameter copy.  Stage 3 keeps only the shard (the
//      gather is deferred to gather_weights before use).
// grads: N pointers to full padded gradient buffers (bf16 or fp32).
// param16_copies: n_copies full padded bf16 buffers back to back.  With
// n_copies == N every rank keeps its own copy (stages 1-2) and step 4 is
// literal; with n_copies == 1 all ranks share one buffer (the state after the
// all-gather) and step 4 has nothing left to copy.
// plant_skip_allgather != 0 omits step 4: a deliberately wrong variant used by
// a test to show the silent divergence described in the notes' §4.3.
// Returns 0, or -1 on invalid input / allocation failure.
// ---------------------------------------------------------------------------
int oracle_zero_step(const float* hyper_f, const int32_t* hyper_i, int32_t stage, int64_t t,
                     int32_t n_units, const int64_t* unit_padded, const int64_t* unit_base,
                     const void* const* grads, float* master, float* m, float* v,
                     uint16_t* param16_copies, int32_t n_copies, int32_t plant_skip_allgather,
                     float max_norm, double* norm_out) {
  const Hyper h = hyper_from(hyper_f, hyper_i);
  if (stage < 1 || stage > 3 || t < 1) return -1;
  if (n_copies != 1 && n_copies != h.n_ranks) return -1;
  if (stage == 3 && n_copies != 1) return -1;
  const int N = h.n_ranks;
  const StepScalars s = step_scalars(h, t);
  int64_t total = 0;
  for (int32_t i = 0; i < n_units; ++i) total += unit_padded[i];

  // 1. reduce-scatter into per-rank fp32 gradient shards, stored at the
  //    shard's own flat positions.
  float* grad_shards = static_cast<float*>(std::malloc(sizeof(float) * (total > 0 ? total : 1)));
  if (!grad_shards) return -1;
  for (int32_t i = 0; i < n_units; ++i) {
    const int64_t shard = unit_padded[i] / N;
    for (int d = 0; d < N; ++d) {
      for (int64_t e = 0; e < shard; ++e) {
        const int64_t j = unit_base[i] + d * shard + e;
        grad_shards[j] = reduce_element(h, s, grads, j);
      }
    }
  }
  // Optional global-norm clipping of the reduced gradient: the norm over all
  // shards of all units, in flat element order; every shard is then scaled
  // by the same coefficient.
  const bool clip = max_norm > 0.0f;
  float coef = 1.0f;
  if (clip) {
    CompensatedSum sum_sq;
    for (int64_t j = 0; j < total; ++j) {
      const double g = static_cast<double>(grad_shards[j]);
      sum_sq.add(g * g);
    }
    const double norm = std::sqrt(sum_sq.value());
    coef = clip_coefficient(norm, max_norm);
    if (norm_out) *norm_out = norm;
  }
  // 2. + 3. each rank updates its own shard and casts it into its own copy.
  for (int32_t i = 0; i < n_units; ++i) {
    const int64_t shard = unit_padded[i] / N;
    for (int d = 0; d < N; ++d) {
      uint16_t* own_copy = param16_copies + (n_copies == 1 ? 0 : static_cast<int64_t>(d) * total);
      for (int64_t e = 0; e < shard; ++e) {
        const int64_t j = unit_base[i] + d * shard + e;
        const float g = clip ? grad_shards[j] * coef : grad_shards[j];
        adam_element(h, s, g, &master[j], &m[j], &v[j]);
        own_copy[j] = narrow_bf16(master[j]);
      }
    }
  }
  // 4. all-gather of the bf16 shards into every rank's full copy.
  if (stage != 3 && n_copies == N && !plant_skip_allgather) {
    for (int32_t i = 0; i < n_units; ++i) {
      const int64_t shard = unit_padded[i] / N;
      for (int d = 0; d < N; ++d) {
        const uint16_t* owner = param16_copies + static_cast<int64_t>(d) * total;
        for (int q = 0; q < N; ++q) {
          if (q == d) continue;
          uint16_t* receiver = param16_copies + static_cast<int64_t>(q) * total;
          for (int64_t e = 0; e < shard; ++e) {
            const int64_t j = unit_base[i] + d * shard + e;
            receiver[j] = owner[j];
          }
        }
      }
    }
  }
  std::free(grad_shards);
  return 0;
}

// Plain data parallelism (stage 0, the unsharded reference): every rank
// averages the full gradient (all-reduce, same fixed rank order) and updates
// the whole fp32 master itself; one element range [0, n).
void oracle_dp_step(const float* hyper_f, const int32_t* hyper_i, int64_t t, int64_t n,
                    const void* const* grads, float* master, float* m, float* v, uint16_t* param16,
                    float max_norm, double* norm_out) {
  const Hyper h = hyper_from(hyper_f, hyper_i);
  const StepScalars s = step_scalars(h, t);
  const bool clip = max_norm > 0.0f;
  float coef = 1.0f;
  if (clip) {
    const double norm = grad_norm(h, s, grads, n);
    coef = clip_coefficient(norm, max_norm);
    if (norm_out) *norm_out = norm;
  }
  for (int64_t j = 0; j < n; ++j) {
    const float reduced = reduce_element(h, s, grads, j);
    const float g = clip ? reduced * coef : reduced;
    adam_element(h, s, g, &master[j], &m[j], &v[j]);
    param16[j] = narrow_bf16(master[j]);
  }
}

// Step t on a window of n consecutive flat elements.  grads are N pointers to
// the window's replica gradients; master/m/v/param16 point at the window.
// Adam is elementwise (lecture notes §3.1), so a window taken anywhere in a
// large buffer is updated exactly as in the full step.
// clip_coef != 1 scales the reduced gradient (the coefficient of a global
// norm computed over the whole buffer, e.g. by oracle_grad_norm).
void oracle_step_window(const float* hyper_f, const int32_t* hyper_i, int64_t t, int64_t n,
                        const void* const* grads, float* master, float* m, float* v, uint16_t* param16,
                        float clip_coef) {
  const Hyper h = hyper_from(hyper_f, hyper_i);
  const StepScalars s = step_scalars(h, t);
  const bool clip = clip_coef != 1.0f;
  for (int64_t j = 0; j < n; ++j) {
    const float reduced = reduce_element(h, s, grads, j);
    const float g = clip ? reduced * clip_coef : reduced;
    adam_element(h, s, g, &master[j], &m[j], &v[j]);
    param16[j] = narrow_bf16(master[j]);
  }
}

// Checkpoint export (lecture notes §5.2: the pads are not parameters; the
// source guide's resharding checkpoints, Femtotron #5's dp_size change): the
// real elements of each unit, in unit order, back to back (the parameters in
// caller order), for one fp32 state array.
void oracle_export(int32_t n_units, const int64_t* unit_numel, const int64_t* unit_base,
                   const float* padded, float* compact) {
  int64_t out = 0;
  for (int32_t i = 0; i < n_units; ++i) {
    for (int64_t e = 0; e < unit_numel[i]; ++e) compact[out + e] = padded[unit_base[i] + e];
    out += unit_numel[i];
  }
}

// Checkpoint import: the inverse into a padded layout of any shard count; the
// pads are zero.
void oracle_import(int32_t n_units, const int64_t* unit_numel, const int64_t* unit_base, int64_t total_padded,
                   const float* compact, float* padded) {
  for (int64_t j = 0; j < total_padded; ++j) padded[j] = 0.0f;
  int64_t in = 0;
  for (int32_t i = 0; i < n_units; ++i) {
    for (int64_t e = 0; e < unit_numel[i]; ++e) padded[unit_base[i] + e] = compact[in + e];
    in += unit_numel[i];
  }
}

// fp32 gradient accumulation of one micro-step for N replicas over n flat
// elements: micro[r] are bf16, acc[r] fp32.  first != 0 starts the sum
// (whatever acc held is discarded).
void oracle_accumulate(int32_t n_ranks, int64_t n, const uint16_t* const* micro, float* const* acc,
                       int32_t first) {
  for (int32_t r = 0; r < n_ranks; ++r) {
    for (int64_t j = 0; j < n; ++j) {
      const float g = widen_bf16(micro[r][j]);
      acc[r][j] = first ? g : acc[r][j] + g;
    }
  }
}

// ZeRO-3 gather of one unit (lecture notes §3.3, §5.1): the N bf16 shards of
// the unit, taken in rank order, concatenated into a full unit buffer of
// padded_i elements.
void oracle_gather_unit(int64_t unit_base, int64_t unit_padded, int32_t n_ranks,
                        const uint16_t* param16, uint16_t* out) {
  const int64_t shard = unit_padded / n_ranks;
  for (int32_t d = 0; d < n_ranks; ++d) {
    const uint16_t* shard_d = param16 + unit_base + d * shard;
    for (int64_t e = 0; e < shard; ++e) out[d * shard + e] = shard_d[e];
  }
}

}  // extern "C"
