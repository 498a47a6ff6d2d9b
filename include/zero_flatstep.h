/*
 * zero_flatstep.h — C ABI of the GB300 (sm_103a) ZeRO-1/2/3 optimizer step
 * over a flattened, padded 1-D FlatParameter, with N data-parallel replicas
 * simulated on one GPU.
 *
 * The calls follow the ShardingStrategy protocol of Femtotron dev log #6
 * ("ZeRO-1 and ZeRO-2: abstraction design", section "ShardingStrategy as a
 * first-class abstraction"): make_master / reduce_grads / gather_weights /
 * post_step are the four points where ZeRO enters a training step, with the
 * optimizer step between reduce_grads and gather_weights.  Plain data
 * parallelism (stage 0, "NoShard") runs through the same calls.
 *
 * Conventions for every call:
 *  - Plain pointers and sizes only.  "dev" pointers are CUDA device memory
 *    owned by the caller; the library never allocates, frees or retains
 *    device memory, and holds only host-side metadata in a zero_ctx.  Two
 *    stated exceptions: zero_clip_grad_norm_static's fixed scratch array in
 *    the library's own device memory, and an offload context's host worker
 *    threads (see the ZeRO-Offload calls).
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Device work is enqueued on it asynchronously; the caller keeps
 *    every buffer alive until that work has completed on the stream.  The
 *    ZeRO-3 gathers and the clip norm pass are launched with programmatic
 *    stream serialization: their thread blocks may become resident while the
 *    kernel before them on the stream finishes, but each waits for that
 *    kernel to complete (and its writes to be visible) before it reads
 *    anything, so the stream's ordering is the usual one.
 *  - Every call returns a zero_status; nothing crosses the ABI as an
 *    exception.  A call that fails leaves the context unchanged.  The text of
 *    the last error is available from zero_last_error().
 *  - A context is not thread-safe: calls on one context must not overlap.
 */
#ifndef ZERO_FLATSTEP_H
#define ZERO_FLATSTEP_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum zero_status {
  ZERO_OK = 0,
  ZERO_EINVAL = 1,   /* invalid argument (null/misaligned pointer, bad size, bad config) */
  ZERO_ENOMEM = 2,   /* host allocation of metadata failed */
  ZERO_ECUDA = 3,    /* a CUDA runtime call or kernel launch failed */
  ZERO_ESTATE = 4,   /* call not allowed in the context's current state */
  ZERO_ENOTSUP = 5   /* valid request this build does not support */
} zero_status;

typedef enum zero_grad_dtype {
  ZERO_GRAD_BF16 = 0,  /* replica gradients are bf16 (2 bytes/element) */
  ZERO_GRAD_FP32 = 1   /* replica gradients are fp32 (fp32 gradient accumulation) */
} zero_grad_dtype;

/*
 * Optimizer and sharding configuration.
 *  stage       0 = plain data parallelism (no sharding, no padding), 1 = ZeRO-1
 *              (optimizer state sharded), 2 = ZeRO-2 (+ gradients), 3 = ZeRO-3
 *              (+ parameters) — CMU 15-779 Lecture 13 notes §3.1-3.3.
 *  n_ranks     N simulated data-parallel replicas, 1..16.
 *  grad_dtype  zero_grad_dtype of the replica gradient buffers.
 *  adamw       1 = decoupled weight decay (AdamW), 0 = Adam (weight_decay must be 0).
 *  lr, beta1, beta2, eps, weight_decay: fp32 Adam hyper-parameters
 *              (notes §2.1); beta1, beta2 in [0, 1), eps >= 0, lr finite.
 */
typedef struct zero_config {
  int32_t stage;
  int32_t n_ranks;
  int32_t grad_dtype;
  int32_t adamw;
  float lr;
  float beta1;
  float beta2;
  float eps;
  float weight_decay;
} zero_config;

/*
 * Caller-allocated device buffers, each of `padded_numel` elements (see
 * zero_plan / zero_padded_numel) and 16-byte aligned:
 *  master      fp32 master weights (the optimizer's copy, notes §2.2)
 *  exp_avg     fp32 Adam first moment m
 *  exp_avg_sq  fp32 Adam second moment v
 *  param16     bf16 parameters.  Stages 0-2: the full compute copy every
 *              replica holds after the all-gather.  Stage 3: the rank-major
 *              shard storage (rank d's shard of unit i at base_i + d*shard_i),
 *              which has the same byte layout.
 */
typedef struct zero_buffers {
  float* master;
  float* exp_avg;
  float* exp_avg_sq;
  void* param16;
} zero_buffers;

typedef struct zero_ctx zero_ctx;

/*
 * zero_plan — FlatParameter layout only (host, no device work).
 * Lecture notes §0.4 and §5.2: each unit's parameters are flattened and
 * concatenated in caller order, right-padded with zeros to a multiple of the
 * shard count F (N for stages 1-3, 1 for stage 0) and split into F equal
 * shards; rank d owns shard d.  Femtotron dev log #6 ("master is sharded 1-D,
 * not by shape").
 *  param_numel[n_params]  element count of each parameter (>= 0)
 *  param_unit[n_params]   unit (FlatParameter) id of each parameter; ids are
 *                         nondecreasing and start at 0 (n_units = last id + 1;
 *                         a skipped id is an empty unit)
 *  out                    receives a context usable for layout / ledger queries;
 *                         step calls on it return ZERO_ESTATE.
 * Errors: ZERO_EINVAL for a bad config, negative sizes, decreasing unit ids or
 * null pointers with n_params > 0; ZERO_ENOMEM.
 */
zero_status zero_plan(const zero_config* cfg, const int64_t* param_numel, const int32_t* param_unit,
                      int32_t n_params, zero_ctx** out);

/*
 * zero_make_master — the protocol's make_master: plan the layout (as
 * zero_plan), then build the fp32 master from the caller's fp32 parameters:
 * copy parameter p (init_params[p], param_numel[p] fp32 device elements,
 * 4-byte aligned) to its flat offset, zero every pad, zero m and v, write
 * param16 = bf16(master) (round to nearest even) and set the step count t = 0.
 * Enqueued on `stream`; init_params may be released once it completes.
 * Errors: as zero_plan, plus ZERO_EINVAL for a null `bufs`, a null or
 * non-16-byte-aligned buffer, a null init pointer for a non-empty parameter,
 * or a pointer that is not device memory; ZERO_ECUDA on launch failure.
 */
zero_status zero_make_master(const zero_config* cfg, const int64_t* param_numel,
                             const int32_t* param_unit, int32_t n_params,
                             const float* const* init_params, const zero_buffers* bufs,
                             void* stream, zero_ctx** out);

/* Number of units; total padded and unpadded element counts. */
zero_status zero_num_units(const zero_ctx* ctx, int32_t* n_units);
zero_status zero_padded_numel(const zero_ctx* ctx, int64_t* padded, int64_t* numel);

/*
 * zero_layout — unit i's element count, padded count (multiple of F), shard
 * length (padded / F) and flat base offset (sum of earlier padded counts).
 * ZERO_EINVAL if unit is out of range.
 */
zero_status zero_layout(const zero_ctx* ctx, int32_t unit, int64_t* numel, int64_t* padded,
                        int64_t* shard, int64_t* base);

/* Flat offset of parameter p inside the padded buffer. */
zero_status zero_param_offset(const zero_ctx* ctx, int32_t param, int64_t* offset);

/*
 * zero_state_bytes — per-rank model-state bytes of this layout under `stage`
 * (lecture notes §2.3 and §9 item 2: bf16 params 2, bf16 grads 2, optimizer
 * state K = 12 bytes per element; stage 1 shards K, stage 2 also the grads,
 * stage 3 also the params): 16P, 4P + 12S, 2P + 14S, 16S with P the total
 * and S the per-rank shard total of the layout as `stage` pads it with the
 * context's N — no padding for stage 0, each unit padded to a multiple of N
 * for stages 1-3 (notes §3.6) — whatever stage the context itself runs (a
 * stage-0 context, which does not pad, still reports the shards a sharded
 * stage would hold).  per_rank_bytes has n_ranks entries.
 */
zero_status zero_state_bytes(const zero_ctx* ctx, int32_t stage, int64_t* per_rank_bytes);

/*
 * zero_stage3_peak_bytes — ZeRO-3 model-state peak of one rank during
 * backward (lecture notes §3.5 and §11 Exercise 5): resident shards, plus the
 * grad shards of units already reduce-scattered, plus the full bf16 params and
 * grads of the unit being processed (units processed last to first), each
 * unit padded to a multiple of N as stage 3 pads it.
 * peak_unit receives the unit where the peak occurs (-1 if none).
 */
zero_status zero_stage3_peak_bytes(const zero_ctx* ctx, int64_t* peak_bytes, int32_t* peak_unit);

/*
 * zero_reduce_grads — the protocol's reduce_grads (Femtotron dev log #7, the
 * ZeRO-2 post-accumulate-grad hook: flatten, zero-pad, reduce-scatter AVG).
 * Registers the N replicas' gradients of one unit (unit >= 0: N pointers to
 * padded_i elements each) or of the whole buffer (unit == -1: N pointers to
 * padded_numel elements each).  Pad entries must be zero, as the hook's zero
 * padding makes them.  The reduction itself — the rank-order fp32 sum scaled
 * by 1/N, the local stand-in for reduce-scatter — is fused into zero_step, so
 * this call does no device work; the buffers must stay valid and unchanged
 * until the zero_step that consumes them has completed on its stream.
 * Registering a unit again replaces its pointers.
 * Errors: ZERO_EINVAL (unit out of range, null pointer, pointer not aligned to
 * the element size); ZERO_ESTATE if no buffers are bound, a step is pending
 * its post_step, or a clip is pending (zero_clip_grad_norm ran on the
 * gradients registered before it: register every unit first, then clip).
 */
zero_status zero_reduce_grads(zero_ctx* ctx, int32_t unit, const void* const* replica_grads,
                              void* stream);

/*
 * zero_accumulate_grads — fp32 gradient accumulation of one micro-step
 * (Femtotron dev log #5: no_sync micro-steps accumulate before the single
 * reduce; the source guide's Megatron main_grad: fp32 accumulation, the
 * 18 B/param case).  For each replica r and element j of the unit (unit >= 0:
 * padded_i elements) or of the whole buffer (unit == -1: padded_numel):
 *   acc[r][j] = (first ? 0 : acc[r][j]) + float(micro[r][j])
 * one fp32 addition per micro-step, no scaling (scale the loss by
 * 1/accum_steps, as the pages do).  micro: N bf16 device buffers (2-byte
 * aligned); acc: N fp32 device buffers (4-byte aligned), caller-owned; both
 * 16-byte aligned for the vector kernel.  The accumulators are then
 * registered with zero_reduce_grads on a context whose grad_dtype is fp32.
 * Enqueued on `stream`; no context state changes.
 * Errors: ZERO_EINVAL (grad_dtype is not fp32, unit out of range, null or
 * misaligned pointer); ZERO_ESTATE (no buffers bound); ZERO_ECUDA.
 */
zero_status zero_accumulate_grads(zero_ctx* ctx, int32_t unit, const void* const* micro_grads_bf16,
                                  float* const* accumulators, int32_t first, void* stream);

/*
 * zero_step — one optimizer step, t <- t + 1, in one fused pass over the
 * padded flat buffer (lecture notes §2.1-§3.3; Femtotron dev logs #4/#5 step
 * order).  For every element j of every rank's shard:
 *   g  = ((G_0[j] + G_1[j]) + ... + G_{N-1}[j]) * (1/N)      fp32, rank order
 *   w  = w * (1 - lr*wd)                                      AdamW only
 *   m  = beta1*m + (1-beta1)*g;  v = beta2*v + (1-beta2)*g*g
 *   w  = w - lr * ((m / (1-beta1^t)) / (sqrt(v / (1-beta2^t)) + eps))
 *   param16[j] = bf16_rne(w)     (the all-gather's stand-in for stages 0-2)
 * Every operation is a separately rounded IEEE fp32 operation (no FMA
 * contraction, IEEE division and square root).  After zero_clip_grad_norm,
 * g is multiplied by the clip coefficient before Adam.  Requires every unit's
 * gradients registered since the last post_step.
 * In capturable mode (zero_enable_capturable) the bias corrections come
 * from the device table and one more one-thread launch advances the device
 * step count.
 * Errors: ZERO_ESTATE (no buffers, missing gradients, step already taken
 * without post_step, an offload context — its step is zero_offload_step);
 * ZERO_ECUDA (a launch failed; t is left unchanged, but
 * when a step needs more than one launch — more than 48 gradient segments, or
 * both aligned and unaligned ones — launches enqueued before the failing one
 * have updated their elements).
 */
zero_status zero_step(zero_ctx* ctx, void* stream);

/*
 * zero_clip_workspace_bytes — size of the device workspace zero_clip_grad_norm
 * needs for this layout: 32 bytes of header plus 8 bytes per norm chunk
 * (every unit is cut into chunks of 16,384 elements).
 */
zero_status zero_clip_workspace_bytes(const zero_ctx* ctx, int64_t* bytes);

/*
 * zero_count_nonfinite — overflow count of the step.  DeepSpeed's ZeRO step
 * checks the gradients for overflow before it clips and updates (source guide
 * §4.3); here the fused step counts, at no extra memory traffic, the elements
 * whose reduced gradient g = (sum of the N replicas, rank order, fp32) / N is
 * inf or NaN — a non-finite replica gradient or an fp32 overflow of the sum —
 * and adds that number to *counter.  Every later zero_step (and
 * zero_offload_step) of this context counts, clipped or not; the step is
 * taken all the same (the non-finite values propagate as IEEE arithmetic
 * makes them), so a caller that wants to skip such steps clips first and
 * reads zero_grad_norm, or restores a checkpoint when the count moves.
 *  counter  caller-owned device uint64_t, 8-byte aligned, on the context's
 *           device; the library adds to it and never clears it (the caller
 *           zeroes it, e.g. with cudaMemsetAsync, for a fresh count) and it
 *           must stay allocated while counting is on.  NULL stops counting.
 * Errors: ZERO_EINVAL (misaligned, host or other-device counter).
 */
zero_status zero_count_nonfinite(zero_ctx* ctx, uint64_t* counter);

/*
 * zero_read_nonfinite — waits for `stream` and copies the counter given to
 * zero_count_nonfinite into *count.  ZERO_ESTATE when no counter is set;
 * ZERO_ECUDA if the copy fails.
 */
zero_status zero_read_nonfinite(zero_ctx* ctx, uint64_t* count, void* stream);

/*
 * zero_clip_grad_norm — global-norm gradient clipping, the ClipGradNorm
 * transform Femtotron dev logs #4/#5 apply to the fp32 gradient before AdamW
 * (the source guide's --clip-grad 1.0 / gradient_clipping 1.0).  On `stream`
 * it computes the L2 norm of the reduced gradient g = (sum of the N
 * registered replicas) / N over every element of every unit, and the
 * coefficient c = min(1, max_norm / (norm + 1e-6)) rounded to fp32; the next
 * zero_step multiplies every reduced gradient by c before Adam.  Non-finite
 * gradients follow IEEE arithmetic and torch's clip_grad_norm_: an inf makes
 * the norm inf and c = 0 (the inf element becomes inf * 0 = NaN, every other
 * gradient 0); a NaN makes the norm NaN and c = NaN (every gradient NaN).  A
 * caller that skips such steps reads zero_grad_norm before zero_step.  The squared
 * norm is summed over fixed chunks of 16,384 elements of each unit (pads
 * included, they add zero) in a fixed order, so the result is reproducible
 * and identical for every stage and for padded or unpadded layouts.
 *  max_norm    > 0 and finite
 *  workspace   caller-allocated device scratch of at least
 *              zero_clip_workspace_bytes() bytes, 16-byte aligned, owned by the
 *              caller; it holds the norm and coefficient until the next clip
 *              and must stay allocated until that zero_step has completed.
 * Call after every unit's gradients are registered and before zero_step.
 * Errors: ZERO_EINVAL (bad max_norm, null/misaligned/small/host workspace);
 * ZERO_ESTATE (no buffers, gradients missing, step pending post_step);
 * ZERO_ECUDA.
 */
zero_status zero_clip_grad_norm(zero_ctx* ctx, float max_norm, void* workspace, int64_t workspace_bytes,
                                void* stream);

/*
 * Flag of zero_clip_grad_norm_ex / zero_clip_workspace_bytes_ex: keep the
 * reduced fp32 gradient in the workspace so that the next zero_step reads it
 * (4 bytes per element) instead of the N replicas (2N or 4N bytes): the
 * clipped step then moves 2N + 34 instead of 4N + 26 bytes per element (bf16
 * replicas), fewer for N > 4.  Results are bit-identical either way.
 */
#define ZERO_CLIP_KEEP_REDUCED 1

/* Workspace size of zero_clip_grad_norm_ex for `flags`: with
 * ZERO_CLIP_KEEP_REDUCED, plus 4 bytes per padded element (256-byte aligned). */
zero_status zero_clip_workspace_bytes_ex(const zero_ctx* ctx, int32_t flags, int64_t* bytes);

/*
 * zero_clip_grad_norm_ex — zero_clip_grad_norm with flags (0 or
 * ZERO_CLIP_KEEP_REDUCED).  With ZERO_CLIP_KEEP_REDUCED the workspace must
 * hold zero_clip_workspace_bytes_ex(ctx, ZERO_CLIP_KEEP_REDUCED) bytes and
 * stay allocated and unchanged until the next zero_step has completed; the
 * registered replica buffers are not read again by that step.
 * Errors: as zero_clip_grad_norm; ZERO_EINVAL for unknown flags.
 */
zero_status zero_clip_grad_norm_ex(zero_ctx* ctx, float max_norm, int32_t flags, void* workspace,
                                   int64_t workspace_bytes, void* stream);

/*
 * zero_clip_grad_norm_static — zero_clip_grad_norm for callers that cannot
 * allocate device memory (for example code running inside an allocator or
 * an out-of-memory handler, or in a loop where allocation is forbidden), so
 * cannot hand in a workspace.  The pages have no counterpart: this is a
 * property of this library's interface, not of the method.
 * Same computation and result as zero_clip_grad_norm; the scratch is a fixed
 * 1 MiB array in the library's own device memory (one per CUDA context that
 * loads the library's device code — normally one per GPU — held until that
 * context ends), so layouts needing more than that — about 2.1e9 padded
 * elements — are rejected with ZERO_EINVAL.  The call allocates nothing.
 * Its first call in a CUDA context looks up the array's device address in
 * that context (set-up, once per context, keyed on the context's unique id,
 * so a second context on the same GPU or the primary context re-created
 * after cudaDeviceReset gets its own lookup); that first lookup may load the
 * library's device code into the context, which creates the array.  So make
 * the first call in each context before any stream capture and before any
 * region that must not allocate.  All calls in a context share the array
 * and it keeps the last call's contents: calls whose device work can overlap
 * race on it, and between a call and the same zero_ctx's zero_step no other
 * static-scratch clip may run unless all are ordered on one stream.
 * Errors: as zero_clip_grad_norm; ZERO_EINVAL when the layout is too large.
 */
zero_status zero_clip_grad_norm_static(zero_ctx* ctx, float max_norm, void* stream);

/*
 * zero_grad_norm — the norm computed by the last zero_clip_grad_norm on this
 * context, copied to the host.  Synchronizes `stream` (the stream the clip
 * ran on).  ZERO_ESTATE if no clip has run.
 */
zero_status zero_grad_norm(zero_ctx* ctx, double* norm, void* stream);

/*
 * zero_gather_weights — the protocol's gather_weights.  Stage 3 (ZeRO-3
 * unshard, lecture notes §3.3 and §5.1): copy unit `unit`'s N bf16 shards, in
 * rank order, into `unit_buf` (padded_i bf16 elements, device, 2-byte
 * aligned); unit == -1 copies the whole padded buffer.  Stages 0-2: the fused
 * step has already written every replica's full bf16 copy, so this returns
 * ZERO_OK without device work (unit_buf may be NULL).
 * Errors: ZERO_EINVAL (unit out of range, null/misaligned unit_buf at stage 3);
 * ZERO_ESTATE (no buffers bound); ZERO_ECUDA.
 */
zero_status zero_gather_weights(zero_ctx* ctx, int32_t unit, void* unit_buf, void* stream);

/*
 * zero_gather_units — zero_gather_weights for `count` consecutive units
 * first_unit .. first_unit + count - 1 at once: unit first_unit + k into
 * unit_bufs[k] (a host array of `count` device pointers, each padded_i bf16
 * elements, 2-byte aligned; NULL allowed only for empty units).  The
 * ZeRO-3 prefetch of the source guide's DeepSpeed section (the parameter
 * coordinator gathers the next modules' parameters ahead of use, several
 * parameters coalesced into one collective) and Megatron's bucket-by-bucket
 * parameter all-gather: the copies are those of zero_gather_weights, issued
 * as one kernel per 32 units instead of one per unit.  The buffers must not
 * overlap one another or the parameter storage.  count == 0 and stages 0-2:
 * ZERO_OK without device work (unit_bufs may be NULL).
 * Errors: ZERO_EINVAL (count < 0, units out of range, null unit_bufs, null
 * or misaligned buffer of a non-empty unit at stage 3); ZERO_ESTATE (no
 * buffers bound); ZERO_ECUDA.
 */
zero_status zero_gather_units(zero_ctx* ctx, int32_t first_unit, int32_t count, void* const* unit_bufs,
                              void* stream);

/*
 * zero_post_step — the protocol's post_step: forget the registered gradients
 * (and the pending clip coefficient) so the next step needs fresh ones.
 * ZERO_ESTATE unless a step was taken since the last post_step.  No device
 * work.
 */
zero_status zero_post_step(zero_ctx* ctx, void* stream);

/*
 * zero_export_state — checkpoint the optimizer state in a layout-free form
 * (lecture notes §5.2: the pads are not parameters): the real elements of
 * master, m and v, unit by unit with the pads dropped — i.e. the parameters
 * back to back in caller order, numel_total elements per array — into
 * caller-allocated device fp32 buffers (4-byte aligned), and the step count
 * into *t.  Any context planned over the same parameter list, with any N,
 * stage or unit grouping of the same order, can import it (resharding; the
 * source guide's resharding checkpoints, Femtotron #5's dp_size change).
 * Enqueued on `stream` (in an offload context: copies up from the host state,
 * which must not change until they complete).  Errors: ZERO_EINVAL
 * (null/misaligned/host pointer); ZERO_ESTATE (no buffers); ZERO_ECUDA.
 */
zero_status zero_export_state(zero_ctx* ctx, float* master_out, float* exp_avg_out, float* exp_avg_sq_out,
                              int64_t* t, void* stream);

/*
 * zero_import_state — restore state exported by zero_export_state (from this
 * or any other layout of the same parameters): master, m and v are written
 * into this context's padded layout with zero pads, param16 = bf16(master)
 * (round to nearest even), and the step count set to t.  Not allowed while
 * a step awaits its post_step.  Enqueued on `stream`; the inputs may be
 * released once it completes (in an offload context the host state is
 * written and the call synchronizes `stream`).  Errors: ZERO_EINVAL
 * (null/misaligned/host pointer, t < 0); ZERO_ESTATE; ZERO_ECUDA.
 */
zero_status zero_import_state(zero_ctx* ctx, const float* master_in, const float* exp_avg_in,
                              const float* exp_avg_sq_in, int64_t t, void* stream);

/* ---- Capturable steps (CUDA graphs) --------------------------------------
 * The pages have no counterpart: this is the library's way of letting a
 * whole step (registration, clip, step, post_step, gathers) be captured once
 * into a CUDA graph and replayed every iteration without host work.  A
 * replayed launch repeats its arguments, so what changes from step to step
 * (the bias corrections 1 - beta^t) must come from device memory: in
 * capturable mode the step count lives on the device and the kernels look up
 * bc1, bc2 of step t in a table the host computed once (the same fp32 values
 * zero_step would pass, so results are bit-identical).  Each zero_step (and
 * each replay of a captured one) reads the count, updates, and then advances
 * the count with one extra one-thread launch.  Replays also repeat the
 * gradient pointers, the clip workspace and the learning rate captured.
 */

/* Bytes of the capturable workspace for up to max_steps steps in total
 * (16 + 8 * max_steps).  Errors: ZERO_EINVAL. */
zero_status zero_capturable_workspace_bytes(const zero_ctx* ctx, int64_t max_steps, int64_t* bytes);

/*
 * zero_enable_capturable — turn the mode on: workspace = device memory of the
 * context's device (16-byte aligned, caller-owned, kept until
 * zero_disable_capturable), holding the step count (set to the steps taken
 * so far) and the bias corrections of steps 1..max_steps.  Synchronizes
 * `stream`.  A step whose count would pass max_steps is skipped by the
 * kernels (nothing changes; zero_step_count then reports ZERO_ESTATE).
 * Errors: ZERO_EINVAL (workspace, max_steps <= steps taken); ZERO_ESTATE (a
 * step awaits post_step); ZERO_ENOTSUP (offload context); ZERO_ENOMEM;
 * ZERO_ECUDA.  Export and import are refused while the mode is on.
 */
zero_status zero_enable_capturable(zero_ctx* ctx, void* workspace, int64_t workspace_bytes, int64_t max_steps,
                                   void* stream);

/*
 * zero_disable_capturable — turn the mode off: the context's step count
 * becomes the device count (capped at max_steps: later steps were skipped).
 * Synchronizes `stream`.  Errors: ZERO_ESTATE (mode not on); ZERO_ECUDA.
 */
zero_status zero_disable_capturable(zero_ctx* ctx, void* stream);

/* ---- ZeRO-Offload -------------------------------------------------------
 * CMU 15-779 Lecture 13 notes §7.1-7.2 (ZeRO-Offload's partition and its
 * timeline): only the 16-bit parameters stay on the GPU; the fp32 master,
 * m and v live in host memory and a multi-threaded CPU Adam updates them
 * chunk by chunk while the GPU produces the next chunk's gradient, the new
 * bf16 parameters going back up chunk by chunk.  Here the gradient that goes
 * down is the reduced fp32 one (sum of the N replicas in rank order x 1/N,
 * times a pending clip coefficient): the host update is the device step's
 * arithmetic, bit for bit, so an offloaded run equals a GPU-resident one.
 */

/*
 * zero_make_master_offload — zero_make_master for an offload context:
 * bufs->master, exp_avg, exp_avg_sq are HOST memory (pageable or pinned,
 * padded_numel floats each, 16-byte aligned, caller-owned), bufs->param16 is
 * device memory as before; init_params are device fp32 buffers.  The host
 * master gets the init params at their offsets (pads, m, v zero), param16 =
 * bf16(init) on the device.  Synchronizes `stream`.  The context then steps
 * with zero_offload_step only (zero_step returns ZERO_ESTATE); registration,
 * clipping (without ZERO_CLIP_KEEP_REDUCED: ZERO_ENOTSUP), accumulation,
 * gather, export/import and post_step work as for any context.
 * Errors: as zero_make_master, plus ZERO_EINVAL for a device state buffer.
 */
zero_status zero_make_master_offload(const zero_config* cfg, const int64_t* param_numel,
                                     const int32_t* param_unit, int32_t n_params,
                                     const float* const* init_params, const zero_buffers* bufs,
                                     void* stream, zero_ctx** out);

/*
 * zero_offload_workspace_bytes — sizes of the two workspaces of
 * zero_offload_step for chunks of `chunk` elements: *host_bytes of pinned
 * host memory (3 chunk slots of fp32 gradient + bf16 parameters) and
 * *device_bytes of device memory (3 slots of fp32 gradient).
 * Errors: ZERO_EINVAL (NULL, chunk < 1).
 */
zero_status zero_offload_workspace_bytes(const zero_ctx* ctx, int64_t chunk, int64_t* host_bytes,
                                         int64_t* device_bytes);

/*
 * zero_offload_step — one optimizer step of an offload context, t += 1.  The
 * padded buffer is processed in chunks of `chunk` elements through a ring of
 * 3 workspace slots: on `stream` a kernel writes chunk c's reduced (clipped)
 * fp32 gradient into a device slot and it is copied to a pinned host slot;
 * the host waits for it, runs Adam / AdamW over the chunk's host master, m, v
 * on n_threads threads (0: one per hardware thread; the calling thread is one
 * of them), writing bf16 parameters into a host slot that is copied into
 * param16 on `copy_stream` (NULL: `stream`) — so the GPU reduction and the
 * copies of other chunks overlap each chunk's host update.  param16 is
 * rewritten only after the work enqueued on `stream` before the call, and
 * work enqueued on `stream` after it sees the new param16.  Blocks the
 * calling thread until every chunk's host update is done.  Workspaces: see
 * zero_offload_workspace_bytes; host_workspace must be page-locked,
 * device_workspace memory of the context's device, both 16-byte aligned.
 * Not thread-safe on one context.  Errors: ZERO_EINVAL (chunk, threads,
 * workspaces); ZERO_ESTATE (not an offload context, unregistered unit,
 * step pending post_step); ZERO_ENOMEM (threads cannot start); ZERO_ECUDA
 * (the chunks done before the failure stay updated on the host).
 */
zero_status zero_offload_step(zero_ctx* ctx, int64_t chunk, void* host_workspace, int64_t host_bytes,
                              void* device_workspace, int64_t device_bytes, int32_t n_threads,
                              void* stream, void* copy_stream);

/*
 * zero_cpu_adam — the CPU Adam of the offload step on its own, over host
 * arrays of n elements: given the reduced fp32 gradient `grad`, updates
 * master, exp_avg, exp_avg_sq in place with step t (>= 1) of cfg's
 * optimizer and writes param16 = bf16(master) (bit patterns, round to
 * nearest even).  Same arithmetic as the device step.  n_threads as above;
 * the threads belong to one process-wide pool kept between calls (calls from
 * several threads take turns).  No CUDA call is made.
 * Errors: ZERO_EINVAL (config, t < 1, n < 0, NULL or misaligned pointer);
 * ZERO_ENOMEM.
 */
zero_status zero_cpu_adam(const zero_config* cfg, int64_t t, const float* grad, float* master,
                          float* exp_avg, float* exp_avg_sq, uint16_t* param16, int64_t n,
                          int32_t n_threads);

/*
 * zero_kernel_timeouts — how many bounded waits of the tile-staged step
 * kernels (used for N = 1..4 or N >= 11 bf16 and N >= 7 fp32 replicas when a
 * launch covers at least 2^23 elements) gave up on the current device since
 * the library was loaded.  A wait gives up only if a
 * bulk copy never lands; the CTA then leaves the rest of its tiles unchanged,
 * so a non-zero count means some step is incomplete.  Reads a device counter:
 * synchronizes with the device.  ctx may be NULL.
 */
zero_status zero_kernel_timeouts(const zero_ctx* ctx, uint32_t* count);

/*
 * zero_debug_inject — test hook for the bounded waits above (the pages have
 * no counterpart).  what = ZERO_INJECT_MISSING_COPY arms it for the next
 * zero_step: if that step's first launch uses a tile-staged kernel, the
 * kernel announces the bytes of the launch's first tile to its mbarrier but
 * issues no copy for it, so that one wait runs out after about a second;
 * the CTA then counts a timeout (zero_kernel_timeouts), waits for the copies
 * it did issue and leaves, and the elements of its tiles stay un-updated.
 * Nothing faults: the device stays usable.  what = 0 disarms.  The hook is
 * consumed by the next vector launch whichever kernel it uses.
 * Errors: ZERO_EINVAL (NULL ctx, unknown value).
 */
#define ZERO_INJECT_MISSING_COPY 1
/*
 * what = ZERO_INJECT_SHORT_BOUNDS: the next zero_step tells its kernels that
 * the state arrays end 8 elements before they really do (the buffers keep
 * their full size, so no access can leave them).  In a debug build the index
 * checks then refuse the last 8 elements (counted, not updated); in a release
 * build the checks do not exist and the step is the normal one.
 */
#define ZERO_INJECT_SHORT_BOUNDS 2
zero_status zero_debug_inject(zero_ctx* ctx, int32_t what);

/*
 * zero_debug_check_failures — in a debug build of the library (compiled with
 * -DZFS_DEBUG_CHECKS: every kernel index is checked before the access it
 * guards; a failed check is counted and the access skipped, never trapped),
 * the number of failed checks on the current device since the library was
 * loaded.  Synchronizes with the device.  The pages have no counterpart.
 * Errors: ZERO_EINVAL (NULL); ZERO_ENOTSUP in a release build (*count = 0);
 * ZERO_ECUDA.
 */
zero_status zero_debug_check_failures(uint32_t* count);

/* Number of steps taken (t).  In capturable mode it is read from the device
 * (synchronizing), and ZERO_ESTATE reports steps skipped past max_steps. */
zero_status zero_step_count(const zero_ctx* ctx, int64_t* t);

/*
 * Number of kernels the last zero_step / zero_gather_weights / zero_gather_units call on this
 * context enqueued (0 when it had nothing to do).  Host bookkeeping only.
 */
zero_status zero_last_launches(const zero_ctx* ctx, int32_t* launches);

/* Set the learning rate used by later steps (a scheduler's lr update).  A
 * step already captured into a CUDA graph keeps the lr (and the AdamW factor
 * 1 - lr*wd) it was captured with: capture it again after a change. */
zero_status zero_set_lr(zero_ctx* ctx, float lr);

/* Release the context's host metadata.  Device buffers stay the caller's. */
zero_status zero_destroy(zero_ctx* ctx);

/*
 * Text of the last error on `ctx`; with ctx == NULL, the last error of a
 * failed zero_plan / zero_make_master on the calling thread.  The string is
 * owned by the library and valid until the next call on the same context
 * (or thread).
 */
const char* zero_last_error(const zero_ctx* ctx);

/* Constant name of a status code. */
const char* zero_status_string(zero_status status);

#ifdef __cplusplus
}
#endif

#endif /* ZERO_FLATSTEP_H */
