/*
 * zeroshard: the data-parallel hot path of ZeRO mixed-precision training on
 * one GB300 (sm_103a) -- the optimizer step of the parameter shard this GPU
 * owns.
 *
 * What the step computes (DeepSpeed Complete Guide, youngju.dev):
 *  - §2 memory table: fp16 (or bf16) parameters and gradients, fp32 master
 *    parameters, fp32 Adam momentum and variance (2+2+4+4+4 = 16 bytes per
 *    parameter).
 *  - §2.1 ZeRO-1: master/momentum/variance are split into N shards; each rank
 *    updates only its own shard and an all-gather rebuilds the parameters.
 *  - §2.2 ZeRO-2: gradients are split too; reduce-scatter hands each rank the
 *    sum of all ranks' gradients over its shard, which it accumulates;
 *    gradients travel in buckets of reduce_bucket_size elements.
 *  - §2.3 ZeRO-3: parameters are split as well (16 bytes / N per parameter).
 *  - §4.2 fp16 settings: dynamic loss scale starting at 2^initial_scale_power,
 *    raised after loss_scale_window clean steps, lowered after `hysteresis`
 *    overflows, never below min_loss_scale; bf16 needs no loss scaling.
 *  - §4.3: the global batch is micro batch x accumulation steps x world size,
 *    so the applied gradient is the mean over ranks and micro-steps.
 *  - §4.1: the optimizer is AdamW with eps 1e-8.
 *
 * The N data-parallel ranks are simulated on one GPU: the caller holds, in
 * this GPU's HBM, each rank's slice of the owned shard (what a reduce-scatter
 * would sum).  The library sums them in fp32 in rank order 0..N-1 onto an
 * fp32 accumulator (micro-step by micro-step), flags any +-inf/NaN before any
 * state is written, and on a clean step applies bias-corrected AdamW with
 * decoupled weight decay to the fp32 master/m/v and writes the half copy
 * (round to nearest even) that an all-gather would consume.  On overflow the
 * step leaves all state untouched and the loss scale is lowered.
 *
 * With real ranks (one process per GPU), a rank that receives the other ranks'
 * slices of its shard (e.g. an all-to-all of each gradient bucket's shard
 * parts) passes the received slices as the n pointers of zs_reduce_check, so
 * the same rank-ordered fp32 sum runs; the flag (and the clipping norm) is
 * all-reduced between the reduce and zs_apply, and the half shards are
 * all-gathered afterwards.  Unclipped steps can instead pass the last
 * micro-step's received slices to zs_update_oop bucket by bucket (sum, flag
 * and update into a second state set in one pass), all-reduce the flag and
 * commit.  The Python package's dp module does this with torch.distributed.
 *
 * Conventions for every call:
 *  - Ownership: every array is caller-owned DEVICE memory on the context's
 *    device; `grads` is a HOST array of n device pointers, read during the
 *    call only.  A context owns only a few device words and a pinned host
 *    mirror.  Arrays must not overlap.
 *  - Layout: contiguous 1-D arrays of `count` elements; half arrays hold
 *    IEEE binary16 (ZS_FP16) or bfloat16 (ZS_BF16) bit patterns.
 *  - Alignment: every device pointer must be 16-byte aligned (ZS_ERR_ALIGN);
 *    count may be any value >= 0 (a ragged tail is handled).
 *  - Limits: 1 <= n <= ZS_MAX_RANKS.
 *  - Ordering: all work is issued on `stream` in order; only zs_shard_step,
 *    zs_shard_step_clipped, zs_shard_step_halfacc, zs_shard_step_oop,
 *    zs_scaler_update and zs_ctx_timing synchronise that stream
 *    (zs_shard_step_async and zs_shard_step_async_oop never do).  The steps of
 *    one context share its flag, scratch and the fused step's barrier: issue
 *    them in stream order (one stream, or streams ordered by events); steps
 *    that must overlap use a context each.
 *  - Errors: a non-zero zs_status; zs_last_error(ctx) gives the message.
 *    Overflow of the gradients is a result, not an error.
 *  - Threads: a context is used by one host thread at a time.
 */
#ifndef ZEROSHARD_H
#define ZEROSHARD_H

#include <stdint.h>
#include <cuda_runtime.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ZS_MAX_RANKS 256
#define ZS_DEFAULT_ALIGN 64

typedef enum {
  ZS_OK = 0,
  ZS_ERR_ARG = -1,     /* a null pointer, a negative size, n out of range */
  ZS_ERR_ALIGN = -2,   /* a device pointer not 16-byte aligned */
  ZS_ERR_DTYPE = -3,   /* dtype is neither ZS_FP16 nor ZS_BF16 */
  ZS_ERR_CUDA = -4,    /* a CUDA runtime error (message in zs_last_error) */
  ZS_ERR_TIMEOUT = -5, /* a bounded device wait gave up (the fused step's barrier) */
  ZS_ERR_LIMIT = -6    /* count beyond ZS_NOALLOC_MAX_COUNT (zs_grad_sumsq_noalloc) */
} zs_status;

typedef enum { ZS_FP16 = 0, ZS_BF16 = 1 } zs_dtype;

/* Shard layout of a flat parameter buffer (§2.1-§2.3). */
typedef struct {
  int64_t psi;        /* number of parameters */
  int64_t psi_pad;    /* psi rounded up to a multiple of n * align */
  int64_t shard_len;  /* psi_pad / n: elements each rank owns, padding included */
  int32_t n;          /* data-parallel ranks */
  int32_t align;      /* alignment unit in elements */
} zs_partition;

/* AdamW hyper-parameters (§4.1), as fp32. */
typedef struct {
  float lr, beta1, beta2, eps, weight_decay;
} zs_adam_hparams;

/* Loss-scale state (§4.2), caller-owned, host memory.  dynamic = 0 keeps the
 * scale fixed (bf16, or a static loss_scale); overflow still skips the step. */
typedef struct {
  float scale;          /* current loss scale S */
  float min_scale;      /* min_loss_scale */
  int32_t window;       /* loss_scale_window: clean steps before S doubles */
  int32_t clean_count;  /* consecutive clean steps since the last overflow or increase */
  int32_t hysteresis;   /* overflows before S halves */
  int32_t hyst_left;    /* overflows still tolerated before the next halving */
  int32_t dynamic;      /* 1: dynamic scaling, 0: static */
  int32_t consecutive_hysteresis; /* 1: a clean step restores hyst_left, so only
                                     consecutive overflows lower the scale */
} zs_scaler;

typedef struct zs_ctx zs_ctx;

/* ---------------------------------------------------------------- host-only */

/* Partition psi parameters over n ranks (§2.1-§2.3): psi_pad = psi rounded up
 * to a multiple of n*align_elems, shard_len = psi_pad/n; rank r owns flat
 * indices [r*shard_len, (r+1)*shard_len), of which those >= psi are padding.
 * psi >= 0, 1 <= n <= ZS_MAX_RANKS, align_elems >= 1 (ZS_DEFAULT_ALIGN = 64
 * keeps every shard 16-byte aligned for both fp32 and half arrays). */
zs_status zs_init_partition(int64_t psi, int32_t n, int32_t align_elems, zs_partition* out);

/* Rank `rank`'s range: begin = rank*shard_len, padded_end = begin+shard_len,
 * valid_end = max(begin, min(padded_end, psi)). */
zs_status zs_shard_range(const zs_partition* p, int32_t rank, int64_t* begin, int64_t* valid_end,
                         int64_t* padded_end);

/* Per-rank model-state bytes for ZeRO stage 0..3 (§2 table, §2.1-§2.3), with
 * E = shard_len: 16*psi, 4*psi + 12*E, 2*psi + 14*E, 16*E. */
zs_status zs_model_state_bytes(const zs_partition* p, int32_t stage, uint64_t* bytes);

/* Fill a scaler: hyst_left = hysteresis, clean_count = 0,
 * consecutive_hysteresis = 0 (set the field to 1 for the §4.2 knob of that
 * name).  §4.2 defaults are scale 2^16, window 1000, hysteresis 2, min_scale 1. */
zs_status zs_scaler_init(zs_scaler* s, float scale, float min_scale, int32_t window,
                         int32_t hysteresis, int32_t dynamic);

/* ---------------------------------------------------------------- context */

/* Create a context on the current CUDA device.  It owns: the step's overflow
 * flag (a device int32, zero at creation), a result word in mapped pinned
 * host memory (the update kernel writes the step's flag and new scale there;
 * the synchronising calls read it after the stream sync, with no copy), 8 MB
 * of scratch for the clipping norm's per-CTA partial sums (sized here, so no
 * later call allocates device memory), a pinned mirror of the norm, and the
 * fused step's grid barrier (16 device bytes) with its timeout word (mapped
 * pinned).  Environment: ZEROSHARD_PDL=0 launches the step's kernels without
 * programmatic dependent launch; ZEROSHARD_FUSED=0 starts the context with
 * the fused step off (zs_ctx_set_fused).
 * *ctx is set to NULL on failure. */
zs_status zs_ctx_create(zs_ctx** ctx);
zs_status zs_ctx_destroy(zs_ctx* ctx);

/* The fused step (§2.2, §4.2: the step's overflow resolved before any state
 * is written, here by a grid barrier inside one kernel).
 * zs_shard_step, zs_shard_step_async, zs_shard_step_oop,
 * zs_shard_step_async_oop, zs_shard_step_clipped,
 * zs_shard_step_async_clipped and the four zs_shard_step_halfacc forms (the
 * sums rounded to the accumulator's format first) run the whole last call of
 * a step as ONE
 * cooperative kernel when one thread per 8 owned elements fits a grid whose
 * CTAs are all resident at once (zs_ctx_fused_capacity: about 0.93M elements
 * on GB300): each thread loads its elements' last micro-step sums (acc + the
 * n slices, in the order zs_grad_accum adds them) and their state into
 * registers, each CTA arrives at one grid barrier counting whether its sums
 * hold a non-finite value (clipped: after writing its total of squares); the
 * last CTA to arrive forms the step's flag from that count and the earlier
 * micro-steps' flag (and, clipped, folds the totals in the order of the norm
 * pass), clears the flag and releases the grid, and a clean step applies the
 * same AdamW arithmetic
 * from the registers; an overflow writes no state.  Results (norm included)
 * are bit for bit those of the multi-kernel path.  The barrier
 * relies on every CTA of the grid being resident at once, which the
 * cooperative launch provides; its wait is bounded for the cases it may not
 * (e.g. fused steps of several contexts running at the same time): a CTA that
 * waits longer than wait_ns gives up and writes nothing, and the context's
 * next call (the synchronising forms: the call itself) returns
 * ZS_ERR_TIMEOUT after resetting the barrier and the flag; the state of that
 * step is then undefined.  Run fused steps of different contexts in order,
 * or turn the fused step off where they must overlap.
 * mode: ZS_FUSED_OFF (always the multi-kernel path), ZS_FUSED_ON (default),
 * ZS_FUSED_TEST_TIMEOUT (as ON, but the barrier waits for one CTA more than
 * the grid has, so every fused step's wait runs out: for testing the timeout
 * path).  wait_ns <= 0 keeps the default of one second.  A device without
 * cooperative launches starts with the fused step off, and turning it on
 * there returns ZS_ERR_ARG. */
#define ZS_FUSED_OFF 0
#define ZS_FUSED_ON 1
#define ZS_FUSED_TEST_TIMEOUT 2
zs_status zs_ctx_set_fused(zs_ctx* ctx, int32_t mode, int64_t wait_ns);
/* The largest count the fused step takes on this context's device (any
 * dtype, accumulator or form); larger shards take the multi-kernel path. */
zs_status zs_ctx_fused_capacity(zs_ctx* ctx, int64_t* elements);
/* Message of the last failed call on ctx ("" if none).  Valid until the next call. */
const char* zs_last_error(const zs_ctx* ctx);
/* Device address of the context's step overflow flag: zs_grad_accum ORs into
 * it and zs_shard_step consumes and clears it.  A multi-GPU caller can
 * all-reduce (MAX) this int32 in place before the last call of the step. */
zs_status zs_ctx_overflow_flag(zs_ctx* ctx, int32_t** d_flag);

/* ---------------------------------------------------------------- the step */

/* Micro-steps 1..G-1 of a step (§2.2, §4.3): for i in [0, count)
 *   acc[i] = (first ? +0.0f : acc[i]) + grads[0][i] + ... + grads[n-1][i]
 * in fp32, in that order, and OR into the context's step flag whether any
 * result is +-inf/NaN (a non-finite input always yields one).  Call it once
 * per micro-step (first = 1 for the step's first) and, if the shard is split
 * into buckets, once per bucket with sub-range pointers; results do not depend
 * on the bucketing. */
zs_status zs_grad_accum(zs_ctx* ctx, const void* const* grads, int32_t n, zs_dtype dt,
                        int64_t count, float* acc, int32_t first, cudaStream_t stream);

/* Two-phase form for a flag that spans several shards, buckets or GPUs.
 * Phase 1: as zs_grad_accum, ORing into the caller's device int32 *d_flag.
 * With acc == NULL it only checks (reads the slices, writes nothing else). */
zs_status zs_reduce_check(zs_ctx* ctx, const void* const* grads, int32_t n, zs_dtype dt,
                          int64_t count, float* acc, int32_t first, int32_t* d_flag,
                          cudaStream_t stream);

/* Phase 1 for the last micro-step when the update re-reads it (zs_apply with
 * grads, which sums acc + the slices again): OR into *d_flag whether any
 *   (acc ? acc[i] : +0.0f) + grads[0][i] + ... + grads[n-1][i]
 * is +-inf/NaN, writing nothing else.  acc is NULL for a one-micro-step step.
 * For fp16 the slices' bit patterns decide (finite halves cannot carry a finite
 * acc past the fp32 maximum), 2n bytes read per element; bf16 on top of acc
 * reads acc too.  With zs_reduce_check for micro-steps 1..G-1 and zs_apply for
 * the update, this is zs_shard_step's re-read form split at the flag, for a
 * caller that exchanges the flag (all ranks skip together, §4.2) before the
 * update; it avoids writing and re-reading acc for the last micro-step
 * (8 bytes per element) when n is small.  Same errors as zs_reduce_check. */
zs_status zs_check_last(zs_ctx* ctx, const void* const* grads, int32_t n, zs_dtype dt,
                        int64_t count, const float* acc, int32_t* d_flag, cudaStream_t stream);

/* Phase 2: if *d_flag != 0 nothing is written.  Otherwise, per element,
 *   s = acc[i] (or +0 if acc == NULL), then s += grads[r][i] for r = 0..n-1
 *       when grads != NULL (the last micro-step, re-read instead of stored),
 *   g = s / grad_div               (grad_div = N * G * S: mean and unscale)
 *   m = beta1*m + (1-beta1)*g ;  v = beta2*v + (1-beta2)*g*g
 *   p = p - lr * ( (m/(1-beta1^step)) / (sqrt(v/(1-beta2^step)) + eps) + wd*p )
 *   half_out[i] = round_to_nearest_even(p)
 * step is Adam's 1-based count of applied updates, this one included. */
zs_status zs_apply(zs_ctx* ctx, const int32_t* d_flag, const void* const* grads, int32_t n,
                   zs_dtype dt, const float* acc, int64_t count, float grad_div, float* master,
                   float* m, float* v, void* half_out, const zs_adam_hparams* hp, int64_t step,
                   cudaStream_t stream);

/* Loss-scale update after phase 2 (§4.2), run on the device from *d_flag:
 * overflow -> clean_count = 0 and, if dynamic, hyst_left -= 1 and at 0
 * scale = max(scale/2, min_scale), hyst_left = hysteresis;
 * clean -> if dynamic, clean_count += 1 and at window scale *= 2,
 * clean_count = 0; with consecutive_hysteresis also hyst_left = hysteresis.  Writes *scaler and *overflow_out (may be NULL) and
 * synchronises `stream`.  Does not clear *d_flag. */
zs_status zs_scaler_update(zs_ctx* ctx, const int32_t* d_flag, zs_scaler* scaler,
                           int32_t* overflow_out, cudaStream_t stream);

/* The whole last call of a step for one owned shard (§2.1, §2.2, §4.2):
 * grads are the n slices of the step's LAST micro-step; micro-steps
 * 1..accum_steps-1 must already be in acc via zs_grad_accum.  It resolves the
 * step's overflow (the context flag, OR this call's slices) before writing any
 * state, applies AdamW with grad_div = n * accum_steps * scaler->scale,
 * updates *scaler, writes *overflow_out and *new_scale_out (either may be
 * NULL), clears the context flag and synchronises `stream`.
 * acc may be NULL only when accum_steps == 1.  A shard that fits the fused
 * step (zs_ctx_set_fused) takes it: one kernel, the sums held in registers
 * across a grid barrier, acc read (accum_steps > 1) and never written.
 * Otherwise, when n < 4 (or acc is NULL) the last slices are checked, then
 * re-read by the update (2n bytes per element) instead of summed into acc and
 * read back (8 bytes per element).  Either way acc holds no defined sums
 * afterwards.  The caller advances `step` only if *overflow_out == 0. */
zs_status zs_shard_step(zs_ctx* ctx, const void* const* grads, int32_t n, zs_dtype dt,
                        int64_t count, float* acc, int32_t accum_steps, float* master, float* m,
                        float* v, void* half_out, const zs_adam_hparams* hp, int64_t step,
                        zs_scaler* scaler, int32_t* overflow_out, float* new_scale_out,
                        cudaStream_t stream);

/* ---------------------------------------------------------------- half accumulator */

/* Variant whose accumulator is kept in the gradient's own 2-byte format, as
 * the pages count gradients (2 bytes per parameter, §2 table; 2Ψ/N per rank
 * under ZeRO-2, §2.2).  Per micro-step and element the ranks are summed in
 * fp32 on top of the widened accumulator (same order as zs_grad_accum) and the
 * sum is rounded to nearest even into acc_half; a sum past the half maximum
 * rounds to infinity and makes the step overflow.  It moves 4 fewer bytes per
 * element per carried micro-step than the fp32 accumulator, at the cost of one
 * rounding per micro-step.  acc_half: count halves, 16-byte aligned. */
zs_status zs_grad_accum_halfacc(zs_ctx* ctx, const void* const* grads, int32_t n, zs_dtype dt,
                                int64_t count, void* acc_half, int32_t first,
                                cudaStream_t stream);
/* The last call of a step with the half accumulator; otherwise as
 * zs_shard_step.  The multi-kernel path sums the last micro-step into acc_half
 * (rounded) and updates from it; a shard that fits the fused step rounds the
 * same sums in registers and leaves acc_half unwritten.  Either way acc_half
 * holds no defined sums after the call. */
zs_status zs_shard_step_halfacc(zs_ctx* ctx, const void* const* grads, int32_t n, zs_dtype dt,
                                int64_t count, void* acc_half, int32_t accum_steps,
                                float* master, float* m, float* v, void* half_out,
                                const zs_adam_hparams* hp, int64_t step, zs_scaler* scaler,
                                int32_t* overflow_out, float* new_scale_out,
                                cudaStream_t stream);

/* The half-accumulator step with the state written out of place, as
 * zs_shard_step_oop is to zs_shard_step: the last micro-step's sums (acc_half
 * widened + the n slices, rounded to the 2-byte format as every micro-step's
 * are), the overflow check (on the rounded sums) and the AdamW update in one
 * pass from master_in/m_in/v_in into master_out/m_out/v_out and half_out (the
 * last micro-step's sums are never written to acc_half); *overflow_out == 0 means the
 * *_out buffers hold the state.  acc_half may be NULL when accum_steps ==
 * 1.  Synchronises `stream`. */
zs_status zs_shard_step_halfacc_oop(zs_ctx* ctx, const void* const* grads, int32_t n,
                                    zs_dtype dt, int64_t count, const void* acc_half,
                                    int32_t accum_steps, const float* master_in,
                                    const float* m_in, const float* v_in, float* master_out,
                                    float* m_out, float* v_out, void* half_out,
                                    const zs_adam_hparams* hp, int64_t step, zs_scaler* scaler,
                                    int32_t* overflow_out, float* new_scale_out,
                                    cudaStream_t stream);

/* ---------------------------------------------------------------- clipping */

/* Global-norm gradient clipping (§4.1 gradient_clipping; §5.1: engine.step()
 * includes gradient clipping).  The pages give the knob, not the formula; the
 * usual one is used: norm = L2 norm of the averaged, unscaled gradient of the
 * whole model; coef = max_norm / (norm + 1e-6) if that is below 1, else 1;
 * the update uses g * coef.
 *
 * Phase 1b (after the flag phase, before phase 2): *d_sumsq (device fp64) =
 *   sum over i in [0, count) of ((acc[i] or +0) + grads[0][i] + ... +
 *   grads[n-1][i])^2 / grad_div^2,
 * with grads == NULL when the sums are already in acc.  Deterministic (fixed
 * summation order for a given count and device).  A caller holding several
 * shards, buckets or GPUs adds their values (an all-reduce) before phase 2.
 * Uses the context's scratch (per-CTA partial sums). */
zs_status zs_grad_sumsq(zs_ctx* ctx, const void* const* grads, int32_t n, zs_dtype dt,
                        const float* acc, int64_t count, float grad_div, double* d_sumsq,
                        cudaStream_t stream);

/* Phase 2 with clipping: zs_apply with g multiplied by the coefficient
 * computed on the device from *d_sumsq and max_norm (max_norm <= 0: no
 * clipping). */
zs_status zs_apply_clipped(zs_ctx* ctx, const int32_t* d_flag, const double* d_sumsq,
                           float max_norm, const void* const* grads, int32_t n, zs_dtype dt,
                           const float* acc, int64_t count, float grad_div, float* master,
                           float* m, float* v, void* half_out, const zs_adam_hparams* hp,
                           int64_t step, cudaStream_t stream);

/* zs_shard_step with global-norm clipping, where the owned shard holds the
 * whole gradient whose norm is clipped (one rank; or a caller that clips per
 * shard).  *grad_norm_out (may be NULL) gets the norm, 0 on a skipped step.
 * The norm is computed inside the last micro-step's pass (the one that sums
 * into acc, or the flag pass of the re-read path, which then also reads acc),
 * so clipping adds no pass over the shard; its per-CTA partial sums live in
 * the context's fixed scratch (beyond 2^31 elements the pass's grid is capped
 * at that scratch and each thread takes several vectors). */
zs_status zs_shard_step_clipped(zs_ctx* ctx, const void* const* grads, int32_t n, zs_dtype dt,
                                int64_t count, float* acc, int32_t accum_steps, float* master,
                                float* m, float* v, void* half_out, const zs_adam_hparams* hp,
                                int64_t step, zs_scaler* scaler, float max_norm,
                                int32_t* overflow_out, float* new_scale_out,
                                float* grad_norm_out, cudaStream_t stream);

/* Allocation-free form of zs_grad_sumsq.  The pages have no counterpart: this
 * exists for callers that cannot call cudaMalloc -- code that must not grow
 * device memory (a framework that owns all of it through its own planner or
 * arena, an out-of-memory handler that still wants the gradient norm) and
 * code that cannot create a zs_ctx, whose creation allocates.
 *
 * Same result and arguments as zs_grad_sumsq, without a context.  Its scratch
 * (one fp64 partial sum per 16,384 elements) is a fixed static device array
 * of ZS_NOALLOC_MAX_PARTS doubles (128 KB) that every GPU loading this library
 * holds until exit, so count is limited to ZS_NOALLOC_MAX_COUNT elements;
 * larger counts return ZS_ERR_LIMIT before any work.  The call allocates
 * nothing: no cudaMalloc, cudaFree or allocating library routine.
 * Set-up: the first call on a device, with that device current, looks up the
 * array's device address (cudaGetSymbolAddress) and loads every kernel this
 * entry point launches (under lazy module loading, the CUDA default, loading
 * a kernel or a module takes device memory).  Make that first call at
 * start-up -- a call with count = 0 is enough -- before memory can run short
 * and before any stream capture.  A device reset (cudaDeviceReset) ends the
 * context the address belongs to; the first call in the new context repeats
 * the set-up, so the same start-up rule applies after a reset.
 * Every call on a device shares the one array and leaves its partial sums in
 * it; each call overwrites the slots it reads, so nothing has to start at
 * zero, but calls whose kernels overlap on the GPU (different streams, no
 * ordering) race on it -- serialise them.
 * Errors: ZS_ERR_ARG / ZS_ERR_ALIGN / ZS_ERR_DTYPE as for zs_grad_sumsq,
 * ZS_ERR_LIMIT for count > ZS_NOALLOC_MAX_COUNT, ZS_ERR_CUDA for a runtime
 * failure (no message: there is no context), including an error already
 * pending from earlier work, which is left pending for the caller. */
#define ZS_NOALLOC_MAX_PARTS 16384
#define ZS_NOALLOC_ELEMS_PER_PART 16384
#define ZS_NOALLOC_MAX_COUNT ((int64_t)ZS_NOALLOC_MAX_PARTS * ZS_NOALLOC_ELEMS_PER_PART)
zs_status zs_grad_sumsq_noalloc(const void* const* grads, int32_t n, zs_dtype dt,
                                const float* acc, int64_t count, float grad_div,
                                double* d_sumsq, cudaStream_t stream);

/* ---------------------------------------------------------------- capture-friendly step */

/* Learning-rate schedules named in §4.4 (LRRangeTest, OneCycle and
 * WarmupCosineLR are named there too but not built).  The pages give
 * WarmupDecayLR's knobs (warmup_min_lr, warmup_max_lr, warmup_num_steps,
 * total_num_steps, warmup_type "linear"); the formulas are the plain linear
 * reading, at Adam's step t (1-based count of applied updates):
 *   ZS_LR_CONSTANT:      max_lr
 *   ZS_LR_WARMUP:        min_lr + (max_lr - min_lr) * min(1, t / warmup_steps)
 *   ZS_LR_WARMUP_DECAY:  the warmup for t <= warmup_steps, then
 *                        max_lr * max(0, (total_steps - t) / (total_steps - warmup_steps)) */
typedef enum { ZS_LR_CONSTANT = 0, ZS_LR_WARMUP = 1, ZS_LR_WARMUP_DECAY = 2 } zs_lr_kind;
typedef struct {
  int32_t kind;          /* zs_lr_kind */
  int32_t pad_;
  int64_t warmup_steps;  /* warmup_num_steps */
  int64_t total_steps;   /* total_num_steps */
  float min_lr, max_lr;  /* warmup_min_lr, warmup_max_lr */
} zs_lr_schedule;

/* Step state kept in DEVICE memory (caller-owned, 8-byte aligned, 64 bytes):
 * the loss scaler, Adam's step count and the last step's outcome.  The caller
 * initialises it (e.g. by copying a host struct whose scaler came from
 * zs_scaler_init, with step = iterations = 0) and may read it back at any time. */
typedef struct {
  zs_scaler scaler;    /* loss-scale state (§4.2) */
  int32_t overflow;    /* 1 if the last step was skipped */
  int32_t buf;         /* out-of-place step: which of the two state buffers holds the
                          current state (flipped by every applied step); 0 otherwise */
  int64_t step;        /* applied updates so far */
  int64_t iterations;  /* steps run so far, skipped ones included */
  float lr;            /* learning rate of the last applied update */
  float grad_div;      /* N * G * S of the last step */
} zs_device_state;

/* zs_shard_step without any host round trip: the scale, Adam's step count and
 * the learning rate are read from and written to *d_state on the device, the
 * learning rate follows *sched (NULL: hp->lr throughout), nothing is copied
 * to the host and the stream is not synchronised.  A whole step -- the
 * zs_grad_accum calls plus this one -- can therefore be captured once in a
 * CUDA graph and replayed every step (make one uncaptured call first so the
 * launch shapes are cached).  Per-kernel timing (zs_ctx_set_timing) is
 * recorded only when `stream` is not capturing.
 * Otherwise identical to zs_shard_step (same kernels, same arithmetic). */
zs_status zs_shard_step_async(zs_ctx* ctx, const void* const* grads, int32_t n, zs_dtype dt,
                              int64_t count, float* acc, int32_t accum_steps, float* master,
                              float* m, float* v, void* half_out, const zs_adam_hparams* hp,
                              const zs_lr_schedule* sched, zs_device_state* d_state,
                              cudaStream_t stream);

/* zs_shard_step_async with global-norm clipping (§4.1 gradient_clipping; §5.1:
 * engine.step() includes gradient clipping), as zs_shard_step_clipped computes
 * it: norm = L2 norm of the averaged, unscaled gradient of the owned shard,
 * coef = max_norm / (norm + 1e-6) when below 1.  The sum of squares is formed
 * inside the last micro-step's pass, unscaled, and divided by N * G * S on the
 * device (the scale lives in *d_state).  d_grad_norm (device fp64, 8-byte
 * aligned, may be NULL) receives the step's norm; on a step that overflows it
 * is not finite and the step is skipped as in zs_shard_step_async.
 * max_norm <= 0 disables clipping (the call is then zs_shard_step_async).
 * Capturable in a CUDA graph like zs_shard_step_async. */
zs_status zs_shard_step_async_clipped(zs_ctx* ctx, const void* const* grads, int32_t n,
                                      zs_dtype dt, int64_t count, float* acc,
                                      int32_t accum_steps, float* master, float* m, float* v,
                                      void* half_out, const zs_adam_hparams* hp,
                                      const zs_lr_schedule* sched, float max_norm,
                                      zs_device_state* d_state, double* d_grad_norm,
                                      cudaStream_t stream);

/* ---------------------------------------------------------------- out-of-place step */

/* The step with the optimizer state written out of place (§2.1, §2.2, §4.2):
 * the last micro-step's sums (acc + the n slices, as zs_shard_step adds them),
 * the overflow check and the AdamW update run as ONE pass that reads the
 * current master/m/v and writes the new values into a second set of buffers;
 * after that pass the step's flag is complete, and only a clean step makes
 * the written set current -- an overflowing step leaves the current set
 * untouched and its written set is garbage (the fused step, for shards that
 * fit it, writes nothing on an overflow), so the skip semantics are those of
 * zs_shard_step.  Nothing is written twice: per element the step moves
 * exactly the algorithmic bytes (2*n*G + 8*(G-1) + 26), against + 8 (the
 * accumulator written and read back) or + 2*n (the last slices read twice) for
 * zs_shard_step, at the cost of a second master/m/v/half set (14 bytes per
 * element of the owned shard).  No clipping (its norm is needed before the
 * update).  Micro-steps 1..G-1 go through zs_grad_accum as usual.
 *
 * zs_shard_step_oop: reads master_in/m_in/v_in, writes master_out/m_out/v_out
 * and half_out; updates *scaler; *overflow_out == 0 means the *_out buffers
 * (and half_out) now hold the state and the caller swaps its pointers;
 * synchronises `stream`.  acc may be NULL when accum_steps == 1.  The six
 * state arrays (and half_out) must not overlap. */
zs_status zs_shard_step_oop(zs_ctx* ctx, const void* const* grads, int32_t n, zs_dtype dt,
                            int64_t count, const float* acc, int32_t accum_steps,
                            const float* master_in, const float* m_in, const float* v_in,
                            float* master_out, float* m_out, float* v_out, void* half_out,
                            const zs_adam_hparams* hp, int64_t step, zs_scaler* scaler,
                            int32_t* overflow_out, float* new_scale_out, cudaStream_t stream);

/* The device-resident form (as zs_shard_step_async: no host round trip,
 * capturable): master, m, v and half are HOST arrays of two device pointers
 * each; d_state->buf says which set is current (0 or 1, initialise it to 0 with
 * the state in set 0); a clean step writes set buf ^ 1 and flips d_state->buf,
 * an overflowing one leaves it. */
zs_status zs_shard_step_async_oop(zs_ctx* ctx, const void* const* grads, int32_t n, zs_dtype dt,
                                  int64_t count, const float* acc, int32_t accum_steps,
                                  float* const* master, float* const* m, float* const* v,
                                  void* const* half, const zs_adam_hparams* hp,
                                  const zs_lr_schedule* sched, zs_device_state* d_state,
                                  cudaStream_t stream);

/* Two-phase form of the out-of-place step, for a flag that spans several
 * buckets, shards or GPUs (§2.2: each rank updates its shard as the reduced
 * buckets arrive; §4.2: all ranks skip together).  For one range of the
 * shard: s = acc[i] (or +0 if acc == NULL) + grads[0][i] + ... in rank order,
 * as zs_grad_accum adds them; OR into *d_flag whether any s is non-finite;
 * then AdamW with g = s / grad_div (grad_div = N * G * scale, N the ranks
 * summed, G the micro-steps) from master_in/m_in/v_in into
 * master_out/m_out/v_out and half_out -- written whatever the flag.  Call it
 * per range (buckets of the last micro-step, as they arrive) with the same
 * d_flag, all-reduce (MAX) the flag across the ranks, and pass it to
 * zs_scaler_update: on 0 the *_out buffers hold the state (swap the sets);
 * otherwise they are garbage and the *_in buffers are untouched.  Ranges are
 * offsets into the same shard arrays (16-byte aligned: multiples of 4
 * elements).  The in and out sets must not overlap.  Does not synchronise.
 * Errors as zs_shard_step_oop. */
zs_status zs_update_oop(zs_ctx* ctx, const void* const* grads, int32_t n, zs_dtype dt,
                        int64_t count, const float* acc, float grad_div, const float* master_in,
                        const float* m_in, const float* v_in, float* master_out, float* m_out,
                        float* v_out, void* half_out, const zs_adam_hparams* hp, int64_t step,
                        int32_t* d_flag, cudaStream_t stream);

/* The half-accumulator step (§2.2's 2-byte gradients, §4.2's skipped
 * overflow) without a host round trip, as zs_shard_step_async is to
 * zs_shard_step: the scale, Adam's step count and the learning rate are read
 * from and written to *d_state on the device, nothing is copied to the host,
 * the stream is not synchronised, and the whole step can be captured in a
 * CUDA graph.  In place, or out of place (zs_shard_step_halfacc_async_oop:
 * master, m, v and half are HOST arrays of two device pointers, d_state->buf
 * names the current set; a clean step writes set buf ^ 1 and flips it; acc_half
 * may be NULL when accum_steps == 1).  acc_half holds no defined sums after
 * the call.  Same kernels and arithmetic as the synchronising forms:
 * bit-identical results.  Errors as zs_shard_step_async (argument checks
 * before any launch; a fused step whose barrier wait ran out is reported by
 * the context's next call). */
zs_status zs_shard_step_halfacc_async(zs_ctx* ctx, const void* const* grads, int32_t n,
                                      zs_dtype dt, int64_t count, void* acc_half,
                                      int32_t accum_steps, float* master, float* m, float* v,
                                      void* half_out, const zs_adam_hparams* hp,
                                      const zs_lr_schedule* sched, zs_device_state* d_state,
                                      cudaStream_t stream);
zs_status zs_shard_step_halfacc_async_oop(zs_ctx* ctx, const void* const* grads, int32_t n,
                                          zs_dtype dt, int64_t count, const void* acc_half,
                                          int32_t accum_steps, float* const* master,
                                          float* const* m, float* const* v, void* const* half,
                                          const zs_adam_hparams* hp,
                                          const zs_lr_schedule* sched,
                                          zs_device_state* d_state, cudaStream_t stream);

/* ---------------------------------------------------------------- engine */

/* The training-loop interface of §5.1 (model_engine.backward(loss) then
 * model_engine.step() for every micro-batch; model_engine.global_steps), for
 * one owned shard, on top of the calls above:
 *   zs_engine_backward(e, grads): this micro-batch's n rank slices (what the
 *     reduce-scatter of its gradient buckets would deliver); micro-batches
 *     1..G-1 are summed into acc at once, the G-th is kept for the step;
 *   zs_engine_step(e, ...): after every backward; at the accumulation boundary
 *     (the G-th micro-batch, §4.3) it runs the optimizer step -- zs_shard_step,
 *     or zs_shard_step_clipped when max_grad_norm > 0 -- with the learning rate
 *     of the schedule at Adam's next step, advances the counts and returns the
 *     overflow flag and the new scale; otherwise it does nothing.
 * The engine borrows the caller's buffers (they must outlive it) and owns the
 * loss scaler and the step counts.  The grads pointer arrays are copied; the
 * slices themselves must stay valid until the step that consumes them. */
typedef struct {
  int32_t n;                 /* simulated data-parallel ranks */
  zs_dtype dt;               /* gradient format */
  int64_t count;             /* elements of the owned shard */
  int32_t accum_steps;       /* micro-batches per optimizer step (G) */
  float* acc;                /* count floats (may be NULL only when G == 1) */
  float *master, *m, *v;     /* count floats each */
  void* half_out;            /* count halves */
  zs_adam_hparams hp;        /* hp.lr is used when has_schedule == 0 */
  zs_lr_schedule schedule;   /* used when has_schedule != 0 */
  int32_t has_schedule;
  zs_scaler scaler;          /* initial loss-scale state */
  float max_grad_norm;       /* gradient_clipping; <= 0 disables */
} zs_engine_config;

typedef struct zs_engine zs_engine;

zs_status zs_engine_create(zs_ctx* ctx, const zs_engine_config* cfg, zs_engine** out);
zs_status zs_engine_destroy(zs_engine* e);
zs_status zs_engine_backward(zs_engine* e, const void* const* grads, cudaStream_t stream);
/* *stepped = 1 when this call ran the optimizer step; then *overflow_out,
 * *scale_out and *grad_norm_out (0 unless clipping) describe it.  Any output
 * pointer may be NULL. */
zs_status zs_engine_step(zs_engine* e, int32_t* stepped, int32_t* overflow_out, float* scale_out,
                         float* grad_norm_out, cudaStream_t stream);
/* global_steps: optimizer steps run (skipped ones included), as §5.1 prints;
 * applied_steps: Adam's step count; micro_steps: backward calls so far. */
zs_status zs_engine_state(const zs_engine* e, int64_t* global_steps, int64_t* applied_steps,
                          int64_t* micro_steps, zs_scaler* scaler);

/* ---------------------------------------------------------------- measurement */

/* HBM roofline probe: copy `bytes` from src to dst (read_only = 0), or only
 * read src (read_only = 1; dst receives at most 16 bytes).  bytes must be a
 * multiple of 16. */
zs_status zs_copy_peak(zs_ctx* ctx, const void* src, void* dst, int64_t bytes, int32_t read_only,
                       cudaStream_t stream);

/* Kernel kinds for the timing counters. */
typedef enum {
  ZS_KERNEL_REDUCE = 0,          /* fp32 accumulate of n slices onto acc (+ flag) */
  ZS_KERNEL_CHECK = 1,           /* flag-only pass over n slices */
  ZS_KERNEL_APPLY = 2,           /* AdamW + cast from the accumulator */
  ZS_KERNEL_APPLY_RECOMPUTE = 3, /* AdamW + cast, re-reading the last slices */
  ZS_KERNEL_SCALER = 4,          /* standalone loss-scale update */
  ZS_KERNEL_COPY = 5,            /* roofline probe */
  ZS_KERNEL_SUMSQ = 6,           /* clipping: sum of squares (+ its finalize) */
  ZS_KERNEL_REDUCE_FIRST = 7,    /* first micro-step: sum of n slices into acc (+ flag) */
  ZS_KERNEL_UPDATE_OOP = 8,      /* out-of-place step: last micro-step + flag + update */
  ZS_KERNEL_FUSED = 9,           /* fused step: last micro-step + flag + barrier + update */
  ZS_KERNEL_KINDS = 10
} zs_kernel_kind;

/* When enabled, each launch is bracketed by CUDA events on its stream. */
zs_status zs_ctx_set_timing(zs_ctx* ctx, int32_t enable);
/* Device time (ms), launches and elements of one kernel kind since the last
 * reset; waits for the recorded events. */
zs_status zs_ctx_timing(zs_ctx* ctx, int32_t kind, double* total_ms, int64_t* launches,
                        int64_t* elements);
zs_status zs_ctx_timing_reset(zs_ctx* ctx);
/* Kernels launched by this context since creation (always counted). */
zs_status zs_ctx_launch_count(const zs_ctx* ctx, int64_t* launches);

#ifdef __cplusplus
}
#endif

#endif /* ZEROSHARD_H */
