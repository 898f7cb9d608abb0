/*
 * CPU oracle for the ZeRO-partitioned mixed-precision optimizer shard step.
 *
 * TEST INFRASTRUCTURE ONLY.  Plain, slow, single-threaded C in fp64 (fp32
 * only where the step itself is defined in fp32: the gradient accumulator and
 * the stored optimizer state).  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark load it; the CUDA library never does, and it
 * shares no code with the CUDA library.
 *
 * Sources (page title, section):
 *  - DeepSpeed Complete Guide (youngju.dev), §2 memory table: fp16 params and
 *    grads (2 bytes each), fp32 master params, Adam momentum and variance
 *    (4 bytes each), 16 bytes per parameter in all.
 *  - same page, §2.1 (ZeRO-1: optimizer state split N ways, each rank updates
 *    only its shard), §2.2 (ZeRO-2: gradients split too; each rank accumulates
 *    only the gradients of its shard, delivered by reduce-scatter), §2.3
 *    (ZeRO-3: parameters split too).
 *  - same page, §4.1 and §4.2: AdamW with eps 1e-8; fp16 dynamic loss scale
 *    starting at 2^16, loss_scale_window clean steps before an increase,
 *    hysteresis overflows before a decrease, min_loss_scale.
 *  - same page, §4.3: train batch = micro batch x accumulation steps x world
 *    size, so the applied gradient is the mean over ranks and micro-steps.
 *  - DeepSpeed (aibars.net), core features: fp16 training, gradient
 *    accumulation, dynamic loss scaling.
 *
 * Readings where the pages are silent:
 *  - Adam is the textbook bias-corrected form with eps added to sqrt(v_hat),
 *    and AdamW's decay is decoupled: p -= lr * (m_hat/(sqrt(v_hat)+eps) + wd*p).
 *  - The accumulator is fp32; per element it adds the slices in micro-step
 *    order, then rank order 0..N-1, starting from +0.0, one IEEE fp32 add each.
 *  - Overflow = any +-inf or NaN in any input slice of the step, or an fp32
 *    accumulated gradient that is not finite (finite bf16 inputs near the top
 *    of their range can sum past the fp32 maximum; fp16 inputs cannot); a
 *    skipped step leaves master, m, v, the half copy and the Adam step count
 *    as they were.
 *  - The scale doubles when `window` consecutive clean steps have passed since
 *    the last overflow or increase; it halves (not below min_scale) on the
 *    `hysteresis`-th overflow since the last decrease; with
 *    consecutive_hysteresis (a §4.2 knob the pages name but do not define) a
 *    clean step restores the count, so only consecutive overflows halve it.
 *  - Hyper-parameters are taken as the fp32 values the library receives;
 *    the arithmetic of one step is fp64; master, m and v are rounded to fp32
 *    (nearest even) between steps and the half copy is the fp32 master
 *    rounded to nearest even.
 *
 * Parity pins (tests/test_oracle_pins.py): memory closed forms; shard bounds
 * by enumeration; exact-rational sums and an order-sensitive case for the
 * accumulator; Adam closed forms at t=1, at every t under a constant gradient
 * and at t=2 for two given gradients; decoupled decay at g=0; the hand-worked
 * scaler trace; half rounding against numpy (fp16) and torch (bf16) over
 * every fp16 pattern and crafted ties; shard union and bucket invariance;
 * ten-step runs (a skipped step, a halved scale, clipping, both accumulator
 * formats) against torch.optim.AdamW and clip_grad_norm_ in fp64 fed the same
 * mean gradient, with master/m/v rounded to fp32 between steps on both sides
 * (that rounding is the one reading those runs share with this file).
 */
#ifndef ZS_ORACLE_H
#define ZS_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ZSO_FP16 0
#define ZSO_BF16 1

typedef struct {
  double lr, beta1, beta2, eps, weight_decay;
} zso_hparams;

typedef struct {
  double scale, min_scale;
  int32_t window, clean_count, hysteresis, hyst_left, dynamic, consecutive;
} zso_scaler;

/* Partition (§2.1-§2.3): psi_pad = round_up(psi, n*align); shard_len = psi_pad/n. */
int zso_partition(int64_t psi, int32_t n, int32_t align, int64_t* psi_pad, int64_t* shard_len);
/* Rank r owns [r*E, (r+1)*E); its valid part ends at min((r+1)*E, psi), clamped to begin. */
int zso_shard_range(int64_t psi, int64_t shard_len, int32_t n, int32_t rank, int64_t* begin,
                    int64_t* valid_end, int64_t* padded_end);
/* Per-rank model-state bytes by ZeRO stage 0..3 (§2 table, §2.1-§2.3), with E = shard_len. */
int zso_state_bytes(int64_t psi, int64_t shard_len, int32_t stage, uint64_t* bytes);

double zso_half_to_double(uint16_t bits, int32_t dtype);
uint16_t zso_f32_to_half(float x, int32_t dtype);
/* Array forms of the two conversions above. */
void zso_half_to_double_array(const uint16_t* bits, int64_t count, int32_t dtype, double* out);
void zso_f32_to_half_array(const float* x, int64_t count, int32_t dtype, uint16_t* out);

/* acc[i] = (first ? +0.0f : acc[i]) + s_0[i] + s_1[i] + ... (fp32, in order). */
void zso_reduce_accumulate(const uint16_t* const* slices, int32_t n, int32_t dtype, int64_t count,
                           float* acc, int32_t first);
/* 1 iff any element of any slice is +-inf or NaN. */
int32_t zso_any_nonfinite(const uint16_t* const* slices, int32_t n, int32_t dtype, int64_t count);
/* 1 iff any fp32 value is +-inf or NaN (an accumulator that overflowed). */
int32_t zso_any_nonfinite_f32(const float* x, int64_t count);
/* Clean-step update of one range: g = acc / grad_div, then AdamW at step t (1-based). */
void zso_adamw_apply(const float* acc, int64_t count, double grad_div, float* master, float* m,
                     float* v, uint16_t* half_out, int32_t dtype, const zso_hparams* hp, int64_t t);
void zso_scaler_update(zso_scaler* s, int32_t overflow);

/* Global-norm gradient clipping (§4.1 gradient_clipping, §5.1 "step() includes
 * gradient clipping"; the formula is the usual one, not printed on the pages):
 * sumsq = sum over the range of (acc[i] / grad_div)^2 in fp64, index order;
 * the norm of the whole model is the square root of the sum over all shards;
 * coef = max_norm / (norm + 1e-6) if that is below 1, else 1 (max_norm <= 0:
 * no clipping); the update then uses g = acc[i] / grad_div * coef. */
double zso_grad_sumsq(const float* acc, int64_t count, double grad_div);
double zso_clip_coef(double sumsq_total, double max_norm);
void zso_adamw_apply_clipped(const float* acc, int64_t count, double grad_div, double coef,
                             float* master, float* m, float* v, uint16_t* half_out,
                             int32_t dtype, const zso_hparams* hp, int64_t t);

/* One optimizer step of one owned-shard view.  grads holds g*n pointers,
 * micro-step major: grads[k*n + r] is rank r's slice in micro-step k.
 * extra_overflow is OR'd into the step's flag (other shards' flags).
 * Returns the flag; advances *t only on a clean step. */
int32_t zso_shard_step(const uint16_t* const* grads, int32_t g, int32_t n, int32_t dtype,
                       int64_t count, float* acc, float* master, float* m, float* v,
                       uint16_t* half_out, const zso_hparams* hp, int64_t* t, zso_scaler* sc,
                       int32_t extra_overflow);

/* Half-precision accumulator variant: the accumulated gradient is kept in the
 * gradient's own 2-byte format, as the pages' accounting counts gradients
 * (2 bytes per parameter, §2 table; 2Ψ/N per rank under ZeRO-2, §2.2).  Per
 * micro-step and element: a = (first ? +0.0f : acc_half as fp32) + s_0 + ...
 * + s_{n-1} in fp32, rank order, then acc_half = a rounded to nearest even.
 * A sum past the half maximum rounds to infinity and makes the step
 * overflow.  The update reads the half accumulator (exactly converted). */
void zso_reduce_accumulate_half(const uint16_t* const* slices, int32_t n, int32_t dtype,
                                int64_t count, uint16_t* acc_half, int32_t first);
int32_t zso_shard_step_halfacc(const uint16_t* const* grads, int32_t g, int32_t n,
                               int32_t dtype, int64_t count, uint16_t* acc_half, float* master,
                               float* m, float* v, uint16_t* half_out, const zso_hparams* hp,
                               int64_t* t, zso_scaler* sc, int32_t extra_overflow);

/* Learning-rate schedules named in §4.4 (the pages give WarmupDecayLR's knobs:
 * warmup_min_lr, warmup_max_lr, warmup_num_steps, total_num_steps,
 * warmup_type "linear"; the formulas are the plain linear reading), at the
 * Adam step t (1-based count of applied updates, this one included):
 *   ZSO_LR_CONSTANT:      max_lr
 *   ZSO_LR_WARMUP:        min_lr + (max_lr - min_lr) * min(1, t / warmup_steps)
 *   ZSO_LR_WARMUP_DECAY:  the warmup above for t <= warmup_steps, then
 *                         max_lr * max(0, (total_steps - t) / (total_steps - warmup_steps)) */
#define ZSO_LR_CONSTANT 0
#define ZSO_LR_WARMUP 1
#define ZSO_LR_WARMUP_DECAY 2
double zso_lr_at(int32_t kind, double min_lr, double max_lr, int64_t warmup_steps,
                 int64_t total_steps, int64_t t);

/* zso_shard_step with global-norm clipping over this view (the view is the
 * whole model, or the caller accepts the view's own norm); *norm_out gets the
 * gradient norm (0 on a skipped step). */
int32_t zso_shard_step_clipped(const uint16_t* const* grads, int32_t g, int32_t n, int32_t dtype,
                               int64_t count, float* acc, float* master, float* m, float* v,
                               uint16_t* half_out, const zso_hparams* hp, int64_t* t,
                               zso_scaler* sc, int32_t extra_overflow, double max_norm,
                               double* norm_out);

#ifdef __cplusplus
}
#endif

#endif
