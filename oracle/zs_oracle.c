/*
 * CPU oracle for the ZeRO shard step.  TEST INFRASTRUCTURE ONLY: see
 * zs_oracle.h for the sources, the readings and the pins.
 * Build: gcc -O1 -std=c11 -ffp-contract=off -fPIC -shared zs_oracle.c -lm
 * (-ffp-contract=off keeps every a*b+c as two rounded ops on x86 and Arm).
 */
#include "zs_oracle.h"

#include <math.h>
#include <stddef.h>

/* ---- partition and memory accounting (§2, §2.1-§2.3) ------------------- */

int zso_partition(int64_t psi, int32_t n, int32_t align, int64_t* psi_pad, int64_t* shard_len) {
  if (psi < 0 || n < 1 || align < 1 || psi_pad == NULL || shard_len == NULL) return -1;
  int64_t unit = (int64_t)n * (int64_t)align;
  int64_t units = psi / unit + (psi % unit != 0 ? 1 : 0);
  *psi_pad = units * unit;
  *shard_len = *psi_pad / n;
  return 0;
}

int zso_shard_range(int64_t psi, int64_t shard_len, int32_t n, int32_t rank, int64_t* begin,
                    int64_t* valid_end, int64_t* padded_end) {
  if (rank < 0 || rank >= n || shard_len < 0) return -1;
  int64_t b = (int64_t)rank * shard_len;
  int64_t e = b + shard_len;
  int64_t ve = e < psi ? e : psi;
  if (ve < b) ve = b;
  *begin = b;
  *valid_end = ve;
  *padded_end = e;
  return 0;
}

int zso_state_bytes(int64_t psi, int64_t shard_len, int32_t stage, uint64_t* bytes) {
  uint64_t P = (uint64_t)psi, E = (uint64_t)shard_len;
  switch (stage) {
    case 0: /* plain data parallel: 2 + 2 + 4 + 4 + 4 bytes per parameter */
      *bytes = 2 * P + 2 * P + 4 * P + 4 * P + 4 * P;
      return 0;
    case 1: /* fp16 params and grads replicated; master, m, v split */
      *bytes = 2 * P + 2 * P + (4 + 4 + 4) * E;
      return 0;
    case 2: /* fp16 params replicated; grads and optimizer state split */
      *bytes = 2 * P + (2 + 4 + 4 + 4) * E;
      return 0;
    case 3: /* everything split */
      *bytes = (2 + 2 + 4 + 4 + 4) * E;
      return 0;
    default:
      return -1;
  }
}

/* ---- IEEE half formats, written from the binary16 / bfloat16 layouts ---- */

typedef struct {
  int mant_bits, exp_bits, bias;
} fmt_t;

static fmt_t fmt_of(int32_t dtype) {
  fmt_t f;
  if (dtype == ZSO_FP16) {
    f.mant_bits = 10;
    f.exp_bits = 5;
    f.bias = 15;
  } else {
    f.mant_bits = 7;
    f.exp_bits = 8;
    f.bias = 127;
  }
  return f;
}

double zso_half_to_double(uint16_t bits, int32_t dtype) {
  fmt_t f = fmt_of(dtype);
  int sign = (bits >> 15) & 1;
  int efield = (bits >> f.mant_bits) & ((1 << f.exp_bits) - 1);
  int mant = bits & ((1 << f.mant_bits) - 1);
  int efield_max = (1 << f.exp_bits) - 1;
  double mag;
  if (efield == efield_max) {
    mag = mant ? NAN : INFINITY;
  } else if (efield == 0) { /* zero or subnormal: mant * 2^(1 - bias - mant_bits) */
    mag = ldexp((double)mant, 1 - f.bias - f.mant_bits);
  } else { /* normal: (2^mant_bits + mant) * 2^(efield - bias - mant_bits) */
    mag = ldexp((double)((1 << f.mant_bits) | mant), efield - f.bias - f.mant_bits);
  }
  return sign ? -mag : mag;
}

uint16_t zso_f32_to_half(float xf, int32_t dtype) {
  fmt_t f = fmt_of(dtype);
  const int mb = f.mant_bits;
  const int efield_max = (1 << f.exp_bits) - 1;
  double x = (double)xf;
  uint16_t sign = signbit(x) ? 0x8000u : 0u;
  if (isnan(x)) return (uint16_t)(sign | (efield_max << mb) | (1 << (mb - 1)));
  if (isinf(x)) return (uint16_t)(sign | (efield_max << mb));
  double a = fabs(x);
  if (a == 0.0) return sign;
  const int emin = 1 - f.bias; /* exponent of the smallest normal */
  int e;
  (void)frexp(a, &e);
  e -= 1; /* a = s * 2^e with s in [1, 2) */
  if (e < emin) e = emin;
  double q = ldexp(1.0, e - mb); /* spacing of the target format around a */
  double y = a / q;              /* exact: power-of-two scaling */
  double r = floor(y);
  double frac = y - r;
  if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0; /* nearest, ties to even */
  double val = r * q;
  double maxf = ldexp((double)((2 << mb) - 1), efield_max - 1 - f.bias - mb);
  if (val > maxf) return (uint16_t)(sign | (efield_max << mb));
  if (val == 0.0) return sign;
  int ev;
  (void)frexp(val, &ev);
  ev -= 1;
  if (ev < emin) { /* subnormal */
    int mant = (int)(val / ldexp(1.0, emin - mb));
    return (uint16_t)(sign | mant);
  }
  int mant = (int)(val / ldexp(1.0, ev - mb)) - (1 << mb);
  return (uint16_t)(sign | ((ev + f.bias) << mb) | mant);
}

void zso_half_to_double_array(const uint16_t* bits, int64_t count, int32_t dtype, double* out) {
  for (int64_t i = 0; i < count; ++i) out[i] = zso_half_to_double(bits[i], dtype);
}

void zso_f32_to_half_array(const float* x, int64_t count, int32_t dtype, uint16_t* out) {
  for (int64_t i = 0; i < count; ++i) out[i] = zso_f32_to_half(x[i], dtype);
}

/* ---- reduce-scatter sum + micro-step accumulation (§2.2, §4.3) ---------- */

void zso_reduce_accumulate(const uint16_t* const* slices, int32_t n, int32_t dtype, int64_t count,
                           float* acc, int32_t first) {
  for (int64_t i = 0; i < count; ++i) {
    float a = first ? 0.0f : acc[i];
    for (int32_t r = 0; r < n; ++r) {
      float gr = (float)zso_half_to_double(slices[r][i], dtype); /* exact */
      a = a + gr;
    }
    acc[i] = a;
  }
}

int32_t zso_any_nonfinite(const uint16_t* const* slices, int32_t n, int32_t dtype, int64_t count) {
  for (int32_t r = 0; r < n; ++r) {
    for (int64_t i = 0; i < count; ++i) {
      double x = zso_half_to_double(slices[r][i], dtype);
      if (isnan(x) || isinf(x)) return 1;
    }
  }
  return 0;
}

int32_t zso_any_nonfinite_f32(const float* x, int64_t count) {
  for (int64_t i = 0; i < count; ++i) {
    if (isnan(x[i]) || isinf(x[i])) return 1;
  }
  return 0;
}

/* ---- AdamW on the fp32 master shard, then the half copy (§2.1, §4.1) ---- */

void zso_adamw_apply_clipped(const float* acc, int64_t count, double grad_div, double coef,
                             float* master, float* m, float* v, uint16_t* half_out,
                             int32_t dtype, const zso_hparams* hp, int64_t t) {
  const double b1 = hp->beta1, b2 = hp->beta2;
  const double bc1 = 1.0 - pow(b1, (double)t);
  const double bc2 = 1.0 - pow(b2, (double)t);
  for (int64_t i = 0; i < count; ++i) {
    double g = (double)acc[i] / grad_div * coef; /* unscale, average, clip */
    double p = (double)master[i];
    double m1 = b1 * (double)m[i] + (1.0 - b1) * g;
    double v1 = b2 * (double)v[i] + (1.0 - b2) * g * g;
    double m_hat = m1 / bc1;
    double v_hat = v1 / bc2;
    double p1 = p - hp->lr * (m_hat / (sqrt(v_hat) + hp->eps) + hp->weight_decay * p);
    master[i] = (float)p1;
    m[i] = (float)m1;
    v[i] = (float)v1;
    half_out[i] = zso_f32_to_half(master[i], dtype);
  }
}

void zso_adamw_apply(const float* acc, int64_t count, double grad_div, float* master, float* m,
                     float* v, uint16_t* half_out, int32_t dtype, const zso_hparams* hp,
                     int64_t t) {
  zso_adamw_apply_clipped(acc, count, grad_div, 1.0, master, m, v, half_out, dtype, hp, t);
}

double zso_grad_sumsq(const float* acc, int64_t count, double grad_div) {
  double s = 0.0;
  for (int64_t i = 0; i < count; ++i) {
    double g = (double)acc[i] / grad_div;
    s += g * g;
  }
  return s;
}

double zso_clip_coef(double sumsq_total, double max_norm) {
  if (!(max_norm > 0.0)) return 1.0;
  double c = max_norm / (sqrt(sumsq_total) + 1e-6);
  return c < 1.0 ? c : 1.0;
}

/* ---- half-precision accumulator variant (§2 table, §2.2) ---------------- */

void zso_reduce_accumulate_half(const uint16_t* const* slices, int32_t n, int32_t dtype,
                                int64_t count, uint16_t* acc_half, int32_t first) {
  for (int64_t i = 0; i < count; ++i) {
    float a = first ? 0.0f : (float)zso_half_to_double(acc_half[i], dtype);
    for (int32_t r = 0; r < n; ++r) a = a + (float)zso_half_to_double(slices[r][i], dtype);
    acc_half[i] = zso_f32_to_half(a, dtype);
  }
}

int32_t zso_shard_step_halfacc(const uint16_t* const* grads, int32_t g, int32_t n,
                               int32_t dtype, int64_t count, uint16_t* acc_half, float* master,
                               float* m, float* v, uint16_t* half_out, const zso_hparams* hp,
                               int64_t* t, zso_scaler* sc, int32_t extra_overflow) {
  for (int32_t k = 0; k < g; ++k)
    zso_reduce_accumulate_half(grads + (size_t)k * n, n, dtype, count, acc_half, k == 0);
  int32_t ovf = extra_overflow != 0;
  for (int32_t k = 0; k < g && !ovf; ++k) ovf = zso_any_nonfinite(grads + (size_t)k * n, n,
                                                                  dtype, count);
  const uint16_t* accp[1] = {acc_half};
  if (!ovf) ovf = zso_any_nonfinite(accp, 1, dtype, count);
  if (!ovf) {
    *t += 1;
    const double div = (double)n * (double)g * sc->scale;
    const double b1 = hp->beta1, b2 = hp->beta2;
    const double bc1 = 1.0 - pow(b1, (double)*t);
    const double bc2 = 1.0 - pow(b2, (double)*t);
    for (int64_t i = 0; i < count; ++i) {
      double gi = zso_half_to_double(acc_half[i], dtype) / div;
      double p = (double)master[i];
      double m1 = b1 * (double)m[i] + (1.0 - b1) * gi;
      double v1 = b2 * (double)v[i] + (1.0 - b2) * gi * gi;
      double p1 = p - hp->lr * ((m1 / bc1) / (sqrt(v1 / bc2) + hp->eps) + hp->weight_decay * p);
      master[i] = (float)p1;
      m[i] = (float)m1;
      v[i] = (float)v1;
      half_out[i] = zso_f32_to_half(master[i], dtype);
    }
  }
  zso_scaler_update(sc, ovf);
  return ovf;
}

/* ---- learning-rate schedules (§4.4) ------------------------------------ */

double zso_lr_at(int32_t kind, double min_lr, double max_lr, int64_t warmup_steps,
                 int64_t total_steps, int64_t t) {
  if (kind == ZSO_LR_CONSTANT) return max_lr;
  double frac = warmup_steps > 0 ? (double)t / (double)warmup_steps : 1.0;
  if (frac > 1.0) frac = 1.0;
  double warm = min_lr + (max_lr - min_lr) * frac;
  if (kind == ZSO_LR_WARMUP || t <= warmup_steps) return warm;
  /* ZSO_LR_WARMUP_DECAY after the warmup */
  if (total_steps <= warmup_steps) return 0.0;
  double rest = (double)(total_steps - t) / (double)(total_steps - warmup_steps);
  if (rest < 0.0) rest = 0.0;
  return max_lr * rest;
}

/* ---- dynamic loss scale (§4.2) ------------------------------------------ */

void zso_scaler_update(zso_scaler* s, int32_t overflow) {
  if (overflow) {
    s->clean_count = 0;
    if (s->dynamic) {
      s->hyst_left -= 1;
      if (s->hyst_left <= 0) {
        double half = s->scale / 2.0;
        s->scale = half > s->min_scale ? half : s->min_scale;
        s->hyst_left = s->hysteresis;
      }
    }
    return;
  }
  if (s->dynamic) {
    s->clean_count += 1;
    if (s->clean_count >= s->window) {
      s->scale *= 2.0;
      s->clean_count = 0;
    }
    if (s->consecutive) s->hyst_left = s->hysteresis;
  }
}

/* ---- one step of one owned shard ---------------------------------------- */

int32_t zso_shard_step_clipped(const uint16_t* const* grads, int32_t g, int32_t n, int32_t dtype,
                               int64_t count, float* acc, float* master, float* m, float* v,
                               uint16_t* half_out, const zso_hparams* hp, int64_t* t,
                               zso_scaler* sc, int32_t extra_overflow, double max_norm,
                               double* norm_out) {
  for (int32_t k = 0; k < g; ++k) zso_reduce_accumulate(grads + (size_t)k * n, n, dtype, count,
                                                        acc, k == 0);
  int32_t ovf = extra_overflow != 0;
  for (int32_t k = 0; k < g && !ovf; ++k) ovf = zso_any_nonfinite(grads + (size_t)k * n, n,
                                                                  dtype, count);
  if (!ovf) ovf = zso_any_nonfinite_f32(acc, count);
  if (norm_out) *norm_out = 0.0;
  if (!ovf) {
    *t += 1;
    const double div = (double)n * (double)g * sc->scale;
    double coef = 1.0;
    if (max_norm > 0.0) {
      const double sumsq = zso_grad_sumsq(acc, count, div);
      coef = zso_clip_coef(sumsq, max_norm);
      if (norm_out) *norm_out = sqrt(sumsq);
    }
    zso_adamw_apply_clipped(acc, count, div, coef, master, m, v, half_out, dtype, hp, *t);
  }
  zso_scaler_update(sc, ovf);
  return ovf;
}

int32_t zso_shard_step(const uint16_t* const* grads, int32_t g, int32_t n, int32_t dtype,
                       int64_t count, float* acc, float* master, float* m, float* v,
                       uint16_t* half_out, const zso_hparams* hp, int64_t* t, zso_scaler* sc,
                       int32_t extra_overflow) {
  return zso_shard_step_clipped(grads, g, n, dtype, count, acc, master, m, v, half_out, hp, t,
                                sc, extra_overflow, 0.0, NULL);
}
