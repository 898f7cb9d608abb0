/*
 * Seeded synthetic inputs for the ZeRO shard step: gradients and fp32 master
 * initial values, as a pure function of (seed, stream, step, micro-step,
 * rank, flat parameter index).
 *
 * This module is shared by the test/bench harness on both sides: the host
 * library (synth_host.c, compiled by gcc) feeds the CPU oracle, and the device
 * library (synth_dev.cu) fills HBM buffers for the CUDA path.  It holds none
 * of the optimizer's arithmetic: no reduction, no unscaling, no Adam, no
 * loss-scale logic and no half-precision rounding (the harness converts the
 * fp32 values returned here with a library RNE conversion on each side).
 *
 * Every floating-point operation below is a single IEEE-754 binary32 op in a
 * fixed order (explicit __f*_rn intrinsics on the device, plain C float ops
 * compiled with -ffp-contract=off on the host), so both sides produce the same
 * bits.
 *
 * Generator: Philox4x64-10, from its published definition (J. Salmon,
 * M. Moraes, R. Dror, D. Shaw, "Parallel random numbers: as easy as 1, 2, 3",
 * SC'11): ten rounds of two 64x64->128 multiplies with the key bumped by the
 * Weyl constants between rounds.  numpy's Philox bit generator implements the
 * same function and pins it in the tests.
 *
 * Normal variates: Irwin-Hall sum of twelve 16-bit uniforms on bin midpoints,
 * z = (2*sum(u_j) - 12*65535) / 131072, so |z| <= 6 and var(z) = 1 - 2^-32.
 * The numerator is an integer below 2^20, so z*c is one rounding.
 * Student-t(3) variates: z0 / sqrt((z1^2 + z2^2 + z3^2) / 3).
 */
#ifndef ZS_SYNTH_H
#define ZS_SYNTH_H

#include <stdint.h>

#ifdef __CUDACC__
#define ZS_SYNTH_FN __host__ __device__ static inline
#else
#define ZS_SYNTH_FN static inline
#endif

/* Stream tags: the third counter word. */
#define ZS_SYNTH_TAG_GRAD 1u
#define ZS_SYNTH_TAG_TAIL 2u
#define ZS_SYNTH_TAG_MASTER 3u

#define ZS_SYNTH_MAX_SEG 4

/* Recipe for one gradient tensor family.  All constants are fp32 values the
 * harness derives once from (sigma, loss scale); both sides receive the same
 * struct. */
typedef struct {
  uint64_t seed;            /* key word 0 */
  uint64_t stream;          /* key word 1: workload id */
  float c_normal;           /* fp32(sigma * S / 131072): z-numerator -> value */
  float c_tail;             /* fp32(sigma * S): Student-t variate -> value */
  uint32_t tail_threshold;  /* element is heavy-tailed iff u32 < threshold; 0 = never */
  int32_t n_seg;            /* flat-index segments with their own c_normal */
  int64_t seg_begin[ZS_SYNTH_MAX_SEG];
  int64_t seg_end[ZS_SYNTH_MAX_SEG];
  float seg_c[ZS_SYNTH_MAX_SEG];
  int32_t pad_;
} zs_synth_grad_recipe;

ZS_SYNTH_FN void zs_synth_mulhilo64(uint64_t a, uint64_t b, uint64_t* hi, uint64_t* lo) {
#ifdef __CUDA_ARCH__
  *lo = a * b;
  *hi = __umul64hi(a, b);
#else
  unsigned __int128 p = (unsigned __int128)a * (unsigned __int128)b;
  *lo = (uint64_t)p;
  *hi = (uint64_t)(p >> 64);
#endif
}

/* Philox4x64 with 10 rounds. */
ZS_SYNTH_FN void zs_synth_philox4x64_10(const uint64_t ctr[4], const uint64_t key[2], uint64_t out[4]) {
  uint64_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
  uint64_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += 0x9E3779B97F4A7C15ull;
      k1 += 0xBB67AE8584CAA73Bull;
    }
    uint64_t hi0, lo0, hi1, lo1;
    zs_synth_mulhilo64(0xD2E7470EE14C6C93ull, c0, &hi0, &lo0);
    zs_synth_mulhilo64(0xCA5A826395121157ull, c2, &hi1, &lo1);
    uint64_t n0 = hi1 ^ c1 ^ k0;
    uint64_t n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
  }
  out[0] = c0;
  out[1] = c1;
  out[2] = c2;
  out[3] = c3;
}

/* Counter word 1 packs (step, micro-step, rank). */
ZS_SYNTH_FN uint64_t zs_synth_srm(uint32_t step, uint32_t micro, uint32_t rank) {
  return ((uint64_t)(step & 0xFFFFFFu) << 40) | ((uint64_t)(micro & 0xFFFFu) << 24) |
         (uint64_t)(rank & 0xFFFFFFu);
}

ZS_SYNTH_FN void zs_synth_block(uint64_t seed, uint64_t stream, uint64_t index, uint64_t srm,
                                uint64_t tag, uint64_t draw, uint64_t out[4]) {
  uint64_t ctr[4];
  uint64_t key[2];
  ctr[0] = index;
  ctr[1] = srm;
  ctr[2] = tag;
  ctr[3] = draw;
  key[0] = seed;
  key[1] = stream;
  zs_synth_philox4x64_10(ctr, key, out);
}

/* Irwin-Hall(12) numerator from the first twelve 16-bit lanes (words 0..2). */
ZS_SYNTH_FN int32_t zs_synth_ih12_num(const uint64_t w[4]) {
  int32_t s = 0;
  for (int k = 0; k < 3; ++k) {
    uint64_t x = w[k];
    for (int j = 0; j < 4; ++j) {
      s += (int32_t)(x & 0xFFFFu);
      x >>= 16;
    }
  }
  return 2 * s - 12 * 65535;
}

ZS_SYNTH_FN float zs_synth_mul(float a, float b) {
#ifdef __CUDA_ARCH__
  return __fmul_rn(a, b);
#else
  return a * b;
#endif
}
ZS_SYNTH_FN float zs_synth_add(float a, float b) {
#ifdef __CUDA_ARCH__
  return __fadd_rn(a, b);
#else
  return a + b;
#endif
}
ZS_SYNTH_FN float zs_synth_div(float a, float b) {
#ifdef __CUDA_ARCH__
  return __fdiv_rn(a, b);
#else
  return a / b;
#endif
}
ZS_SYNTH_FN float zs_synth_sqrt(float a) {
#ifdef __CUDA_ARCH__
  return __fsqrt_rn(a);
#else
  return __builtin_sqrtf(a);
#endif
}

/* Student-t(3) variate built from four Irwin-Hall normals (draws 0..3 of the
 * tail stream). */
ZS_SYNTH_FN float zs_synth_t3(uint64_t seed, uint64_t stream, uint64_t index, uint64_t srm) {
  float z[4];
  for (int d = 0; d < 4; ++d) {
    uint64_t w[4];
    zs_synth_block(seed, stream, index, srm, ZS_SYNTH_TAG_TAIL, (uint64_t)d, w);
    /* exact: |num| < 2^20 and the factor is a power of two */
    z[d] = zs_synth_mul((float)zs_synth_ih12_num(w), 1.0f / 131072.0f);
  }
  float q = zs_synth_mul(z[1], z[1]);
  q = zs_synth_add(q, zs_synth_mul(z[2], z[2]));
  q = zs_synth_add(q, zs_synth_mul(z[3], z[3]));
  float den = zs_synth_sqrt(zs_synth_div(q, 3.0f));
  return zs_synth_div(z[0], den);
}

/* fp32 gradient value (before the half conversion) of rank `rank`, micro-step
 * `micro`, step `step` at flat index `index`.  Padding is the caller's job. */
ZS_SYNTH_FN float zs_synth_grad_value(const zs_synth_grad_recipe* r, uint64_t index, uint32_t step,
                                      uint32_t micro, uint32_t rank) {
  uint64_t srm = zs_synth_srm(step, micro, rank);
  uint64_t w[4];
  zs_synth_block(r->seed, r->stream, index, srm, ZS_SYNTH_TAG_GRAD, 0, w);
  if (r->tail_threshold != 0u && (uint32_t)(w[3] & 0xFFFFFFFFu) < r->tail_threshold) {
    return zs_synth_mul(zs_synth_t3(r->seed, r->stream, index, srm), r->c_tail);
  }
  float c = r->c_normal;
  for (int s = 0; s < r->n_seg && s < ZS_SYNTH_MAX_SEG; ++s) {
    if ((int64_t)index >= r->seg_begin[s] && (int64_t)index < r->seg_end[s]) c = r->seg_c[s];
  }
  return zs_synth_mul((float)zs_synth_ih12_num(w), c);
}

/* fp32 master initial value at flat index `index`: Irwin-Hall normal times
 * c = fp32(sigma / 131072). */
ZS_SYNTH_FN float zs_synth_master_value(uint64_t seed, uint64_t stream, float c, uint64_t index) {
  uint64_t w[4];
  zs_synth_block(seed, stream, index, 0, ZS_SYNTH_TAG_MASTER, 0, w);
  return zs_synth_mul((float)zs_synth_ih12_num(w), c);
}

#endif /* ZS_SYNTH_H */
