/* A plain C caller of libzeroshard: no Python, no torch.  Reads a step's
 * inputs from a file, runs G micro-steps through zs_grad_accum and
 * zs_shard_step with cudaMalloc'ed buffers, and writes the updated state.
 * A third argument picks another form of the last call: "oop" is
 * zs_shard_step_oop (the new state lands in a second set of buffers, which a
 * clean step makes current); "multi" is zs_shard_step with the fused
 * single-kernel step turned off (zs_ctx_set_fused); "twophase" is
 * zs_update_oop over two ranges with the context's flag, then
 * zs_scaler_update on that flag.
 *
 * Input file:  int64 count, n, g; float scale; float lr, beta1, beta2, eps, wd;
 *              g*n*count uint16 gradients (micro-step major); count float master.
 * Output file: int32 overflow; float new_scale; count float master, m, v;
 *              count uint16 half copy.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "zeroshard.h"

#define CHECK(x)                                                         \
  do {                                                                   \
    if (!(x)) {                                                          \
      fprintf(stderr, "failed: %s (line %d)\n", #x, __LINE__);           \
      return 1;                                                          \
    }                                                                    \
  } while (0)

int main(int argc, char** argv) {
  CHECK(argc == 3 || argc == 4);
  const char* form = argc == 4 ? argv[3] : "";
  const int oop = strcmp(form, "oop") == 0;
  const int multi = strcmp(form, "multi") == 0;
  const int twophase = strcmp(form, "twophase") == 0;
  CHECK(argc == 3 || oop || multi || twophase);
  FILE* in = fopen(argv[1], "rb");
  CHECK(in != NULL);
  int64_t hdr[3];
  float f[6];
  CHECK(fread(hdr, sizeof(int64_t), 3, in) == 3);
  CHECK(fread(f, sizeof(float), 6, in) == 6);
  const int64_t count = hdr[0], n = hdr[1], g = hdr[2];
  const size_t ng = (size_t)(n * g);
  uint16_t* hgrad = (uint16_t*)malloc(ng * count * 2);
  float* hmaster = (float*)malloc(count * 4);
  CHECK(hgrad && hmaster);
  CHECK(fread(hgrad, 2, ng * count, in) == ng * count);
  CHECK(fread(hmaster, 4, count, in) == (size_t)count);
  fclose(in);

  /* every slice on its own allocation: 256-byte aligned */
  void** dgrad = (void**)malloc(ng * sizeof(void*));
  for (size_t i = 0; i < ng; ++i) {
    CHECK(cudaMalloc(&dgrad[i], count * 2) == cudaSuccess);
    CHECK(cudaMemcpy(dgrad[i], hgrad + i * count, count * 2, cudaMemcpyHostToDevice) ==
          cudaSuccess);
  }
  float *acc, *master, *m, *v;
  void* half;
  CHECK(cudaMalloc((void**)&acc, count * 4) == cudaSuccess);
  CHECK(cudaMalloc((void**)&master, count * 4) == cudaSuccess);
  CHECK(cudaMalloc((void**)&m, count * 4) == cudaSuccess);
  CHECK(cudaMalloc((void**)&v, count * 4) == cudaSuccess);
  CHECK(cudaMalloc(&half, count * 2) == cudaSuccess);
  CHECK(cudaMemcpy(master, hmaster, count * 4, cudaMemcpyHostToDevice) == cudaSuccess);
  CHECK(cudaMemset(m, 0, count * 4) == cudaSuccess);
  CHECK(cudaMemset(v, 0, count * 4) == cudaSuccess);

  zs_ctx* ctx = NULL;
  CHECK(zs_ctx_create(&ctx) == ZS_OK);
  if (multi) CHECK(zs_ctx_set_fused(ctx, ZS_FUSED_OFF, 0) == ZS_OK);
  zs_scaler sc;
  CHECK(zs_scaler_init(&sc, f[0], 1.0f, 1000, 1, 1) == ZS_OK);
  zs_adam_hparams hp = {f[1], f[2], f[3], f[4], f[5]};
  for (int64_t k = 0; k + 1 < g; ++k) {
    zs_status st = zs_grad_accum(ctx, (const void* const*)(dgrad + k * n), (int32_t)n, ZS_FP16,
                                 count, acc, k == 0, 0);
    if (st != ZS_OK) fprintf(stderr, "zs_grad_accum: %s\n", zs_last_error(ctx));
    CHECK(st == ZS_OK);
  }
  int32_t ovf = -1;
  float new_scale = 0.0f;
  zs_status st;
  if (twophase) {
    /* two ranges of the last micro-step, each summed, flagged and updated into
     * the second set; the context's flag decides the commit */
    float *master2, *m2, *v2;
    uint16_t* half2;
    CHECK(cudaMalloc((void**)&master2, count * 4) == cudaSuccess);
    CHECK(cudaMalloc((void**)&m2, count * 4) == cudaSuccess);
    CHECK(cudaMalloc((void**)&v2, count * 4) == cudaSuccess);
    CHECK(cudaMalloc((void**)&half2, count * 2) == cudaSuccess);
    int32_t* d_flag = NULL;
    CHECK(zs_ctx_overflow_flag(ctx, &d_flag) == ZS_OK);
    const int64_t cut = count / 2 / 64 * 64;
    const float div = (float)n * (float)g * sc.scale;
    st = ZS_OK;
    for (int part = 0; part < 2 && st == ZS_OK; ++part) {
      const int64_t lo = part ? cut : 0, len = part ? count - cut : cut;
      const void* rows[256];
      for (int64_t r = 0; r < n; ++r) rows[r] = (const uint16_t*)dgrad[(g - 1) * n + r] + lo;
      st = zs_update_oop(ctx, rows, (int32_t)n, ZS_FP16, len, g > 1 ? acc + lo : NULL, div,
                         master + lo, m + lo, v + lo, master2 + lo, m2 + lo, v2 + lo, half2 + lo,
                         &hp, 1, d_flag, 0);
    }
    if (st == ZS_OK) st = zs_scaler_update(ctx, d_flag, &sc, &ovf, 0);
    new_scale = sc.scale;
    if (st == ZS_OK && ovf == 0) {
      master = master2;
      m = m2;
      v = v2;
      half = half2;
    }
  } else if (!oop) {
    st = zs_shard_step(ctx, (const void* const*)(dgrad + (g - 1) * n), (int32_t)n, ZS_FP16, count,
                       acc, (int32_t)g, master, m, v, half, &hp, 1, &sc, &ovf, &new_scale, 0);
  } else {
    float *master2, *m2, *v2;
    void* half2;
    CHECK(cudaMalloc((void**)&master2, count * 4) == cudaSuccess);
    CHECK(cudaMalloc((void**)&m2, count * 4) == cudaSuccess);
    CHECK(cudaMalloc((void**)&v2, count * 4) == cudaSuccess);
    CHECK(cudaMalloc(&half2, count * 2) == cudaSuccess);
    st = zs_shard_step_oop(ctx, (const void* const*)(dgrad + (g - 1) * n), (int32_t)n, ZS_FP16,
                           count, acc, (int32_t)g, master, m, v, master2, m2, v2, half2, &hp, 1,
                           &sc, &ovf, &new_scale, 0);
    if (st == ZS_OK && ovf == 0) { /* the written set is now the state */
      master = master2;
      m = m2;
      v = v2;
      half = half2;
    }
  }
  if (st != ZS_OK) fprintf(stderr, "step: %s\n", zs_last_error(ctx));
  CHECK(st == ZS_OK);

  float* out = (float*)malloc(count * 4);
  uint16_t* outh = (uint16_t*)malloc(count * 2);
  FILE* o = fopen(argv[2], "wb");
  CHECK(o != NULL && out && outh);
  fwrite(&ovf, 4, 1, o);
  fwrite(&new_scale, 4, 1, o);
  float* srcs[3] = {master, m, v};
  for (int k = 0; k < 3; ++k) {
    CHECK(cudaMemcpy(out, srcs[k], count * 4, cudaMemcpyDeviceToHost) == cudaSuccess);
    fwrite(out, 4, count, o);
  }
  CHECK(cudaMemcpy(outh, half, count * 2, cudaMemcpyDeviceToHost) == cudaSuccess);
  fwrite(outh, 2, count, o);
  fclose(o);
  CHECK(zs_ctx_destroy(ctx) == ZS_OK);
  return 0;
}
