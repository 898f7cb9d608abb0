/*
 * Device side of the seeded synthetic-input generator (see zs_synth.h): fills
 * HBM buffers with the same values the host side computes, converted to
 * fp16/bf16 with CUDA's round-to-nearest-even intrinsics.  Used by tests and
 * the benchmark to build inputs; never part of a timed step.
 */
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include "zs_synth.h"

namespace {

__global__ void fill_grads_kernel(uint16_t* out, int dtype, int64_t count, int64_t global_begin,
                                  int64_t psi, uint32_t step, uint32_t micro, uint32_t rank,
                                  zs_synth_grad_recipe r) {
  int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < count; j += stride) {
    int64_t i = global_begin + j;
    float x = (i < psi) ? zs_synth_grad_value(&r, (uint64_t)i, step, micro, rank) : 0.0f;
    uint16_t bits;
    if (dtype == 0) {
      bits = __half_as_ushort(__float2half_rn(x));
    } else {
      bits = __bfloat16_as_ushort(__float2bfloat16_rn(x));
    }
    out[j] = bits;
  }
}

__global__ void fill_master_kernel(float* out, int64_t count, int64_t global_begin, int64_t psi,
                                   uint64_t seed, uint64_t stream, float c) {
  int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < count; j += stride) {
    int64_t i = global_begin + j;
    out[j] = (i < psi) ? zs_synth_master_value(seed, stream, c, (uint64_t)i) : 0.0f;
  }
}

int grid_for(int64_t count) {
  int64_t blocks = (count + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (blocks < 1) blocks = 1;
  return (int)blocks;
}

}  // namespace

extern "C" int zs_synth_dev_fill_grads(void* out, int dtype, int64_t count, int64_t global_begin,
                                       int64_t psi, uint32_t step, uint32_t micro, uint32_t rank,
                                       const zs_synth_grad_recipe* r, cudaStream_t s) {
  if (count < 0 || (count > 0 && out == nullptr) || r == nullptr || (dtype != 0 && dtype != 1))
    return -1;
  if (count == 0) return 0;
  fill_grads_kernel<<<grid_for(count), 256, 0, s>>>((uint16_t*)out, dtype, count, global_begin,
                                                      psi, step, micro, rank, *r);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

extern "C" int zs_synth_dev_fill_master(float* out, int64_t count, int64_t global_begin,
                                        int64_t psi, uint64_t seed, uint64_t stream, float c,
                                        cudaStream_t s) {
  if (count < 0 || (count > 0 && out == nullptr)) return -1;
  if (count == 0) return 0;
  fill_master_kernel<<<grid_for(count), 256, 0, s>>>(out, count, global_begin, psi, seed, stream,
                                                       c);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}
