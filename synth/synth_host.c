/*
 * Host side of the seeded synthetic-input generator (see zs_synth.h).
 * Gather form: values at an arbitrary list of flat indices, so the CPU oracle
 * can be fed either a contiguous range or a sample of a full-size workload.
 * Indices at or beyond psi (alignment padding) yield 0.
 * Build: gcc -O2 -ffp-contract=off -fPIC -shared.
 */
#include "zs_synth.h"

void zs_synth_host_grad_values(const int64_t* idx, int64_t k, int64_t psi, uint32_t step,
                               uint32_t micro, uint32_t rank, const zs_synth_grad_recipe* r,
                               float* out) {
  for (int64_t j = 0; j < k; ++j) {
    int64_t i = idx[j];
    out[j] = (i >= 0 && i < psi) ? zs_synth_grad_value(r, (uint64_t)i, step, micro, rank) : 0.0f;
  }
}

void zs_synth_host_master_values(const int64_t* idx, int64_t k, int64_t psi, uint64_t seed,
                                 uint64_t stream, float c, float* out) {
  for (int64_t j = 0; j < k; ++j) {
    int64_t i = idx[j];
    out[j] = (i >= 0 && i < psi) ? zs_synth_master_value(seed, stream, c, (uint64_t)i) : 0.0f;
  }
}

void zs_synth_host_philox(const uint64_t* ctr, const uint64_t* key, uint64_t* out) {
  zs_synth_philox4x64_10(ctr, key, out);
}
