// C ABI of the ZeRO shard step (declarations and contracts in zeroshard.h):
// argument checks, launch shapes, the per-step host/device handshake and the
// optional per-kernel event timing.  Every step of the arithmetic runs in
// the kernels of zs_kernels.cuh.
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <unordered_map>
#include <utility>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "zeroshard.h"
#include "zs_kernels.cuh"

// Capacity of the per-CTA partial sums of the clipping norm (one double each).
#define ZS_SUMSQ_MAX_PARTS 4096
// Capacity of the per-CTA norm partials of the fused last-micro-step pass,
// allocated with the context (8 MB): one CTA per 2048 elements covers 2^31
// elements; larger calls cap the grid here and each thread takes several
// vector units (the pass is grid-stride), so no call allocates.
#define ZS_NORM_MAX_PARTS (1 << 20)
// The half-accumulator reduce prefetches ahead into L2 for at most this many ranks.
#ifndef ZS_HACC_PREFETCH_MAX_N
#define ZS_HACC_PREFETCH_MAX_N 2
#endif
// Accumulators up to this size keep an evict-last L2 policy (they are read
// back by the next micro-step and by the update; L2 is 129 MB on GB300).
#ifndef ZS_ACC_KEEP_MAX_BYTES
#define ZS_ACC_KEEP_MAX_BYTES (64ll << 20)
#endif

// How long a CTA of the fused step waits at its grid barrier before it gives
// up (the wait normally lasts microseconds: every CTA is co-resident).
#define ZS_DEFAULT_WAIT_NS 1000000000ull

static inline uint32_t acc_keep_for(int64_t count) {
  return count * 4 <= ZS_ACC_KEEP_MAX_BYTES ? 1u : 0u;
}

struct zs_ctx {
  int device = 0;
  int sms = 0;
  int32_t* d_flag = nullptr;          // the step's overflow flag
  double* d_partials = nullptr;        // scratch: per-CTA sums of squares
  double* d_sumsq = nullptr;           // the step's squared gradient norm (zs_shard_step_clipped)
  float* d_coef = nullptr;             // scratch: clipping coefficient
  zs::AdamArgs* d_args = nullptr;      // scratch: per-step constants of the async step
  double* d_norm_parts = nullptr;      // scratch: ZS_NORM_MAX_PARTS per-CTA norm partials
  double* h_sumsq = nullptr;           // pinned mirror of d_sumsq
  // the step's result, written by the loss-scale update straight into mapped
  // pinned host memory (d_result is the device's address of h_result), so the
  // synchronising calls read it after the stream sync without a copy
  zs::StepResult* d_result = nullptr;
  zs::StepResult* h_result = nullptr;
  // the fused step: its grid barrier, and a mapped pinned word that a fused
  // step whose bounded wait ran out sets (d_fused_err is its device address)
  zs::FusedSync* d_sync = nullptr;
  int32_t* h_fused_err = nullptr;
  int32_t* d_fused_err = nullptr;
  int32_t fused_mode = ZS_FUSED_ON;
  uint64_t wait_ns = ZS_DEFAULT_WAIT_NS;
  int64_t coop_max_grid = INT64_MAX;  // lowered when the runtime refuses a cooperative grid
  std::string err;
  std::unordered_map<const void*, int> occupancy;  // resident CTAs per SM, per kernel
  int64_t launches = 0;
  bool pdl = true;  // launch the step's kernels as programmatic dependents
  bool coop_pdl = true;  // the fused step's cooperative launch too (off once refused)
  // timing
  bool timing = false;
  struct Rec {
    int kind;
    cudaEvent_t start, stop;
    int64_t elements;
  };
  std::vector<Rec> pending;
  std::vector<cudaEvent_t> pool;
  double total_ms[ZS_KERNEL_KINDS] = {};
  int64_t total_launches[ZS_KERNEL_KINDS] = {};
  int64_t total_elements[ZS_KERNEL_KINDS] = {};
};

namespace {

// NVTX range around each entry point (visible to ncu/nsys; a no-op otherwise).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};

zs_status fail(zs_ctx* c, zs_status code, const char* fmt, ...) {
  if (c != nullptr) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    c->err = buf;
  }
  return code;
}

zs_status cuda_fail(zs_ctx* c, cudaError_t e, const char* what) {
  return fail(c, ZS_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

cudaEvent_t take_event(zs_ctx* c) {
  if (!c->pool.empty()) {
    cudaEvent_t e = c->pool.back();
    c->pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// Folds finished timing records into the totals without blocking, so a
// context that keeps timing on for a long run holds a bounded set of events.
void fold_finished(zs_ctx* c) {
  size_t keep = 0;
  for (size_t i = 0; i < c->pending.size(); ++i) {
    auto& r = c->pending[i];
    float ms = 0.0f;
    if (cudaEventQuery(r.stop) == cudaSuccess &&
        cudaEventElapsedTime(&ms, r.start, r.stop) == cudaSuccess) {
      c->total_ms[r.kind] += ms;
      c->total_launches[r.kind] += 1;
      c->total_elements[r.kind] += r.elements;
      c->pool.push_back(r.start);
      c->pool.push_back(r.stop);
    } else {
      c->pending[keep++] = r;
    }
  }
  c->pending.resize(keep);
}

// Whether `s` is capturing into a graph (also when the query itself fails,
// e.g. on the legacy stream while another stream captures).
bool stream_capturing(cudaStream_t s) {
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) {
    (void)cudaGetLastError();
    return true;
  }
  return cap != cudaStreamCaptureStatusNone;
}

// Bracket one launch with events when timing is on -- never on a capturing
// stream: an event recorded into a graph would be timed once per capture, not
// per replay, and could not be waited on once the graph is gone.
struct LaunchScope {
  zs_ctx* c;
  cudaStream_t s;
  int kind;
  int64_t elements;
  cudaEvent_t start = nullptr;
  LaunchScope(zs_ctx* c_, cudaStream_t s_, int kind_, int64_t el)
      : c(c_), s(s_), kind(kind_), elements(el) {
    if (c->timing && !stream_capturing(s)) {
      start = take_event(c);
      if (start) cudaEventRecord(start, s);
    }
  }
  // the launch did not happen: hand the start event back
  void cancel() {
    if (start) c->pool.push_back(start);
    start = nullptr;
  }
  void done() {
    c->launches += 1;
    if (c->timing && start) {
      cudaEvent_t stop = take_event(c);
      if (stop) {
        cudaEventRecord(stop, s);
        c->pending.push_back({kind, start, stop, elements});
        if (c->pending.size() >= 1024) fold_finished(c);
      } else {
        c->pool.push_back(start);
      }
    }
  }
};

// Launch one of the step's kernels on `s`.  With c->pdl the launch allows
// programmatic dependent launch: the kernel's CTAs may be scheduled while the
// previous kernel in the stream is finishing, and each kernel waits
// (griddepcontrol.wait, its first instruction) until its predecessor has
// completed and its writes are visible.  This removes the launch gap between
// the short kernels of a step.
template <typename... KArgs, typename... Args>
void launch_k(zs_ctx* c, void (*kernel)(KArgs...), int grid, int block, cudaStream_t s,
              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)block);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = c->pdl ? 1 : 0;
  (void)cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Resident CTAs per SM of `kernel` at kThreads threads (cached per kernel).
template <typename K>
int resident_ctas(zs_ctx* c, K kernel) {
  const void* key = reinterpret_cast<const void*>(kernel);
  auto it = c->occupancy.find(key);
  if (it != c->occupancy.end()) return it->second;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, zs::kThreads, 0) !=
          cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  c->occupancy.emplace(key, per_sm);
  return per_sm;
}

template <typename K>
int grid_for(zs_ctx* c, K kernel, int64_t items, int waves = ZS_GRID_WAVES) {
  const int per_sm = resident_ctas(c, kernel);
  int64_t need = (items + zs::kThreads - 1) / zs::kThreads;
  if (need < 1) need = 1;
  if (waves > 0) {
    const int64_t cap = (int64_t)per_sm * c->sms * waves;
    if (need > cap) need = cap;
  }
  if (need > 0x7fffffff) need = 0x7fffffff;
  return (int)need;
}

// A fused step of this context gave up its bounded grid wait: that step's
// state is undefined.  Once the device is idle the barrier and the step's flag
// are reset, so the context stays usable; the call reports ZS_ERR_TIMEOUT.
zs_status fused_timeout(zs_ctx* c) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemset(c->d_sync, 0, sizeof(zs::FusedSync));
  if (e == cudaSuccess) e = cudaMemset(c->d_flag, 0, sizeof(int32_t));
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  *reinterpret_cast<volatile int32_t*>(c->h_fused_err) = 0;
  if (e != cudaSuccess) return cuda_fail(c, e, "reset after a fused-step timeout");
  return fail(c, ZS_ERR_TIMEOUT,
              "a fused step's grid barrier wait ran out (limit %llu ns): that step wrote at most "
              "part of the state; the barrier and the flag have been reset",
              (unsigned long long)c->wait_ns);
}

bool fused_timed_out(const zs_ctx* c) {
  return c->h_fused_err != nullptr && *reinterpret_cast<volatile int32_t*>(c->h_fused_err) != 0;
}

zs_status check_ctx(zs_ctx* c) {
  if (c == nullptr) return ZS_ERR_ARG;
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(c, e, "cudaGetDevice");
  if (dev != c->device)
    return fail(c, ZS_ERR_ARG, "current device %d is not the context's device %d", dev,
                c->device);
  c->err.clear();
  if (fused_timed_out(c)) return fused_timeout(c);
  return ZS_OK;
}

zs_status check_slices(zs_ctx* c, const void* const* grads, int32_t n, int64_t count,
                       zs::SlicePtrs* out) {
  if (n < 1 || n > ZS_MAX_RANKS)
    return fail(c, ZS_ERR_ARG, "n = %d is outside [1, %d]", n, ZS_MAX_RANKS);
  if (grads == nullptr) return fail(c, ZS_ERR_ARG, "grads is NULL");
  std::memset(out, 0, sizeof(*out));
  for (int r = 0; r < n; ++r) {
    if (count > 0 && grads[r] == nullptr) return fail(c, ZS_ERR_ARG, "grads[%d] is NULL", r);
    if (!aligned16(grads[r]))
      return fail(c, ZS_ERR_ALIGN, "grads[%d] is not 16-byte aligned", r);
    out->p[r] = static_cast<const uint4*>(grads[r]);
  }
  return ZS_OK;
}

zs_status check_array(zs_ctx* c, const void* p, const char* name, int64_t count) {
  if (count > 0 && p == nullptr) return fail(c, ZS_ERR_ARG, "%s is NULL", name);
  if (!aligned16(p)) return fail(c, ZS_ERR_ALIGN, "%s is not 16-byte aligned", name);
  return ZS_OK;
}

#define ZS_TRY(x)                       \
  do {                                  \
    zs_status st_ = (x);                \
    if (st_ != ZS_OK) return st_;       \
  } while (0)

int vpt_for(int32_t n) {
  if (n <= 2) return ZS_VPT_SMALL_N;
  if (n <= 8) return ZS_VPT_MID_N;
  return 1;
}

template <int DT, bool RA, bool ST, int VPT>
void launch_reduce_k(zs_ctx* c, const zs::SlicePtrs& sp, int32_t n, float* acc, int64_t count,
                     int32_t* flag, cudaStream_t s) {
  const int64_t units = (count >> 3) / VPT + 8;
  auto k = zs::k_reduce<DT, RA, ST, VPT>;
  const int waves = ST ? ZS_GRID_WAVES : ZS_CHECK_WAVES;
  launch_k(c, k, grid_for(c, k, units, waves), zs::kThreads, s, sp, n, acc, count, flag,
           (double*)nullptr, acc_keep_for(count), 0);
}

// The last micro-step's pass with the clipping norm fused in: per-CTA sums of
// squares of the final sums into the context's partials (a fixed capacity:
// the grid is capped there, and the pass strides over the rest).
template <int DT, bool RA, bool ST>
zs_status launch_reduce_norm_k(zs_ctx* c, const zs::SlicePtrs& sp, int32_t n, float* acc,
                               int64_t count, int32_t* flag, int* nparts, cudaStream_t s) {
  constexpr int VPT = ZS_NORM_VPT;
  auto k = zs::k_reduce<DT, RA, ST, VPT, false, true>;
  int grid = grid_for(c, k, (count >> 3) / VPT + 8, ZS_GRID_WAVES);
  if (grid > ZS_NORM_MAX_PARTS) grid = ZS_NORM_MAX_PARTS;
  launch_k(c, k, grid, zs::kThreads, s, sp, n, acc, count, flag, c->d_norm_parts,
           acc_keep_for(count), 0);
  *nparts = grid;
  return ZS_OK;
}

zs_status reduce_norm_any(zs_ctx* c, zs_dtype dt, const zs::SlicePtrs& sp, int32_t n, float* acc,
                          int64_t count, bool read_acc, bool store, int32_t* flag, float grad_div,
                          double* out, cudaStream_t s) {
  const int kind = store ? (read_acc ? ZS_KERNEL_REDUCE : ZS_KERNEL_REDUCE_FIRST)
                         : ZS_KERNEL_CHECK;
  LaunchScope ls(c, s, kind, count);
  int nparts = 0;
  zs_status st;
  if (dt == ZS_FP16) {
    if (store && read_acc) st = launch_reduce_norm_k<ZS_FP16, true, true>(c, sp, n, acc, count, flag, &nparts, s);
    else if (store) st = launch_reduce_norm_k<ZS_FP16, false, true>(c, sp, n, acc, count, flag, &nparts, s);
    else if (read_acc) st = launch_reduce_norm_k<ZS_FP16, true, false>(c, sp, n, acc, count, flag, &nparts, s);
    else st = launch_reduce_norm_k<ZS_FP16, false, false>(c, sp, n, acc, count, flag, &nparts, s);
  } else {
    if (store && read_acc) st = launch_reduce_norm_k<ZS_BF16, true, true>(c, sp, n, acc, count, flag, &nparts, s);
    else if (store) st = launch_reduce_norm_k<ZS_BF16, false, true>(c, sp, n, acc, count, flag, &nparts, s);
    else if (read_acc) st = launch_reduce_norm_k<ZS_BF16, true, false>(c, sp, n, acc, count, flag, &nparts, s);
    else st = launch_reduce_norm_k<ZS_BF16, false, false>(c, sp, n, acc, count, flag, &nparts, s);
  }
  if (st != ZS_OK) return st;
  const double div = (double)grad_div;
  const double* parts = c->d_norm_parts;
  if (nparts > ZS_SUMSQ_MAX_PARTS) {
    // one partial per CTA of a full grid can be millions: fold them into at
    // most ZS_SUMSQ_MAX_PARTS chunk sums first (fixed order, deterministic)
    const int64_t chunk = (nparts + ZS_SUMSQ_MAX_PARTS - 1) / ZS_SUMSQ_MAX_PARTS;
    const int blocks = (int)((nparts + chunk - 1) / chunk);
    launch_k(c, zs::k_partials_reduce, blocks, zs::kThreads, s,
             (const double*)c->d_norm_parts, (int64_t)nparts, chunk, c->d_partials);
    c->launches += 1;
    parts = c->d_partials;
    nparts = blocks;
  }
  launch_k(c, zs::k_sumsq_finalize, 1, zs::kThreads, s, parts, nparts, 1.0 / (div * div), out);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(c, e, "reduce launch");
  ls.done();
  c->launches += 1;  // the finalize kernel
  return ZS_OK;
}

template <int DT, bool RA, bool ST>
void launch_reduce_v(zs_ctx* c, const zs::SlicePtrs& sp, int32_t n, float* acc, int64_t count,
                     int32_t* flag, cudaStream_t s) {
  const int vpt = (!ST && n <= 2)  ? ZS_CHECK_VPT
                  : (!RA && n <= 2) ? ZS_VPT_FIRST_SMALL_N
                                    : vpt_for(n);
  switch (vpt) {
    case 8: launch_reduce_k<DT, RA, ST, 8>(c, sp, n, acc, count, flag, s); break;
    case 4: launch_reduce_k<DT, RA, ST, 4>(c, sp, n, acc, count, flag, s); break;
    case 2: launch_reduce_k<DT, RA, ST, 2>(c, sp, n, acc, count, flag, s); break;
    default: launch_reduce_k<DT, RA, ST, 1>(c, sp, n, acc, count, flag, s); break;
  }
}

template <int DT>
zs_status launch_reduce(zs_ctx* c, const zs::SlicePtrs& sp, int32_t n, float* acc, int64_t count,
                        bool read_acc, bool store, int32_t* flag, cudaStream_t s) {
  const int kind = store ? (read_acc ? ZS_KERNEL_REDUCE : ZS_KERNEL_REDUCE_FIRST)
                         : ZS_KERNEL_CHECK;
  LaunchScope ls(c, s, kind, count);
  if (!store && !read_acc && (DT == ZS_FP16 || n == 1)) {
    // flag only, from the raw bit patterns (exact here: see k_check_bits)
    constexpr int VPT = ZS_CHECK_VPT;
    auto k = zs::k_check_bits<DT, VPT>;
    launch_k(c, k, grid_for(c, k, (count >> 3) / VPT + 8, ZS_CHECK_WAVES), zs::kThreads, s, sp,
             n, count, flag);
  } else if (read_acc && store) {
    launch_reduce_v<DT, true, true>(c, sp, n, acc, count, flag, s);
  } else if (store) {
    launch_reduce_v<DT, false, true>(c, sp, n, acc, count, flag, s);
  } else if (read_acc) {
    launch_reduce_v<DT, true, false>(c, sp, n, acc, count, flag, s);
  } else {
    launch_reduce_v<DT, false, false>(c, sp, n, acc, count, flag, s);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(c, e, "reduce launch");
  ls.done();
  return ZS_OK;
}

zs_status reduce_any(zs_ctx* c, zs_dtype dt, const zs::SlicePtrs& sp, int32_t n, float* acc,
                     int64_t count, bool read_acc, bool store, int32_t* flag, cudaStream_t s) {
  if (dt == ZS_FP16) return launch_reduce<ZS_FP16>(c, sp, n, acc, count, read_acc, store, flag, s);
  return launch_reduce<ZS_BF16>(c, sp, n, acc, count, read_acc, store, flag, s);
}

zs::AdamArgs adam_args(const zs_adam_hparams* hp, int64_t step, float grad_div) {
  return zs::make_adam_args(hp->lr, *hp, step, grad_div);
}

template <int DT, bool HA, bool RC>
void launch_apply_k(zs_ctx* c, const int32_t* flag, const zs::SlicePtrs& sp, int32_t n,
                    const float* acc, int64_t count, const zs::AdamArgs& ad, float* master,
                    float* m, float* v, uint16_t* ho, const zs_scaler& sc_in,
                    zs::StepResult* result, const float* coef, cudaStream_t s) {
  constexpr int VPT = ZS_APPLY_VPT;
  const int64_t units = (count >> 3) / VPT + 8;
  if (coef != nullptr) {
    auto k = zs::k_apply<DT, HA, RC, VPT, true>;
    launch_k(c, k, grid_for(c, k, units), zs::kThreads, s, flag, sp, n, acc, master, m, v, ho,
             count, ad, sc_in, result, coef, (const zs::AdamArgs*)nullptr,
             (zs_device_state*)nullptr, acc_keep_for(count));
  } else {
    auto k = zs::k_apply<DT, HA, RC, VPT, false>;
    launch_k(c, k, grid_for(c, k, units), zs::kThreads, s, flag, sp, n, acc, master, m, v, ho,
             count, ad, sc_in, result, (const float*)nullptr, (const zs::AdamArgs*)nullptr,
             (zs_device_state*)nullptr, acc_keep_for(count));
  }
}

template <int DT>
zs_status launch_apply(zs_ctx* c, const int32_t* flag, const zs::SlicePtrs& sp, int32_t n,
                       bool recompute, const float* acc, int64_t count, const zs::AdamArgs& ad,
                       float* master, float* m, float* v, void* half_out,
                       const zs_scaler* scaler_in, zs::StepResult* result, const float* coef,
                       cudaStream_t s) {
  zs_scaler sc_in{};
  if (scaler_in) sc_in = *scaler_in;
  uint16_t* ho = static_cast<uint16_t*>(half_out);
  LaunchScope ls(c, s, recompute ? ZS_KERNEL_APPLY_RECOMPUTE : ZS_KERNEL_APPLY, count);
  if (!recompute) {
    launch_apply_k<DT, true, false>(c, flag, sp, n, acc, count, ad, master, m, v, ho, sc_in,
                                    result, coef, s);
  } else if (acc != nullptr) {
    launch_apply_k<DT, true, true>(c, flag, sp, n, acc, count, ad, master, m, v, ho, sc_in,
                                   result, coef, s);
  } else {
    launch_apply_k<DT, false, true>(c, flag, sp, n, acc, count, ad, master, m, v, ho, sc_in,
                                    result, coef, s);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(c, e, "apply launch");
  ls.done();
  return ZS_OK;
}

zs_status apply_any(zs_ctx* c, zs_dtype dt, const int32_t* flag, const zs::SlicePtrs& sp,
                    int32_t n, bool recompute, const float* acc, int64_t count,
                    const zs::AdamArgs& ad, float* master, float* m, float* v, void* half_out,
                    const zs_scaler* scaler_in, zs::StepResult* result, cudaStream_t s,
                    const float* coef = nullptr) {
  if (dt == ZS_FP16)
    return launch_apply<ZS_FP16>(c, flag, sp, n, recompute, acc, count, ad, master, m, v,
                                 half_out, scaler_in, result, coef, s);
  return launch_apply<ZS_BF16>(c, flag, sp, n, recompute, acc, count, ad, master, m, v, half_out,
                               scaler_in, result, coef, s);
}

// Sum of squares of the final gradient sums of a range, then / grad_div^2,
// into *out (device).  Grid capped at ZS_SUMSQ_MAX_PARTS CTAs (one partial each).
template <int DT, bool HA, bool RC>
void launch_sumsq_k(zs_ctx* c, const zs::SlicePtrs& sp, int32_t n, const float* acc,
                    int64_t count, double* partials, int* nparts, cudaStream_t s) {
  auto k = zs::k_sumsq<DT, HA, RC>;
  int grid = grid_for(c, k, (count >> 3) + 8, 1);
  if (grid > ZS_SUMSQ_MAX_PARTS) grid = ZS_SUMSQ_MAX_PARTS;
  *nparts = grid;
  launch_k(c, k, grid, zs::kThreads, s, sp, n, acc, count, partials);
}

zs_status sumsq_any(zs_ctx* c, zs_dtype dt, const zs::SlicePtrs& sp, int32_t n, bool recompute,
                    const float* acc, int64_t count, float grad_div, double* partials,
                    double* out, cudaStream_t s) {
  LaunchScope ls(c, s, ZS_KERNEL_SUMSQ, count);
  int nparts = 0;
  const bool ha = acc != nullptr;
  if (dt == ZS_FP16) {
    if (recompute && ha) launch_sumsq_k<ZS_FP16, true, true>(c, sp, n, acc, count, partials, &nparts, s);
    else if (recompute) launch_sumsq_k<ZS_FP16, false, true>(c, sp, n, acc, count, partials, &nparts, s);
    else launch_sumsq_k<ZS_FP16, true, false>(c, sp, n, acc, count, partials, &nparts, s);
  } else {
    if (recompute && ha) launch_sumsq_k<ZS_BF16, true, true>(c, sp, n, acc, count, partials, &nparts, s);
    else if (recompute) launch_sumsq_k<ZS_BF16, false, true>(c, sp, n, acc, count, partials, &nparts, s);
    else launch_sumsq_k<ZS_BF16, true, false>(c, sp, n, acc, count, partials, &nparts, s);
  }
  const double div = (double)grad_div;
  launch_k(c, zs::k_sumsq_finalize, 1, zs::kThreads, s, (const double*)partials, nparts,
           1.0 / (div * div), out);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(c, e, "sumsq launch");
  ls.done();
  c->launches += 1;  // the finalize kernel
  return ZS_OK;
}

zs_status clip_coef_launch(zs_ctx* c, const double* d_sumsq, float max_norm, cudaStream_t s) {
  launch_k(c, zs::k_clip_coef, 1, 32, s, d_sumsq, max_norm, c->d_coef);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(c, e, "clip coefficient launch");
  c->launches += 1;
  return ZS_OK;
}

zs_status check_hparams(zs_ctx* c, const zs_adam_hparams* hp, int64_t step) {
  if (hp == nullptr) return fail(c, ZS_ERR_ARG, "hparams is NULL");
  if (step < 1) return fail(c, ZS_ERR_ARG, "step must be >= 1 (got %lld)", (long long)step);
  if (!(hp->beta1 >= 0.0f && hp->beta1 < 1.0f) || !(hp->beta2 >= 0.0f && hp->beta2 < 1.0f))
    return fail(c, ZS_ERR_ARG, "betas must lie in [0, 1)");
  if (!(hp->eps > 0.0f) || !std::isfinite(hp->lr) || !std::isfinite(hp->weight_decay))
    return fail(c, ZS_ERR_ARG, "eps must be > 0 and lr, weight_decay finite");
  return ZS_OK;
}

zs_status check_scaler(zs_ctx* c, const zs_scaler* s) {
  if (s == nullptr) return fail(c, ZS_ERR_ARG, "scaler is NULL");
  if (!(s->scale > 0.0f) || !std::isfinite(s->scale) || !(s->min_scale > 0.0f) ||
      s->window < 1 || s->hysteresis < 1)
    return fail(c, ZS_ERR_ARG, "scaler needs scale > 0, min_scale > 0, window >= 1, hysteresis >= 1");
  return ZS_OK;
}

zs_status finish_step(zs_ctx* c, zs_scaler* scaler, int32_t* overflow_out, float* new_scale_out,
                      int32_t* flag_to_clear, cudaStream_t s) {
  cudaError_t e = cudaSuccess;
  if (flag_to_clear) {
    launch_k(c, zs::k_clear_flag, 1, 32, s, flag_to_clear);
    c->launches += 1;
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(c, e, "flag reset");
  }
  e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(c, e, "step synchronisation");
  *scaler = c->h_result->scaler;
  if (overflow_out) *overflow_out = c->h_result->overflow;
  if (new_scale_out) *new_scale_out = c->h_result->scaler.scale;
  return ZS_OK;
}

// finish_step after a fused step: its bounded wait may have run out, in
// which case the loss-scale result was not written.
zs_status finish_fused_step(zs_ctx* c, zs_scaler* scaler, int32_t* overflow_out,
                            float* new_scale_out, cudaStream_t s) {
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(c, e, "step synchronisation");
  if (fused_timed_out(c)) return fused_timeout(c);
  return finish_step(c, scaler, overflow_out, new_scale_out, nullptr, s);
}

template <int DT, bool HA, bool RC, bool CLIP>
void launch_apply_dev_k(zs_ctx* c, const int32_t* flag, const zs::SlicePtrs& sp, int32_t n,
                        const float* acc, int64_t count, float* master, float* m, float* v,
                        uint16_t* ho, const zs::AdamArgs* ad_dev, zs_device_state* st,
                        const float* coef, cudaStream_t s) {
  constexpr int VPT = ZS_APPLY_VPT;
  const int64_t units = (count >> 3) / VPT + 8;
  auto k = zs::k_apply<DT, HA, RC, VPT, CLIP, true>;
  const zs::AdamArgs unused{};
  const zs_scaler unused_sc{};
  launch_k(c, k, grid_for(c, k, units), zs::kThreads, s, flag, sp, n, acc, master, m, v, ho,
           count, unused, unused_sc, (zs::StepResult*)nullptr, coef, ad_dev, st,
           acc_keep_for(count));
}

template <int DT, bool CLIP>
void apply_dev_c(zs_ctx* c, const int32_t* flag, const zs::SlicePtrs& sp, int32_t n,
                 bool recompute, const float* acc, int64_t count, float* master, float* m,
                 float* v, uint16_t* ho, const zs::AdamArgs* ad_dev, zs_device_state* st,
                 const float* coef, cudaStream_t s) {
  if (!recompute)
    launch_apply_dev_k<DT, true, false, CLIP>(c, flag, sp, n, acc, count, master, m, v, ho,
                                              ad_dev, st, coef, s);
  else if (acc != nullptr)
    launch_apply_dev_k<DT, true, true, CLIP>(c, flag, sp, n, acc, count, master, m, v, ho,
                                             ad_dev, st, coef, s);
  else
    launch_apply_dev_k<DT, false, true, CLIP>(c, flag, sp, n, acc, count, master, m, v, ho,
                                              ad_dev, st, coef, s);
}

// The device-resident update (clipped with the context's coefficient when coef != NULL).
template <int DT>
void apply_dev(zs_ctx* c, const int32_t* flag, const zs::SlicePtrs& sp, int32_t n,
               bool recompute, const float* acc, int64_t count, float* master, float* m,
               float* v, uint16_t* ho, const zs::AdamArgs* ad_dev, zs_device_state* st,
               const float* coef, cudaStream_t s) {
  if (coef != nullptr)
    apply_dev_c<DT, true>(c, flag, sp, n, recompute, acc, count, master, m, v, ho, ad_dev, st,
                          coef, s);
  else
    apply_dev_c<DT, false>(c, flag, sp, n, recompute, acc, count, master, m, v, ho, ad_dev, st,
                           nullptr, s);
}

// Out-of-place step: the update kernel and its commit.
template <int DT, bool HA, bool DEV, bool HACC = false>
void launch_oop_k(zs_ctx* c, const zs::SlicePtrs& sp, int32_t n, const float* acc,
                  const zs::OopBufs& b, int64_t count, const zs::AdamArgs& ad,
                  const zs::AdamArgs* ad_dev, const zs_device_state* st, int32_t* flag,
                  cudaStream_t s) {
  auto k = zs::k_update_oop<DT, HA, DEV, HACC>;
  launch_k(c, k, grid_for(c, k, (count >> 3) + 8), zs::kThreads, s, sp, n, acc, b, count, ad,
           ad_dev, st, flag, acc_keep_for(count));
}

template <bool DEV>
zs_status update_oop(zs_ctx* c, zs_dtype dt, const zs::SlicePtrs& sp, int32_t n,
                     const float* acc, const zs::OopBufs& b, int64_t count,
                     const zs::AdamArgs& ad, const zs::AdamArgs* ad_dev,
                     const zs_device_state* st, cudaStream_t s, int32_t* flag = nullptr) {
  if (flag == nullptr) flag = c->d_flag;
  LaunchScope ls(c, s, ZS_KERNEL_UPDATE_OOP, count);
  if (count > 0) {
    if (dt == ZS_FP16) {
      if (acc) launch_oop_k<ZS_FP16, true, DEV>(c, sp, n, acc, b, count, ad, ad_dev, st, flag, s);
      else launch_oop_k<ZS_FP16, false, DEV>(c, sp, n, acc, b, count, ad, ad_dev, st, flag, s);
    } else {
      if (acc) launch_oop_k<ZS_BF16, true, DEV>(c, sp, n, acc, b, count, ad, ad_dev, st, flag, s);
      else launch_oop_k<ZS_BF16, false, DEV>(c, sp, n, acc, b, count, ad, ad_dev, st, flag, s);
    }
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(c, e, "out-of-place update launch");
  if (count > 0) ls.done();
  return ZS_OK;
}

// A cooperative launch (every CTA co-resident, or the launch fails); with
// c->pdl also a programmatic dependent of its predecessor, like the step's
// other kernels, unless the driver refused that pair before.
template <typename... KArgs, typename... Args>
cudaError_t launch_coop(zs_ctx* c, void (*kernel)(KArgs...), int grid, cudaStream_t s,
                        Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)zs::kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = c->pdl && c->coop_pdl ? 2 : 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
  if (cfg.numAttrs == 2 && (e == cudaErrorNotSupported || e == cudaErrorInvalidValue)) {
    // a driver that refuses the pair of attributes: from now on a plain
    // cooperative launch (the kernel then starts once its predecessor has
    // completed; its griddepcontrol instructions do nothing)
    (void)cudaGetLastError();
    c->coop_pdl = false;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kernel, args...);
  }
  return e;
}

// The arguments of one fused step (k_step_fused) besides the kernel choice.
struct FusedCall {
  zs::SlicePtrs sp;
  int32_t n = 0;
  const float* acc = nullptr;  // the carried micro-steps' sums, or NULL (accum_steps == 1)
  zs::OopBufs b{};             // in place: both entries of each pair equal
  int64_t count = 0;
  zs::AdamArgs ad{};           // host constants (not DEV)
  zs_scaler scaler{};          // scaler before the step (not DEV)
  zs_device_state* dstate = nullptr;
  zs_adam_hparams hp{};
  zs_lr_schedule sched{};
  int32_t has_sched = 0;
  int32_t accum_steps = 1;
  float max_norm = 0.0f;       // clipping (> 0): the fused kernel forms the norm too
  double inv_div2 = 1.0;       // 1 / grad_div^2 (host constants) for the squared norm
  double* norm_out = nullptr;  // device forms: the step's norm (may be NULL)
  bool hacc = false;           // acc holds halves (the half accumulator; unclipped)
};

template <int DT, bool HA, bool DEV, bool FLIP, bool CLIP, int EPT, bool HACC = false>
int fused_launch_k(zs_ctx* c, const FusedCall& f, cudaStream_t s, cudaError_t* e) {
  auto k = zs::k_step_fused<DT, HA, DEV, FLIP, CLIP, EPT, HACC>;
  const int64_t per_grid = (int64_t)resident_ctas(c, k) * c->sms;
  int64_t grid = ((f.count / EPT) + zs::kThreads - 1) / zs::kThreads;
  if (grid < 1) grid = 1;
  // the barrier counts arrivals in 16 bits (a co-resident grid is far smaller)
  if (grid > per_grid || grid > c->coop_max_grid || grid > 0xFFFE) return 0;
  // ZS_FUSED_TEST_TIMEOUT: the barrier waits for one CTA more than the grid has
  const unsigned expect = (unsigned)grid + (c->fused_mode == ZS_FUSED_TEST_TIMEOUT ? 1u : 0u);
  LaunchScope ls(c, s, ZS_KERNEL_FUSED, f.count);
  *e = launch_coop(c, k, (int)grid, s, f.sp, f.n, f.acc, f.b, f.count, f.ad, f.scaler,
                   DEV ? (zs::StepResult*)nullptr : c->d_result, f.dstate, f.hp, f.sched,
                   f.has_sched, f.accum_steps, c->d_args, c->d_flag, c->d_sync, expect,
                   (uint64_t)c->wait_ns, c->d_fused_err, f.max_norm, f.inv_div2,
                   c->d_norm_parts, c->d_sumsq, f.norm_out);
  if (*e == cudaErrorCooperativeLaunchTooLarge) {
    // fewer SMs than the occupancy query assumed (e.g. a share of the GPU under
    // MPS): nothing was launched; the multi-kernel path takes the step
    (void)cudaGetLastError();
    ls.cancel();
    c->coop_max_grid = grid - 1;
    return 0;
  }
  if (*e == cudaSuccess) ls.done();
  else ls.cancel();
  return (int)grid;
}

// The whole last call of a step as ONE kernel where it applies (the mode is on,
// there is work, and one 8-element unit per thread fits a co-resident grid).
// Returns false to take the multi-pass path; otherwise *st is the launch's status.
template <bool DEV, bool FLIP, bool CLIP, int EPT>
int fused_dispatch(zs_ctx* c, zs_dtype dt, const FusedCall& f, cudaStream_t s, cudaError_t* e) {
  if constexpr (!CLIP) {
    if (f.hacc) {
      if (dt == ZS_FP16)
        return f.acc ? fused_launch_k<ZS_FP16, true, DEV, FLIP, false, EPT, true>(c, f, s, e)
                     : fused_launch_k<ZS_FP16, false, DEV, FLIP, false, EPT, true>(c, f, s, e);
      return f.acc ? fused_launch_k<ZS_BF16, true, DEV, FLIP, false, EPT, true>(c, f, s, e)
                   : fused_launch_k<ZS_BF16, false, DEV, FLIP, false, EPT, true>(c, f, s, e);
    }
  }
  if (dt == ZS_FP16)
    return f.acc ? fused_launch_k<ZS_FP16, true, DEV, FLIP, CLIP, EPT>(c, f, s, e)
                 : fused_launch_k<ZS_FP16, false, DEV, FLIP, CLIP, EPT>(c, f, s, e);
  return f.acc ? fused_launch_k<ZS_BF16, true, DEV, FLIP, CLIP, EPT>(c, f, s, e)
               : fused_launch_k<ZS_BF16, false, DEV, FLIP, CLIP, EPT>(c, f, s, e);
}

template <bool DEV, bool FLIP, bool CLIP = false>
bool try_fused(zs_ctx* c, zs_dtype dt, const FusedCall& f, cudaStream_t s, zs_status* st) {
  if (c->fused_mode == ZS_FUSED_OFF || f.count <= 0) return false;
  cudaError_t e = cudaSuccess;
  int grid = 0;
  // 4-element units (twice the threads, for latency) where they fit one
  // co-resident grid; else 8-element units (the clipped forms always: their
  // norm keeps the norm pass's CTA partition)
  if constexpr (!CLIP) grid = fused_dispatch<DEV, FLIP, false, 4>(c, dt, f, s, &e);
  if (grid == 0) grid = fused_dispatch<DEV, FLIP, CLIP, 8>(c, dt, f, s, &e);
  if (grid == 0) return false;
  *st = e == cudaSuccess ? ZS_OK : cuda_fail(c, e, "fused step launch");
  return true;
}

// Co-resident CTAs per SM of the fused step: the fewest over its variants.
template <bool DEV, bool FLIP, bool CLIP>
int fused_resident(zs_ctx* c) {
  int r = resident_ctas(c, zs::k_step_fused<ZS_FP16, true, DEV, FLIP, CLIP, 8>);
  r = std::min(r, resident_ctas(c, zs::k_step_fused<ZS_FP16, false, DEV, FLIP, CLIP, 8>));
  r = std::min(r, resident_ctas(c, zs::k_step_fused<ZS_BF16, true, DEV, FLIP, CLIP, 8>));
  r = std::min(r, resident_ctas(c, zs::k_step_fused<ZS_BF16, false, DEV, FLIP, CLIP, 8>));
  if constexpr (!CLIP) {  // the half-accumulator forms
    r = std::min(r, resident_ctas(c, zs::k_step_fused<ZS_FP16, true, DEV, FLIP, false, 8, true>));
    r = std::min(r, resident_ctas(c, zs::k_step_fused<ZS_BF16, true, DEV, FLIP, false, 8, true>));
  }
  return r;
}

zs::OopBufs in_place_bufs(float* master, float* m, float* v, void* half_out) {
  zs::OopBufs b;
  for (int i = 0; i < 2; ++i) {
    b.p[i] = master;
    b.m[i] = m;
    b.v[i] = v;
    b.h[i] = static_cast<uint16_t*>(half_out);
  }
  return b;
}

// [a, a + la) and [b, b + lb) share a byte.
bool overlaps(const void* a, int64_t la, const void* b, int64_t lb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return la > 0 && lb > 0 && x < y + (uintptr_t)lb && y < x + (uintptr_t)la;
}

// Half-precision accumulator variants (always materialise the sums).
template <int DT, bool RA>
void launch_reduce_hacc_k(zs_ctx* c, const zs::SlicePtrs& sp, int32_t n, float* acc,
                          int64_t count, int32_t* flag, cudaStream_t s) {
  constexpr int VPT = ZS_HACC_VPT;
  const int64_t units = (count >> 3) / VPT + 8;
  auto k = zs::k_reduce<DT, RA, true, VPT, true>;
  const int grid = grid_for(c, k, units);
  // one or two ranks: 16-32 bytes of loads per thread leave this pass latency-
  // bound, so each CTA prefetches into L2 the data of the CTA one full wave of
  // resident CTAs ahead (measured: 6470 -> 7144 GB/s on later micro-steps, 6095
  // -> 7087 on the first; with 8 or 16 ranks it only added traffic and lost)
  const int wave = c->occupancy[reinterpret_cast<const void*>(k)] * c->sms;
  const int ahead = n <= ZS_HACC_PREFETCH_MAX_N ? wave : 0;
  launch_k(c, k, grid, zs::kThreads, s, sp, n, acc, count, flag, (double*)nullptr, 0u, ahead);
}

zs_status reduce_hacc(zs_ctx* c, zs_dtype dt, const zs::SlicePtrs& sp, int32_t n, void* acc,
                      int64_t count, bool read_acc, int32_t* flag, cudaStream_t s) {
  LaunchScope ls(c, s, read_acc ? ZS_KERNEL_REDUCE : ZS_KERNEL_REDUCE_FIRST, count);
  float* a = static_cast<float*>(acc);
  if (dt == ZS_FP16) {
    if (read_acc) launch_reduce_hacc_k<ZS_FP16, true>(c, sp, n, a, count, flag, s);
    else launch_reduce_hacc_k<ZS_FP16, false>(c, sp, n, a, count, flag, s);
  } else {
    if (read_acc) launch_reduce_hacc_k<ZS_BF16, true>(c, sp, n, a, count, flag, s);
    else launch_reduce_hacc_k<ZS_BF16, false>(c, sp, n, a, count, flag, s);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(c, e, "reduce launch");
  ls.done();
  return ZS_OK;
}

template <int DT, bool DEV>
void launch_apply_hacc_k(zs_ctx* c, const int32_t* flag, const float* a, int64_t count,
                         const zs::AdamArgs& ad, float* master, float* m, float* v, uint16_t* ho,
                         const zs_scaler& sc_in, zs::StepResult* result,
                         const zs::AdamArgs* ad_dev, zs_device_state* st, cudaStream_t s) {
  zs::SlicePtrs sp;
  std::memset(&sp, 0, sizeof sp);
  auto k = zs::k_apply<DT, true, false, 1, false, DEV, true>;
  launch_k(c, k, grid_for(c, k, (count >> 3) + 8), zs::kThreads, s, flag, sp, 0, a, master, m, v,
           ho, count, ad, sc_in, result, (const float*)nullptr, ad_dev, st, 0u);
}

// The update from the half accumulator: host constants and the scale update
// into `result` (ad_dev == NULL), or the device-resident form (constants from
// ad_dev, the state in st).
zs_status apply_hacc(zs_ctx* c, zs_dtype dt, const int32_t* flag, const void* acc, int64_t count,
                     const zs::AdamArgs& ad, float* master, float* m, float* v, void* half_out,
                     const zs_scaler* scaler_in, zs::StepResult* result, cudaStream_t s,
                     const zs::AdamArgs* ad_dev = nullptr, zs_device_state* st = nullptr) {
  LaunchScope ls(c, s, ZS_KERNEL_APPLY, count);
  const float* a = static_cast<const float*>(acc);
  uint16_t* ho = static_cast<uint16_t*>(half_out);
  const zs_scaler sc_in = scaler_in ? *scaler_in : zs_scaler{};
  if (ad_dev != nullptr) {
    if (dt == ZS_FP16)
      launch_apply_hacc_k<ZS_FP16, true>(c, flag, a, count, ad, master, m, v, ho, sc_in, result,
                                         ad_dev, st, s);
    else
      launch_apply_hacc_k<ZS_BF16, true>(c, flag, a, count, ad, master, m, v, ho, sc_in, result,
                                         ad_dev, st, s);
  } else {
    if (dt == ZS_FP16)
      launch_apply_hacc_k<ZS_FP16, false>(c, flag, a, count, ad, master, m, v, ho, sc_in, result,
                                          nullptr, nullptr, s);
    else
      launch_apply_hacc_k<ZS_BF16, false>(c, flag, a, count, ad, master, m, v, ho, sc_in, result,
                                          nullptr, nullptr, s);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(c, e, "apply launch");
  ls.done();
  return ZS_OK;
}

}  // namespace

extern "C" {

zs_status zs_init_partition(int64_t psi, int32_t n, int32_t align_elems, zs_partition* out) {
  if (out == nullptr || psi < 0 || n < 1 || n > ZS_MAX_RANKS || align_elems < 1) return ZS_ERR_ARG;
  const int64_t unit = (int64_t)n * align_elems;
  if (psi > INT64_MAX - unit) return ZS_ERR_ARG;
  const int64_t psi_pad = (psi + unit - 1) / unit * unit;
  out->psi = psi;
  out->psi_pad = psi_pad;
  out->shard_len = psi_pad / n;
  out->n = n;
  out->align = align_elems;
  return ZS_OK;
}

zs_status zs_shard_range(const zs_partition* p, int32_t rank, int64_t* begin, int64_t* valid_end,
                         int64_t* padded_end) {
  if (p == nullptr || begin == nullptr || valid_end == nullptr || padded_end == nullptr ||
      rank < 0 || rank >= p->n)
    return ZS_ERR_ARG;
  const int64_t b = (int64_t)rank * p->shard_len;
  const int64_t e = b + p->shard_len;
  int64_t ve = e < p->psi ? e : p->psi;
  if (ve < b) ve = b;
  *begin = b;
  *valid_end = ve;
  *padded_end = e;
  return ZS_OK;
}

zs_status zs_model_state_bytes(const zs_partition* p, int32_t stage, uint64_t* bytes) {
  if (p == nullptr || bytes == nullptr) return ZS_ERR_ARG;
  const uint64_t P = (uint64_t)p->psi, E = (uint64_t)p->shard_len;
  const uint64_t half = 2, full = 4;  // bytes per element
  switch (stage) {
    case 0: *bytes = (half + half + 3 * full) * P; return ZS_OK;
    case 1: *bytes = (half + half) * P + 3 * full * E; return ZS_OK;
    case 2: *bytes = half * P + (half + 3 * full) * E; return ZS_OK;
    case 3: *bytes = (half + half + 3 * full) * E; return ZS_OK;
    default: return ZS_ERR_ARG;
  }
}

zs_status zs_scaler_init(zs_scaler* s, float scale, float min_scale, int32_t window,
                         int32_t hysteresis, int32_t dynamic) {
  if (s == nullptr || !(scale > 0.0f) || !(min_scale > 0.0f) || window < 1 || hysteresis < 1)
    return ZS_ERR_ARG;
  s->scale = scale;
  s->min_scale = min_scale;
  s->window = window;
  s->clean_count = 0;
  s->hysteresis = hysteresis;
  s->hyst_left = hysteresis;
  s->dynamic = dynamic ? 1 : 0;
  s->consecutive_hysteresis = 0;
  return ZS_OK;
}

zs_status zs_ctx_create(zs_ctx** out) {
  if (out == nullptr) return ZS_ERR_ARG;
  *out = nullptr;
  zs_ctx* c = new zs_ctx();
  const char* pdl = std::getenv("ZEROSHARD_PDL");
  c->pdl = !(pdl != nullptr && pdl[0] == '0');
  const char* fused = std::getenv("ZEROSHARD_FUSED");
  if (fused != nullptr && fused[0] == '0') c->fused_mode = ZS_FUSED_OFF;
  cudaError_t e = cudaGetDevice(&c->device);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&c->sms, cudaDevAttrMultiProcessorCount, c->device);
  int coop = 0;
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, c->device);
  if (coop == 0) c->fused_mode = ZS_FUSED_OFF;  // no cooperative launches: multi-kernel path
  if (e == cudaSuccess) e = cudaMalloc(&c->d_flag, sizeof(int32_t));
  if (e == cudaSuccess) e = cudaMemset(c->d_flag, 0, sizeof(int32_t));
  if (e == cudaSuccess)
    e = cudaHostAlloc(reinterpret_cast<void**>(&c->h_result), sizeof(zs::StepResult),
                      cudaHostAllocMapped);
  if (e == cudaSuccess) {
    std::memset(c->h_result, 0, sizeof(zs::StepResult));
    e = cudaHostGetDevicePointer(reinterpret_cast<void**>(&c->d_result), c->h_result, 0);
  }
  if (e == cudaSuccess) e = cudaMalloc(&c->d_partials, ZS_SUMSQ_MAX_PARTS * sizeof(double));
  if (e == cudaSuccess) e = cudaMalloc(&c->d_sumsq, sizeof(double));
  if (e == cudaSuccess) e = cudaMemset(c->d_sumsq, 0, sizeof(double));
  if (e == cudaSuccess) e = cudaMalloc(&c->d_coef, sizeof(float));
  if (e == cudaSuccess) e = cudaMallocHost(&c->h_sumsq, sizeof(double));
  if (e == cudaSuccess) e = cudaMalloc(&c->d_args, sizeof(zs::AdamArgs));
  if (e == cudaSuccess)
    e = cudaMalloc(&c->d_norm_parts, (size_t)ZS_NORM_MAX_PARTS * sizeof(double));
  if (e == cudaSuccess) e = cudaMalloc(&c->d_sync, sizeof(zs::FusedSync));
  if (e == cudaSuccess) e = cudaMemset(c->d_sync, 0, sizeof(zs::FusedSync));
  if (e == cudaSuccess)
    e = cudaHostAlloc(reinterpret_cast<void**>(&c->h_fused_err), sizeof(int32_t),
                      cudaHostAllocMapped);
  if (e == cudaSuccess) {
    *c->h_fused_err = 0;
    e = cudaHostGetDevicePointer(reinterpret_cast<void**>(&c->d_fused_err), c->h_fused_err, 0);
  }
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    if (c->d_flag) cudaFree(c->d_flag);
    if (c->h_result) cudaFreeHost(c->h_result);
    if (c->d_partials) cudaFree(c->d_partials);
    if (c->d_sumsq) cudaFree(c->d_sumsq);
    if (c->d_coef) cudaFree(c->d_coef);
    if (c->h_sumsq) cudaFreeHost(c->h_sumsq);
    if (c->d_args) cudaFree(c->d_args);
    if (c->d_norm_parts) cudaFree(c->d_norm_parts);
    if (c->d_sync) cudaFree(c->d_sync);
    if (c->h_fused_err) cudaFreeHost(c->h_fused_err);
    delete c;
    return ZS_ERR_CUDA;
  }
  *out = c;
  return ZS_OK;
}

zs_status zs_ctx_destroy(zs_ctx* c) {
  if (c == nullptr) return ZS_ERR_ARG;
  for (auto& r : c->pending) {  // released by the runtime once complete
    cudaEventDestroy(r.start);
    cudaEventDestroy(r.stop);
  }
  for (auto ev : c->pool) cudaEventDestroy(ev);
  cudaFree(c->d_flag);
  cudaFreeHost(c->h_result);  // d_result is its device address
  cudaFree(c->d_partials);
  cudaFree(c->d_sumsq);
  cudaFree(c->d_coef);
  cudaFreeHost(c->h_sumsq);
  cudaFree(c->d_args);
  cudaFree(c->d_norm_parts);
  cudaFree(c->d_sync);
  cudaFreeHost(c->h_fused_err);  // d_fused_err is its device address
  delete c;
  return ZS_OK;
}

const char* zs_last_error(const zs_ctx* c) { return c ? c->err.c_str() : "null context"; }

zs_status zs_ctx_fused_capacity(zs_ctx* c, int64_t* elements) {
  if (c == nullptr || elements == nullptr) return ZS_ERR_ARG;
  int r = fused_resident<false, false, false>(c);
  r = std::min(r, fused_resident<true, false, false>(c));
  r = std::min(r, fused_resident<true, true, false>(c));
  r = std::min(r, fused_resident<false, false, true>(c));
  r = std::min(r, fused_resident<true, false, true>(c));
  // one 8-element unit per thread; the < 8 tail elements ride on CTA 0
  *elements = (int64_t)r * c->sms * zs::kThreads * 8 + 7;
  return ZS_OK;
}

zs_status zs_ctx_set_fused(zs_ctx* c, int32_t mode, int64_t wait_ns) {
  if (c == nullptr) return ZS_ERR_ARG;
  if (mode != ZS_FUSED_OFF && mode != ZS_FUSED_ON && mode != ZS_FUSED_TEST_TIMEOUT)
    return fail(c, ZS_ERR_ARG, "unknown fused mode %d", (int)mode);
  int coop = 0;
  if (mode != ZS_FUSED_OFF &&
      (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, c->device) != cudaSuccess ||
       coop == 0))
    return fail(c, ZS_ERR_ARG, "device %d has no cooperative launches", c->device);
  c->fused_mode = mode;
  c->wait_ns = wait_ns > 0 ? (uint64_t)wait_ns : ZS_DEFAULT_WAIT_NS;
  return ZS_OK;
}

zs_status zs_ctx_overflow_flag(zs_ctx* c, int32_t** d_flag) {
  if (c == nullptr || d_flag == nullptr) return ZS_ERR_ARG;
  *d_flag = c->d_flag;
  return ZS_OK;
}

zs_status zs_reduce_check(zs_ctx* c, const void* const* grads, int32_t n, zs_dtype dt,
                          int64_t count, float* acc, int32_t first, int32_t* d_flag,
                          cudaStream_t stream) {
  NvtxRange nvtx_("zs_reduce_check");
  ZS_TRY(check_ctx(c));
  if (dt != ZS_FP16 && dt != ZS_BF16) return fail(c, ZS_ERR_DTYPE, "unknown dtype %d", (int)dt);
  if (count < 0) return fail(c, ZS_ERR_ARG, "count < 0");
  if (d_flag == nullptr) return fail(c, ZS_ERR_ARG, "d_flag is NULL");
  zs::SlicePtrs sp;
  ZS_TRY(check_slices(c, grads, n, count, &sp));
  ZS_TRY(check_array(c, acc, "acc", 0));
  if (count == 0) return ZS_OK;
  if (acc == nullptr && !first)
    return fail(c, ZS_ERR_ARG, "a check-only call (acc == NULL) must have first = 1");
  return reduce_any(c, dt, sp, n, acc, count, acc != nullptr && !first, acc != nullptr, d_flag,
                    stream);
}

zs_status zs_check_last(zs_ctx* c, const void* const* grads, int32_t n, zs_dtype dt,
                        int64_t count, const float* acc, int32_t* d_flag, cudaStream_t stream) {
  NvtxRange nvtx_("zs_check_last");
  ZS_TRY(check_ctx(c));
  if (dt != ZS_FP16 && dt != ZS_BF16) return fail(c, ZS_ERR_DTYPE, "unknown dtype %d", (int)dt);
  if (count < 0) return fail(c, ZS_ERR_ARG, "count < 0");
  if (d_flag == nullptr) return fail(c, ZS_ERR_ARG, "d_flag is NULL");
  zs::SlicePtrs sp;
  ZS_TRY(check_slices(c, grads, n, count, &sp));
  ZS_TRY(check_array(c, acc, "acc", 0));
  if (count == 0) return ZS_OK;
  // fp16: finite halves cannot sum past the fp32 maximum on top of a finite
  // acc, so the slices decide; bf16 sums on top of acc as the update will
  const bool with_acc = dt == ZS_BF16 && acc != nullptr;
  return reduce_any(c, dt, sp, n, with_acc ? const_cast<float*>(acc) : nullptr, count, with_acc,
                    false, d_flag, stream);
}

zs_status zs_grad_accum(zs_ctx* c, const void* const* grads, int32_t n, zs_dtype dt,
                        int64_t count, float* acc, int32_t first, cudaStream_t stream) {
  NvtxRange nvtx_("zs_grad_accum");
  ZS_TRY(check_ctx(c));
  if (count > 0 && acc == nullptr) return fail(c, ZS_ERR_ARG, "acc is NULL");
  return zs_reduce_check(c, grads, n, dt, count, acc, first, c->d_flag, stream);
}

zs_status zs_apply(zs_ctx* c, const int32_t* d_flag, const void* const* grads, int32_t n,
                   zs_dtype dt, const float* acc, int64_t count, float grad_div, float* master,
                   float* m, float* v, void* half_out, const zs_adam_hparams* hp, int64_t step,
                   cudaStream_t stream) {
  NvtxRange nvtx_("zs_apply");
  ZS_TRY(check_ctx(c));
  if (dt != ZS_FP16 && dt != ZS_BF16) return fail(c, ZS_ERR_DTYPE, "unknown dtype %d", (int)dt);
  if (count < 0) return fail(c, ZS_ERR_ARG, "count < 0");
  if (d_flag == nullptr) return fail(c, ZS_ERR_ARG, "d_flag is NULL");
  if (!(grad_div > 0.0f) || !std::isfinite(grad_div))
    return fail(c, ZS_ERR_ARG, "grad_div must be a positive finite number");
  ZS_TRY(check_hparams(c, hp, step));
  zs::SlicePtrs sp;
  std::memset(&sp, 0, sizeof sp);
  const bool recompute = grads != nullptr;
  if (recompute) ZS_TRY(check_slices(c, grads, n, count, &sp));
  if (!recompute && count > 0 && acc == nullptr)
    return fail(c, ZS_ERR_ARG, "need acc, grads or both");
  ZS_TRY(check_array(c, acc, "acc", 0));
  ZS_TRY(check_array(c, master, "master", count));
  ZS_TRY(check_array(c, m, "m", count));
  ZS_TRY(check_array(c, v, "v", count));
  ZS_TRY(check_array(c, half_out, "half_out", count));
  if (count == 0) return ZS_OK;
  const zs::AdamArgs ad = adam_args(hp, step, grad_div);
  return apply_any(c, dt, d_flag, sp, recompute ? n : 0, recompute, acc, count, ad, master, m, v,
                   half_out, nullptr, nullptr, stream);
}

zs_status zs_scaler_update(zs_ctx* c, const int32_t* d_flag, zs_scaler* scaler,
                           int32_t* overflow_out, cudaStream_t stream) {
  NvtxRange nvtx_("zs_scaler_update");
  ZS_TRY(check_ctx(c));
  if (d_flag == nullptr) return fail(c, ZS_ERR_ARG, "d_flag is NULL");
  ZS_TRY(check_scaler(c, scaler));
  LaunchScope ls(c, stream, ZS_KERNEL_SCALER, 1);
  launch_k(c, zs::k_scaler, 1, 32, stream, d_flag, *scaler, c->d_result);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(c, e, "scaler launch");
  ls.done();
  return finish_step(c, scaler, overflow_out, nullptr, nullptr, stream);
}

static zs_status shard_step_impl(zs_ctx* c, const void* const* grads, int32_t n, zs_dtype dt,
                                 int64_t count, float* acc, int32_t accum_steps, float* master,
                                 float* m, float* v, void* half_out, const zs_adam_hparams* hp,
                                 int64_t step, zs_scaler* scaler, float max_norm,
                                 int32_t* overflow_out, float* new_scale_out,
                                 float* grad_norm_out, cudaStream_t stream) {
  ZS_TRY(check_ctx(c));
  if (dt != ZS_FP16 && dt != ZS_BF16) return fail(c, ZS_ERR_DTYPE, "unknown dtype %d", (int)dt);
  if (count < 0) return fail(c, ZS_ERR_ARG, "count < 0");
  if (accum_steps < 1) return fail(c, ZS_ERR_ARG, "accum_steps must be >= 1");
  if (accum_steps > 1 && acc == nullptr && count > 0)
    return fail(c, ZS_ERR_ARG, "acc is required when accum_steps > 1");
  if (!std::isfinite(max_norm)) return fail(c, ZS_ERR_ARG, "max_norm must be finite");
  ZS_TRY(check_hparams(c, hp, step));
  ZS_TRY(check_scaler(c, scaler));
  zs::SlicePtrs sp;
  ZS_TRY(check_slices(c, grads, n, count, &sp));
  ZS_TRY(check_array(c, acc, "acc", 0));
  ZS_TRY(check_array(c, master, "master", count));
  ZS_TRY(check_array(c, m, "m", count));
  ZS_TRY(check_array(c, v, "v", count));
  ZS_TRY(check_array(c, half_out, "half_out", count));
  const double div = (double)n * (double)accum_steps * (double)scaler->scale;
  const float grad_div = (float)div;
  if (!(grad_div > 0.0f) || !std::isfinite(grad_div))
    return fail(c, ZS_ERR_ARG, "n * accum_steps * scale is not a positive finite fp32");
  const zs::AdamArgs ad = adam_args(hp, step, grad_div);
  const bool recompute = (n < 4) || acc == nullptr;
  const bool clip = max_norm > 0.0f;
  const float* acc_in = (accum_steps > 1 || !recompute) ? acc : nullptr;
  {
    FusedCall f;
    f.sp = sp;
    f.n = n;
    f.acc = accum_steps > 1 ? acc : nullptr;
    f.b = in_place_bufs(master, m, v, half_out);
    f.count = count;
    f.ad = ad;
    f.scaler = *scaler;
    f.accum_steps = accum_steps;
    f.max_norm = max_norm;
    f.inv_div2 = 1.0 / (div * div);
    zs_status fst = ZS_OK;
    const bool fused = clip ? try_fused<false, false, true>(c, dt, f, stream, &fst)
                            : try_fused<false, false>(c, dt, f, stream, &fst);
    if (fused) {
      ZS_TRY(fst);
      if (clip) {
        cudaError_t e = cudaMemcpyAsync(c->h_sumsq, c->d_sumsq, sizeof(double),
                                        cudaMemcpyDeviceToHost, stream);
        if (e != cudaSuccess) return cuda_fail(c, e, "sumsq copy");
      }
      ZS_TRY(finish_fused_step(c, scaler, overflow_out, new_scale_out, stream));
      if (grad_norm_out) {
        *grad_norm_out = 0.0f;
        if (clip && c->h_result->overflow == 0) *grad_norm_out = (float)std::sqrt(*c->h_sumsq);
      }
      return ZS_OK;
    }
  }
  if (count > 0 && clip) {
    // the last micro-step's pass also produces the clipping norm: materialise
    // (sums into acc) or, on the re-read path, sums acc + the last slices
    const bool read = recompute ? acc_in != nullptr : accum_steps > 1;
    ZS_TRY(reduce_norm_any(c, dt, sp, n, recompute ? const_cast<float*>(acc_in) : acc, count,
                           read, !recompute, c->d_flag, grad_div, c->d_sumsq, stream));
  } else if (count > 0) {
    if (recompute) {
      // fp16: finite halves cannot sum past the fp32 maximum, so a check of
      // the last slices alone decides; bf16 sums on top of acc as the update will.
      const bool with_acc = (dt == ZS_BF16) && accum_steps > 1;
      ZS_TRY(reduce_any(c, dt, sp, n, with_acc ? acc : nullptr, count, with_acc, false, c->d_flag,
                        stream));
    } else {
      ZS_TRY(reduce_any(c, dt, sp, n, acc, count, accum_steps > 1, true, c->d_flag, stream));
    }
  }
  if (clip) {
    if (count == 0) {
      cudaError_t e = cudaMemsetAsync(c->d_sumsq, 0, sizeof(double), stream);
      if (e != cudaSuccess) return cuda_fail(c, e, "sumsq reset");
    }
    ZS_TRY(clip_coef_launch(c, c->d_sumsq, max_norm, stream));
    cudaError_t e = cudaMemcpyAsync(c->h_sumsq, c->d_sumsq, sizeof(double),
                                    cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return cuda_fail(c, e, "sumsq copy");
  }
  ZS_TRY(apply_any(c, dt, c->d_flag, sp, recompute ? n : 0, recompute, acc_in, count, ad, master,
                   m, v, half_out, scaler, c->d_result, stream, clip ? c->d_coef : nullptr));
  ZS_TRY(finish_step(c, scaler, overflow_out, new_scale_out, c->d_flag, stream));
  if (grad_norm_out) {
    *grad_norm_out = 0.0f;
    if (clip && c->h_result->overflow == 0) *grad_norm_out = (float)std::sqrt(*c->h_sumsq);
  }
  return ZS_OK;
}

zs_status zs_shard_step(zs_ctx* c, const void* const* grads, int32_t n, zs_dtype dt,
                        int64_t count, float* acc, int32_t accum_steps, float* master, float* m,
                        float* v, void* half_out, const zs_adam_hparams* hp, int64_t step,
                        zs_scaler* scaler, int32_t* overflow_out, float* new_scale_out,
                        cudaStream_t stream) {
  NvtxRange nvtx_("zs_shard_step");
  return shard_step_impl(c, grads, n, dt, count, acc, accum_steps, master, m, v, half_out, hp,
                         step, scaler, 0.0f, overflow_out, new_scale_out, nullptr, stream);
}

zs_status zs_shard_step_clipped(zs_ctx* c, const void* const* grads, int32_t n, zs_dtype dt,
                                int64_t count, float* acc, int32_t accum_steps, float* master,
                                float* m, float* v, void* half_out, const zs_adam_hparams* hp,
                                int64_t step, zs_scaler* scaler, float max_norm,
                                int32_t* overflow_out, float* new_scale_out,
                                float* grad_norm_out, cudaStream_t stream) {
  NvtxRange nvtx_("zs_shard_step_clipped");
  return shard_step_impl(c, grads, n, dt, count, acc, accum_steps, master, m, v, half_out, hp,
                         step, scaler, max_norm, overflow_out, new_scale_out, grad_norm_out,
                         stream);
}

static zs_status shard_step_async_impl(zs_ctx* c, const void* const* grads, int32_t n,
                                       zs_dtype dt, int64_t count, float* acc,
                                       int32_t accum_steps, float* master, float* m, float* v,
                                       void* half_out, const zs_adam_hparams* hp,
                                       const zs_lr_schedule* sched, zs_device_state* d_state,
                                       float max_norm, double* d_norm, cudaStream_t stream) {
  ZS_TRY(check_ctx(c));
  if (dt != ZS_FP16 && dt != ZS_BF16) return fail(c, ZS_ERR_DTYPE, "unknown dtype %d", (int)dt);
  if (count < 0) return fail(c, ZS_ERR_ARG, "count < 0");
  if (accum_steps < 1) return fail(c, ZS_ERR_ARG, "accum_steps must be >= 1");
  if (accum_steps > 1 && acc == nullptr && count > 0)
    return fail(c, ZS_ERR_ARG, "acc is required when accum_steps > 1");
  if (d_state == nullptr) return fail(c, ZS_ERR_ARG, "d_state is NULL");
  if ((reinterpret_cast<uintptr_t>(d_state) & 7u) != 0)
    return fail(c, ZS_ERR_ALIGN, "d_state is not 8-byte aligned");
  if ((reinterpret_cast<uintptr_t>(d_norm) & 7u) != 0)
    return fail(c, ZS_ERR_ALIGN, "d_norm is not 8-byte aligned");
  if (!std::isfinite(max_norm)) return fail(c, ZS_ERR_ARG, "max_norm must be finite");
  ZS_TRY(check_hparams(c, hp, 1));
  if (sched != nullptr && (sched->kind < ZS_LR_CONSTANT || sched->kind > ZS_LR_WARMUP_DECAY ||
                           sched->warmup_steps < 0 || !std::isfinite(sched->min_lr) ||
                           !std::isfinite(sched->max_lr)))
    return fail(c, ZS_ERR_ARG, "bad learning-rate schedule");
  zs::SlicePtrs sp;
  ZS_TRY(check_slices(c, grads, n, count, &sp));
  ZS_TRY(check_array(c, acc, "acc", 0));
  ZS_TRY(check_array(c, master, "master", count));
  ZS_TRY(check_array(c, m, "m", count));
  ZS_TRY(check_array(c, v, "v", count));
  ZS_TRY(check_array(c, half_out, "half_out", count));
  const bool recompute = (n < 4) || acc == nullptr;
  const bool clip = max_norm > 0.0f;
  const float* acc_in = (accum_steps > 1 || !recompute) ? acc : nullptr;
  // per-kernel event timing only outside stream capture (an event recorded
  // into a graph would be timed once per capture, not per replay)
  const bool timing = c->timing;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) {
    (void)cudaGetLastError();  // e.g. the legacy stream while another stream captures
    cap = cudaStreamCaptureStatusActive;
  }
  if (cap != cudaStreamCaptureStatusNone) c->timing = false;
  zs_status st = ZS_OK;
  {
    FusedCall f;
    f.sp = sp;
    f.n = n;
    f.acc = accum_steps > 1 ? acc : nullptr;
    f.b = in_place_bufs(master, m, v, half_out);
    f.count = count;
    f.dstate = d_state;
    f.hp = *hp;
    if (sched) {
      f.sched = *sched;
      f.has_sched = 1;
    }
    f.accum_steps = accum_steps;
    f.max_norm = max_norm;
    f.norm_out = d_norm;
    const bool fused = clip ? try_fused<true, false, true>(c, dt, f, stream, &st)
                            : try_fused<true, false>(c, dt, f, stream, &st);
    if (fused) {
      c->timing = timing;
      return st;
    }
  }
  if (count > 0 && clip) {
    // the last micro-step's pass also forms the sum of squares of the final
    // sums, unscaled (grad_div 1): the scale lives on the device, and the
    // coefficient kernel divides by N*G*S from the step's constants
    const bool read = recompute ? acc_in != nullptr : accum_steps > 1;
    st = reduce_norm_any(c, dt, sp, n, recompute ? const_cast<float*>(acc_in) : acc, count, read,
                         !recompute, c->d_flag, 1.0f, c->d_sumsq, stream);
  } else if (count > 0) {
    if (recompute) {
      const bool with_acc = (dt == ZS_BF16) && accum_steps > 1;
      st = reduce_any(c, dt, sp, n, with_acc ? acc : nullptr, count, with_acc, false, c->d_flag,
                      stream);
    } else {
      st = reduce_any(c, dt, sp, n, acc, count, accum_steps > 1, true, c->d_flag, stream);
    }
  } else if (clip) {
    cudaError_t e = cudaMemsetAsync(c->d_sumsq, 0, sizeof(double), stream);
    if (e != cudaSuccess) st = cuda_fail(c, e, "sumsq reset");
  }
  if (st != ZS_OK) {
    c->timing = timing;
    return st;
  }
  zs_lr_schedule sc{};
  if (sched) sc = *sched;
  launch_k(c, zs::k_step_prologue, 1, 32, stream, (const zs_device_state*)d_state, n,
           accum_steps, *hp, sc, sched ? 1 : 0, c->d_args);
  c->launches += 1;
  if (clip) {
    launch_k(c, zs::k_clip_coef_dev, 1, 32, stream, (const double*)c->d_sumsq,
             (const zs::AdamArgs*)c->d_args, max_norm, c->d_coef, d_norm);
    c->launches += 1;
  }
  uint16_t* ho = static_cast<uint16_t*>(half_out);
  const float* coef = clip ? c->d_coef : nullptr;
  {
    LaunchScope ls(c, stream, recompute ? ZS_KERNEL_APPLY_RECOMPUTE : ZS_KERNEL_APPLY, count);
    if (dt == ZS_FP16)
      apply_dev<ZS_FP16>(c, c->d_flag, sp, recompute ? n : 0, recompute, acc_in, count, master,
                         m, v, ho, c->d_args, d_state, coef, stream);
    else
      apply_dev<ZS_BF16>(c, c->d_flag, sp, recompute ? n : 0, recompute, acc_in, count, master,
                         m, v, ho, c->d_args, d_state, coef, stream);
    ls.done();
  }
  c->timing = timing;
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(c, e, "async step launch");
  launch_k(c, zs::k_clear_flag, 1, 32, stream, c->d_flag);
  c->launches += 1;
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(c, e, "flag reset");
  return ZS_OK;
}

zs_status zs_shard_step_async(zs_ctx* c, const void* const* grads, int32_t n, zs_dtype dt,
                              int64_t count, float* acc, int32_t accum_steps, float* master,
                              float* m, float* v, void* half_out, const zs_adam_hparams* hp,
                              const zs_lr_schedule* sched, zs_device_state* d_state,
                              cudaStream_t stream) {
  NvtxRange nvtx_("zs_shard_step_async");
  return shard_step_async_impl(c, grads, n, dt, count, acc, accum_steps, master, m, v, half_out,
                               hp, sched, d_state, 0.0f, nullptr, stream);
}

zs_status zs_shard_step_async_clipped(zs_ctx* c, const void* const* grads, int32_t n,
                                      zs_dtype dt, int64_t count, float* acc,
                                      int32_t accum_steps, float* master, float* m, float* v,
                                      void* half_out, const zs_adam_hparams* hp,
                                      const zs_lr_schedule* sched, float max_norm,
                                      zs_device_state* d_state, double* d_grad_norm,
                                      cudaStream_t stream) {
  NvtxRange nvtx_("zs_shard_step_async_clipped");
  return shard_step_async_impl(c, grads, n, dt, count, acc, accum_steps, master, m, v, half_out,
                               hp, sched, d_state, max_norm, d_grad_norm, stream);
}

// Checks shared by the out-of-place calls: the step's arguments and the two
// buffer sets (16-byte aligned, each of count elements, no overlap between them).
// h[0] may be NULL (the synchronising call writes one half copy only).
static zs_status check_oop(zs_ctx* c, const void* const* grads, int32_t n, zs_dtype dt,
                           int64_t count, const float* acc, int32_t accum_steps,
                           const float* const p[2], const float* const m[2],
                           const float* const v[2], const void* const h[2], zs::SlicePtrs* sp) {
  if (dt != ZS_FP16 && dt != ZS_BF16) return fail(c, ZS_ERR_DTYPE, "unknown dtype %d", (int)dt);
  if (count < 0) return fail(c, ZS_ERR_ARG, "count < 0");
  if (accum_steps < 1) return fail(c, ZS_ERR_ARG, "accum_steps must be >= 1");
  if (accum_steps > 1 && acc == nullptr && count > 0)
    return fail(c, ZS_ERR_ARG, "acc is required when accum_steps > 1");
  ZS_TRY(check_slices(c, grads, n, count, sp));
  ZS_TRY(check_array(c, acc, "acc", 0));
  const char* names[8] = {"master[0]", "master[1]", "m[0]", "m[1]", "v[0]", "v[1]",
                          "half[0]", "half[1]"};
  const void* arr[8] = {p[0], p[1], m[0], m[1], v[0], v[1], h[0], h[1]};
  const int64_t bytes[8] = {4 * count, 4 * count, 4 * count, 4 * count,
                            4 * count, 4 * count, 2 * count, 2 * count};
  for (int i = 0; i < 8; ++i)
    if (i != 6 || h[0] != nullptr) ZS_TRY(check_array(c, arr[i], names[i], count));
  for (int i = 0; i < 8; ++i)
    for (int j = i + 1; j < 8; ++j)
      if (arr[i] != nullptr && arr[j] != nullptr && overlaps(arr[i], bytes[i], arr[j], bytes[j]))
        return fail(c, ZS_ERR_ARG, "%s and %s overlap", names[i], names[j]);
  return ZS_OK;
}

zs_status zs_shard_step_oop(zs_ctx* c, const void* const* grads, int32_t n, zs_dtype dt,
                            int64_t count, const float* acc, int32_t accum_steps,
                            const float* master_in, const float* m_in, const float* v_in,
                            float* master_out, float* m_out, float* v_out, void* half_out,
                            const zs_adam_hparams* hp, int64_t step, zs_scaler* scaler,
                            int32_t* overflow_out, float* new_scale_out, cudaStream_t stream) {
  NvtxRange nvtx_("zs_shard_step_oop");
  ZS_TRY(check_ctx(c));
  ZS_TRY(check_hparams(c, hp, step));
  ZS_TRY(check_scaler(c, scaler));
  zs::SlicePtrs sp;
  const float* pp[2] = {master_in, master_out};
  const float* mm[2] = {m_in, m_out};
  const float* vv[2] = {v_in, v_out};
  const void* hh[2] = {nullptr, half_out};  // the previous half copy is not read
  ZS_TRY(check_oop(c, grads, n, dt, count, accum_steps > 1 ? acc : nullptr, accum_steps, pp, mm,
                   vv, hh, &sp));
  const double div = (double)n * (double)accum_steps * (double)scaler->scale;
  const float grad_div = (float)div;
  if (!(grad_div > 0.0f) || !std::isfinite(grad_div))
    return fail(c, ZS_ERR_ARG, "n * accum_steps * scale is not a positive finite fp32");
  const zs::AdamArgs ad = adam_args(hp, step, grad_div);
  zs::OopBufs b;
  b.p[0] = const_cast<float*>(master_in);
  b.p[1] = master_out;
  b.m[0] = const_cast<float*>(m_in);
  b.m[1] = m_out;
  b.v[0] = const_cast<float*>(v_in);
  b.v[1] = v_out;
  b.h[0] = nullptr;
  b.h[1] = static_cast<uint16_t*>(half_out);
  {
    FusedCall f;
    f.sp = sp;
    f.n = n;
    f.acc = accum_steps > 1 ? acc : nullptr;
    f.b = b;
    f.count = count;
    f.ad = ad;
    f.scaler = *scaler;
    f.accum_steps = accum_steps;
    zs_status fst = ZS_OK;
    if (try_fused<false, false>(c, dt, f, stream, &fst)) {
      ZS_TRY(fst);
      return finish_fused_step(c, scaler, overflow_out, new_scale_out, stream);
    }
  }
  ZS_TRY(update_oop<false>(c, dt, sp, n, accum_steps > 1 ? acc : nullptr, b, count, ad, nullptr,
                           nullptr, stream));
  launch_k(c, zs::k_commit_oop<false>, 1, 32, stream, c->d_flag, (zs_device_state*)nullptr,
           (const zs::AdamArgs*)nullptr, *scaler, c->d_result);
  c->launches += 1;
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(c, e, "commit launch");
  return finish_step(c, scaler, overflow_out, new_scale_out, nullptr, stream);
}

zs_status zs_update_oop(zs_ctx* c, const void* const* grads, int32_t n, zs_dtype dt,
                        int64_t count, const float* acc, float grad_div, const float* master_in,
                        const float* m_in, const float* v_in, float* master_out, float* m_out,
                        float* v_out, void* half_out, const zs_adam_hparams* hp, int64_t step,
                        int32_t* d_flag, cudaStream_t stream) {
  NvtxRange nvtx_("zs_update_oop");
  ZS_TRY(check_ctx(c));
  ZS_TRY(check_hparams(c, hp, step));
  if (d_flag == nullptr) return fail(c, ZS_ERR_ARG, "d_flag is NULL");
  if (!(grad_div > 0.0f) || !std::isfinite(grad_div))
    return fail(c, ZS_ERR_ARG, "grad_div must be a positive finite number");
  zs::SlicePtrs sp;
  const float* pp[2] = {master_in, master_out};
  const float* mm[2] = {m_in, m_out};
  const float* vv[2] = {v_in, v_out};
  const void* hh[2] = {nullptr, half_out};
  ZS_TRY(check_oop(c, grads, n, dt, count, acc, acc ? 2 : 1, pp, mm, vv, hh, &sp));
  if (count == 0) return ZS_OK;
  const zs::AdamArgs ad = adam_args(hp, step, grad_div);
  zs::OopBufs b;
  b.p[0] = const_cast<float*>(master_in);
  b.p[1] = master_out;
  b.m[0] = const_cast<float*>(m_in);
  b.m[1] = m_out;
  b.v[0] = const_cast<float*>(v_in);
  b.v[1] = v_out;
  b.h[0] = nullptr;
  b.h[1] = static_cast<uint16_t*>(half_out);
  return update_oop<false>(c, dt, sp, n, acc, b, count, ad, nullptr, nullptr, stream, d_flag);
}

zs_status zs_shard_step_async_oop(zs_ctx* c, const void* const* grads, int32_t n, zs_dtype dt,
                                  int64_t count, const float* acc, int32_t accum_steps,
                                  float* const* master, float* const* m, float* const* v,
                                  void* const* half, const zs_adam_hparams* hp,
                                  const zs_lr_schedule* sched, zs_device_state* d_state,
                                  cudaStream_t stream) {
  NvtxRange nvtx_("zs_shard_step_async_oop");
  ZS_TRY(check_ctx(c));
  if (master == nullptr || m == nullptr || v == nullptr || half == nullptr)
    return fail(c, ZS_ERR_ARG, "a buffer pair is NULL");
  if (d_state == nullptr) return fail(c, ZS_ERR_ARG, "d_state is NULL");
  if ((reinterpret_cast<uintptr_t>(d_state) & 7u) != 0)
    return fail(c, ZS_ERR_ALIGN, "d_state is not 8-byte aligned");
  ZS_TRY(check_hparams(c, hp, 1));
  if (sched != nullptr && (sched->kind < ZS_LR_CONSTANT || sched->kind > ZS_LR_WARMUP_DECAY ||
                           sched->warmup_steps < 0 || !std::isfinite(sched->min_lr) ||
                           !std::isfinite(sched->max_lr)))
    return fail(c, ZS_ERR_ARG, "bad learning-rate schedule");
  zs::SlicePtrs sp;
  const float* pp[2] = {master[0], master[1]};
  const float* mm[2] = {m[0], m[1]};
  const float* vv[2] = {v[0], v[1]};
  const void* hh[2] = {half[0], half[1]};
  const float* acc_in = accum_steps > 1 ? acc : nullptr;
  ZS_TRY(check_oop(c, grads, n, dt, count, acc_in, accum_steps, pp, mm, vv, hh, &sp));
  zs_lr_schedule sc{};
  if (sched) sc = *sched;
  // per-kernel event timing only outside stream capture
  const bool timing = c->timing;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) {
    (void)cudaGetLastError();
    cap = cudaStreamCaptureStatusActive;
  }
  if (cap != cudaStreamCaptureStatusNone) c->timing = false;
  zs::OopBufs b;
  for (int i = 0; i < 2; ++i) {
    b.p[i] = master[i];
    b.m[i] = m[i];
    b.v[i] = v[i];
    b.h[i] = static_cast<uint16_t*>(half[i]);
  }
  {
    FusedCall f;
    f.sp = sp;
    f.n = n;
    f.acc = acc_in;
    f.b = b;
    f.count = count;
    f.dstate = d_state;
    f.hp = *hp;
    f.sched = sc;
    f.has_sched = sched ? 1 : 0;
    f.accum_steps = accum_steps;
    zs_status fst = ZS_OK;
    if (try_fused<true, true>(c, dt, f, stream, &fst)) {
      c->timing = timing;
      return fst;
    }
  }
  launch_k(c, zs::k_step_prologue, 1, 32, stream, (const zs_device_state*)d_state, n,
           accum_steps, *hp, sc, sched ? 1 : 0, c->d_args);
  c->launches += 1;
  const zs::AdamArgs unused{};
  zs_status st = update_oop<true>(c, dt, sp, n, acc_in, b, count, unused, c->d_args, d_state,
                                  stream);
  c->timing = timing;
  ZS_TRY(st);
  const zs_scaler unused_sc{};
  launch_k(c, zs::k_commit_oop<true>, 1, 32, stream, c->d_flag, d_state,
           (const zs::AdamArgs*)c->d_args, unused_sc, (zs::StepResult*)nullptr);
  c->launches += 1;
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(c, e, "commit launch");
  return ZS_OK;
}

zs_status zs_grad_accum_halfacc(zs_ctx* c, const void* const* grads, int32_t n, zs_dtype dt,
                                int64_t count, void* acc_half, int32_t first,
                                cudaStream_t stream) {
  NvtxRange nvtx_("zs_grad_accum_halfacc");
  ZS_TRY(check_ctx(c));
  if (dt != ZS_FP16 && dt != ZS_BF16) return fail(c, ZS_ERR_DTYPE, "unknown dtype %d", (int)dt);
  if (count < 0) return fail(c, ZS_ERR_ARG, "count < 0");
  zs::SlicePtrs sp;
  ZS_TRY(check_slices(c, grads, n, count, &sp));
  ZS_TRY(check_array(c, acc_half, "acc_half", count));
  if (count == 0) return ZS_OK;
  return reduce_hacc(c, dt, sp, n, acc_half, count, !first, c->d_flag, stream);
}

zs_status zs_shard_step_halfacc(zs_ctx* c, const void* const* grads, int32_t n, zs_dtype dt,
                                int64_t count, void* acc_half, int32_t accum_steps,
                                float* master, float* m, float* v, void* half_out,
                                const zs_adam_hparams* hp, int64_t step, zs_scaler* scaler,
                                int32_t* overflow_out, float* new_scale_out,
                                cudaStream_t stream) {
  NvtxRange nvtx_("zs_shard_step_halfacc");
  ZS_TRY(check_ctx(c));
  if (dt != ZS_FP16 && dt != ZS_BF16) return fail(c, ZS_ERR_DTYPE, "unknown dtype %d", (int)dt);
  if (count < 0) return fail(c, ZS_ERR_ARG, "count < 0");
  if (accum_steps < 1) return fail(c, ZS_ERR_ARG, "accum_steps must be >= 1");
  ZS_TRY(check_hparams(c, hp, step));
  ZS_TRY(check_scaler(c, scaler));
  zs::SlicePtrs sp;
  ZS_TRY(check_slices(c, grads, n, count, &sp));
  ZS_TRY(check_array(c, acc_half, "acc_half", count));
  ZS_TRY(check_array(c, master, "master", count));
  ZS_TRY(check_array(c, m, "m", count));
  ZS_TRY(check_array(c, v, "v", count));
  ZS_TRY(check_array(c, half_out, "half_out", count));
  const double div = (double)n * (double)accum_steps * (double)scaler->scale;
  const float grad_div = (float)div;
  if (!(grad_div > 0.0f) || !std::isfinite(grad_div))
    return fail(c, ZS_ERR_ARG, "n * accum_steps * scale is not a positive finite fp32");
  const zs::AdamArgs ad = adam_args(hp, step, grad_div);
  {
    FusedCall f;
    f.sp = sp;
    f.n = n;
    f.acc = accum_steps > 1 ? static_cast<const float*>(acc_half) : nullptr;
    f.b = in_place_bufs(master, m, v, half_out);
    f.count = count;
    f.ad = ad;
    f.scaler = *scaler;
    f.accum_steps = accum_steps;
    f.hacc = true;
    zs_status fst = ZS_OK;
    if (try_fused<false, false>(c, dt, f, stream, &fst)) {
      ZS_TRY(fst);
      return finish_fused_step(c, scaler, overflow_out, new_scale_out, stream);
    }
  }
  if (count > 0)
    ZS_TRY(reduce_hacc(c, dt, sp, n, acc_half, count, accum_steps > 1, c->d_flag, stream));
  ZS_TRY(apply_hacc(c, dt, c->d_flag, acc_half, count, ad, master, m, v, half_out, scaler,
                    c->d_result, stream));
  return finish_step(c, scaler, overflow_out, new_scale_out, c->d_flag, stream);
}

zs_status zs_shard_step_halfacc_oop(zs_ctx* c, const void* const* grads, int32_t n,
                                    zs_dtype dt, int64_t count, const void* acc_half,
                                    int32_t accum_steps, const float* master_in,
                                    const float* m_in, const float* v_in, float* master_out,
                                    float* m_out, float* v_out, void* half_out,
                                    const zs_adam_hparams* hp, int64_t step, zs_scaler* scaler,
                                    int32_t* overflow_out, float* new_scale_out,
                                    cudaStream_t stream) {
  NvtxRange nvtx_("zs_shard_step_halfacc_oop");
  ZS_TRY(check_ctx(c));
  ZS_TRY(check_hparams(c, hp, step));
  ZS_TRY(check_scaler(c, scaler));
  zs::SlicePtrs sp;
  const float* pp[2] = {master_in, master_out};
  const float* mm[2] = {m_in, m_out};
  const float* vv[2] = {v_in, v_out};
  const void* hh[2] = {nullptr, half_out};
  const float* acc = accum_steps > 1 ? static_cast<const float*>(acc_half) : nullptr;
  ZS_TRY(check_oop(c, grads, n, dt, count, acc, accum_steps, pp, mm, vv, hh, &sp));
  const double div = (double)n * (double)accum_steps * (double)scaler->scale;
  const float grad_div = (float)div;
  if (!(grad_div > 0.0f) || !std::isfinite(grad_div))
    return fail(c, ZS_ERR_ARG, "n * accum_steps * scale is not a positive finite fp32");
  const zs::AdamArgs ad = adam_args(hp, step, grad_div);
  zs::OopBufs b;
  b.p[0] = const_cast<float*>(master_in);
  b.p[1] = master_out;
  b.m[0] = const_cast<float*>(m_in);
  b.m[1] = m_out;
  b.v[0] = const_cast<float*>(v_in);
  b.v[1] = v_out;
  b.h[0] = nullptr;
  b.h[1] = static_cast<uint16_t*>(half_out);
  {
    FusedCall f;
    f.sp = sp;
    f.n = n;
    f.acc = acc;
    f.b = b;
    f.count = count;
    f.ad = ad;
    f.scaler = *scaler;
    f.accum_steps = accum_steps;
    f.hacc = true;
    zs_status fst = ZS_OK;
    if (try_fused<false, false>(c, dt, f, stream, &fst)) {
      ZS_TRY(fst);
      return finish_fused_step(c, scaler, overflow_out, new_scale_out, stream);
    }
  }
  if (count > 0) {
    LaunchScope ls(c, stream, ZS_KERNEL_UPDATE_OOP, count);
    if (dt == ZS_FP16) {
      if (acc) launch_oop_k<ZS_FP16, true, false, true>(c, sp, n, acc, b, count, ad, nullptr, nullptr, c->d_flag, stream);
      else launch_oop_k<ZS_FP16, false, false, true>(c, sp, n, acc, b, count, ad, nullptr, nullptr, c->d_flag, stream);
    } else {
      if (acc) launch_oop_k<ZS_BF16, true, false, true>(c, sp, n, acc, b, count, ad, nullptr, nullptr, c->d_flag, stream);
      else launch_oop_k<ZS_BF16, false, false, true>(c, sp, n, acc, b, count, ad, nullptr, nullptr, c->d_flag, stream);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(c, e, "out-of-place update launch");
    ls.done();
  }
  launch_k(c, zs::k_commit_oop<false>, 1, 32, stream, c->d_flag, (zs_device_state*)nullptr,
           (const zs::AdamArgs*)nullptr, *scaler, c->d_result);
  c->launches += 1;
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(c, e, "commit launch");
  return finish_step(c, scaler, overflow_out, new_scale_out, nullptr, stream);
}

// Checks shared by the device-resident half-accumulator calls.
static zs_status check_device_args(zs_ctx* c, const zs_adam_hparams* hp,
                                   const zs_lr_schedule* sched, const zs_device_state* d_state) {
  if (d_state == nullptr) return fail(c, ZS_ERR_ARG, "d_state is NULL");
  if ((reinterpret_cast<uintptr_t>(d_state) & 7u) != 0)
    return fail(c, ZS_ERR_ALIGN, "d_state is not 8-byte aligned");
  ZS_TRY(check_hparams(c, hp, 1));
  if (sched != nullptr && (sched->kind < ZS_LR_CONSTANT || sched->kind > ZS_LR_WARMUP_DECAY ||
                           sched->warmup_steps < 0 || !std::isfinite(sched->min_lr) ||
                           !std::isfinite(sched->max_lr)))
    return fail(c, ZS_ERR_ARG, "bad learning-rate schedule");
  return ZS_OK;
}

zs_status zs_shard_step_halfacc_async(zs_ctx* c, const void* const* grads, int32_t n,
                                      zs_dtype dt, int64_t count, void* acc_half,
                                      int32_t accum_steps, float* master, float* m, float* v,
                                      void* half_out, const zs_adam_hparams* hp,
                                      const zs_lr_schedule* sched, zs_device_state* d_state,
                                      cudaStream_t stream) {
  NvtxRange nvtx_("zs_shard_step_halfacc_async");
  ZS_TRY(check_ctx(c));
  if (dt != ZS_FP16 && dt != ZS_BF16) return fail(c, ZS_ERR_DTYPE, "unknown dtype %d", (int)dt);
  if (count < 0) return fail(c, ZS_ERR_ARG, "count < 0");
  if (accum_steps < 1) return fail(c, ZS_ERR_ARG, "accum_steps must be >= 1");
  ZS_TRY(check_device_args(c, hp, sched, d_state));
  zs::SlicePtrs sp;
  ZS_TRY(check_slices(c, grads, n, count, &sp));
  ZS_TRY(check_array(c, acc_half, "acc_half", count));
  ZS_TRY(check_array(c, master, "master", count));
  ZS_TRY(check_array(c, m, "m", count));
  ZS_TRY(check_array(c, v, "v", count));
  ZS_TRY(check_array(c, half_out, "half_out", count));
  zs_lr_schedule sc{};
  if (sched) sc = *sched;
  {
    FusedCall f;
    f.sp = sp;
    f.n = n;
    f.acc = accum_steps > 1 ? static_cast<const float*>(acc_half) : nullptr;
    f.b = in_place_bufs(master, m, v, half_out);
    f.count = count;
    f.dstate = d_state;
    f.hp = *hp;
    f.sched = sc;
    f.has_sched = sched ? 1 : 0;
    f.accum_steps = accum_steps;
    f.hacc = true;
    zs_status fst = ZS_OK;
    if (try_fused<true, false>(c, dt, f, stream, &fst)) return fst;
  }
  if (count > 0)
    ZS_TRY(reduce_hacc(c, dt, sp, n, acc_half, count, accum_steps > 1, c->d_flag, stream));
  launch_k(c, zs::k_step_prologue, 1, 32, stream, (const zs_device_state*)d_state, n,
           accum_steps, *hp, sc, sched ? 1 : 0, c->d_args);
  c->launches += 1;
  const zs::AdamArgs unused{};
  ZS_TRY(apply_hacc(c, dt, c->d_flag, acc_half, count, unused, master, m, v, half_out, nullptr,
                    nullptr, stream, c->d_args, d_state));
  launch_k(c, zs::k_clear_flag, 1, 32, stream, c->d_flag);
  c->launches += 1;
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? ZS_OK : cuda_fail(c, e, "flag reset");
}

zs_status zs_shard_step_halfacc_async_oop(zs_ctx* c, const void* const* grads, int32_t n,
                                          zs_dtype dt, int64_t count, const void* acc_half,
                                          int32_t accum_steps, float* const* master,
                                          float* const* m, float* const* v, void* const* half,
                                          const zs_adam_hparams* hp,
                                          const zs_lr_schedule* sched,
                                          zs_device_state* d_state, cudaStream_t stream) {
  NvtxRange nvtx_("zs_shard_step_halfacc_async_oop");
  ZS_TRY(check_ctx(c));
  if (master == nullptr || m == nullptr || v == nullptr || half == nullptr)
    return fail(c, ZS_ERR_ARG, "a buffer pair is NULL");
  ZS_TRY(check_device_args(c, hp, sched, d_state));
  zs::SlicePtrs sp;
  const float* pp[2] = {master[0], master[1]};
  const float* mm[2] = {m[0], m[1]};
  const float* vv[2] = {v[0], v[1]};
  const void* hh[2] = {half[0], half[1]};
  const float* acc = accum_steps > 1 ? static_cast<const float*>(acc_half) : nullptr;
  ZS_TRY(check_oop(c, grads, n, dt, count, acc, accum_steps, pp, mm, vv, hh, &sp));
  zs_lr_schedule sc{};
  if (sched) sc = *sched;
  zs::OopBufs b;
  for (int i = 0; i < 2; ++i) {
    b.p[i] = master[i];
    b.m[i] = m[i];
    b.v[i] = v[i];
    b.h[i] = static_cast<uint16_t*>(half[i]);
  }
  {
    FusedCall f;
    f.sp = sp;
    f.n = n;
    f.acc = acc;
    f.b = b;
    f.count = count;
    f.dstate = d_state;
    f.hp = *hp;
    f.sched = sc;
    f.has_sched = sched ? 1 : 0;
    f.accum_steps = accum_steps;
    f.hacc = true;
    zs_status fst = ZS_OK;
    if (try_fused<true, true>(c, dt, f, stream, &fst)) return fst;
  }
  launch_k(c, zs::k_step_prologue, 1, 32, stream, (const zs_device_state*)d_state, n,
           accum_steps, *hp, sc, sched ? 1 : 0, c->d_args);
  c->launches += 1;
  if (count > 0) {
    LaunchScope ls(c, stream, ZS_KERNEL_UPDATE_OOP, count);
    const zs::AdamArgs unused{};
    const zs::AdamArgs* ad = c->d_args;
    if (dt == ZS_FP16) {
      if (acc) launch_oop_k<ZS_FP16, true, true, true>(c, sp, n, acc, b, count, unused, ad, d_state, c->d_flag, stream);
      else launch_oop_k<ZS_FP16, false, true, true>(c, sp, n, acc, b, count, unused, ad, d_state, c->d_flag, stream);
    } else {
      if (acc) launch_oop_k<ZS_BF16, true, true, true>(c, sp, n, acc, b, count, unused, ad, d_state, c->d_flag, stream);
      else launch_oop_k<ZS_BF16, false, true, true>(c, sp, n, acc, b, count, unused, ad, d_state, c->d_flag, stream);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(c, e, "out-of-place update launch");
    ls.done();
  }
  const zs_scaler unused_sc{};
  launch_k(c, zs::k_commit_oop<true>, 1, 32, stream, c->d_flag, d_state,
           (const zs::AdamArgs*)c->d_args, unused_sc, (zs::StepResult*)nullptr);
  c->launches += 1;
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? ZS_OK : cuda_fail(c, e, "commit launch");
}

zs_status zs_grad_sumsq(zs_ctx* c, const void* const* grads, int32_t n, zs_dtype dt,
                        const float* acc, int64_t count, float grad_div, double* d_sumsq,
                        cudaStream_t stream) {
  NvtxRange nvtx_("zs_grad_sumsq");
  ZS_TRY(check_ctx(c));
  if (dt != ZS_FP16 && dt != ZS_BF16) return fail(c, ZS_ERR_DTYPE, "unknown dtype %d", (int)dt);
  if (count < 0) return fail(c, ZS_ERR_ARG, "count < 0");
  if (d_sumsq == nullptr) return fail(c, ZS_ERR_ARG, "d_sumsq is NULL");
  if (!(grad_div > 0.0f) || !std::isfinite(grad_div))
    return fail(c, ZS_ERR_ARG, "grad_div must be a positive finite number");
  zs::SlicePtrs sp;
  std::memset(&sp, 0, sizeof sp);
  const bool recompute = grads != nullptr;
  if (recompute) ZS_TRY(check_slices(c, grads, n, count, &sp));
  if (!recompute && count > 0 && acc == nullptr)
    return fail(c, ZS_ERR_ARG, "need acc, grads or both");
  ZS_TRY(check_array(c, acc, "acc", 0));
  if (count == 0) {
    cudaError_t e = cudaMemsetAsync(d_sumsq, 0, sizeof(double), stream);
    return e == cudaSuccess ? ZS_OK : cuda_fail(c, e, "sumsq reset");
  }
  return sumsq_any(c, dt, sp, recompute ? n : 0, recompute, acc, count, grad_div, c->d_partials,
                   d_sumsq, stream);
}

zs_status zs_apply_clipped(zs_ctx* c, const int32_t* d_flag, const double* d_sumsq,
                           float max_norm, const void* const* grads, int32_t n, zs_dtype dt,
                           const float* acc, int64_t count, float grad_div, float* master,
                           float* m, float* v, void* half_out, const zs_adam_hparams* hp,
                           int64_t step, cudaStream_t stream) {
  NvtxRange nvtx_("zs_apply_clipped");
  ZS_TRY(check_ctx(c));
  if (!std::isfinite(max_norm)) return fail(c, ZS_ERR_ARG, "max_norm must be finite");
  if (max_norm <= 0.0f)
    return zs_apply(c, d_flag, grads, n, dt, acc, count, grad_div, master, m, v, half_out, hp,
                    step, stream);
  if (d_sumsq == nullptr) return fail(c, ZS_ERR_ARG, "d_sumsq is NULL");
  if (dt != ZS_FP16 && dt != ZS_BF16) return fail(c, ZS_ERR_DTYPE, "unknown dtype %d", (int)dt);
  if (count < 0) return fail(c, ZS_ERR_ARG, "count < 0");
  if (d_flag == nullptr) return fail(c, ZS_ERR_ARG, "d_flag is NULL");
  if (!(grad_div > 0.0f) || !std::isfinite(grad_div))
    return fail(c, ZS_ERR_ARG, "grad_div must be a positive finite number");
  ZS_TRY(check_hparams(c, hp, step));
  zs::SlicePtrs sp;
  std::memset(&sp, 0, sizeof sp);
  const bool recompute = grads != nullptr;
  if (recompute) ZS_TRY(check_slices(c, grads, n, count, &sp));
  if (!recompute && count > 0 && acc == nullptr)
    return fail(c, ZS_ERR_ARG, "need acc, grads or both");
  ZS_TRY(check_array(c, acc, "acc", 0));
  ZS_TRY(check_array(c, master, "master", count));
  ZS_TRY(check_array(c, m, "m", count));
  ZS_TRY(check_array(c, v, "v", count));
  ZS_TRY(check_array(c, half_out, "half_out", count));
  if (count == 0) return ZS_OK;
  ZS_TRY(clip_coef_launch(c, d_sumsq, max_norm, stream));
  const zs::AdamArgs ad = adam_args(hp, step, grad_div);
  return apply_any(c, dt, d_flag, sp, recompute ? n : 0, recompute, acc, count, ad, master, m, v,
                   half_out, nullptr, nullptr, stream, c->d_coef);
}

zs_status zs_copy_peak(zs_ctx* c, const void* src, void* dst, int64_t bytes, int32_t read_only,
                       cudaStream_t stream) {
  NvtxRange nvtx_("zs_copy_peak");
  ZS_TRY(check_ctx(c));
  if (bytes < 0 || bytes % 16 != 0) return fail(c, ZS_ERR_ARG, "bytes must be a multiple of 16");
  ZS_TRY(check_array(c, src, "src", bytes));
  ZS_TRY(check_array(c, dst, "dst", 1));
  if (bytes == 0) return ZS_OK;
  const int64_t nvec = bytes / 16;
  LaunchScope ls(c, stream, ZS_KERNEL_COPY, bytes);
  if (read_only) {
    zs::k_read<<<grid_for(c, zs::k_read, nvec / 4 + 1), zs::kThreads, 0, stream>>>(
        static_cast<const uint4*>(src), nvec, static_cast<uint4*>(dst), 0x9E3779B9u);
  } else {
    zs::k_copy<<<grid_for(c, zs::k_copy, nvec / 4 + 1), zs::kThreads, 0, stream>>>(
        static_cast<const uint4*>(src), static_cast<uint4*>(dst), nvec);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(c, e, "copy launch");
  ls.done();
  return ZS_OK;
}

// ---------------------------------------------------------------- engine

}  // extern "C"

struct zs_engine {
  zs_ctx* ctx = nullptr;
  zs_engine_config cfg{};
  int32_t micro = 0;                // backward calls in the current step
  std::vector<const void*> last;    // the G-th micro-batch's slices
  int64_t global_steps = 0, applied = 0, micro_total = 0;
};

namespace {

// The schedules' learning rate at Adam step t, computed the way the device
// prologue does (fp64, one rounding to fp32).
float host_lr_at(const zs_lr_schedule& sc, int64_t t) {
  const double mn = sc.min_lr, mx = sc.max_lr;
  if (sc.kind == ZS_LR_CONSTANT) return (float)mx;
  double frac = sc.warmup_steps > 0 ? (double)t / (double)sc.warmup_steps : 1.0;
  if (frac > 1.0) frac = 1.0;
  const double warm = mn + (mx - mn) * frac;
  if (sc.kind == ZS_LR_WARMUP || t <= sc.warmup_steps) return (float)warm;
  if (sc.total_steps <= sc.warmup_steps) return 0.0f;
  double rest = (double)(sc.total_steps - t) / (double)(sc.total_steps - sc.warmup_steps);
  if (rest < 0.0) rest = 0.0;
  return (float)(mx * rest);
}

}  // namespace

extern "C" {

zs_status zs_engine_create(zs_ctx* c, const zs_engine_config* cfg, zs_engine** out) {
  if (out == nullptr) return ZS_ERR_ARG;
  *out = nullptr;
  ZS_TRY(check_ctx(c));
  if (cfg == nullptr) return fail(c, ZS_ERR_ARG, "cfg is NULL");
  if (cfg->n < 1 || cfg->n > ZS_MAX_RANKS) return fail(c, ZS_ERR_ARG, "n out of range");
  if (cfg->dt != ZS_FP16 && cfg->dt != ZS_BF16) return fail(c, ZS_ERR_DTYPE, "unknown dtype");
  if (cfg->count < 0 || cfg->accum_steps < 1) return fail(c, ZS_ERR_ARG, "bad count or accum_steps");
  if (cfg->accum_steps > 1 && cfg->acc == nullptr && cfg->count > 0)
    return fail(c, ZS_ERR_ARG, "acc is required when accum_steps > 1");
  ZS_TRY(check_hparams(c, &cfg->hp, 1));
  ZS_TRY(check_scaler(c, &cfg->scaler));
  if (cfg->has_schedule &&
      (cfg->schedule.kind < ZS_LR_CONSTANT || cfg->schedule.kind > ZS_LR_WARMUP_DECAY))
    return fail(c, ZS_ERR_ARG, "bad learning-rate schedule");
  zs_engine* e = new zs_engine();
  e->ctx = c;
  e->cfg = *cfg;
  *out = e;
  return ZS_OK;
}

zs_status zs_engine_destroy(zs_engine* e) {
  if (e == nullptr) return ZS_ERR_ARG;
  delete e;
  return ZS_OK;
}

zs_status zs_engine_backward(zs_engine* e, const void* const* grads, cudaStream_t stream) {
  if (e == nullptr) return ZS_ERR_ARG;
  NvtxRange nvtx_("zs_engine_backward");
  zs_ctx* c = e->ctx;
  const zs_engine_config& f = e->cfg;
  if (e->micro >= f.accum_steps)
    return fail(c, ZS_ERR_ARG, "zs_engine_step must follow the last micro-batch's backward");
  if (grads == nullptr) return fail(c, ZS_ERR_ARG, "grads is NULL");
  if (e->micro < f.accum_steps - 1) {
    ZS_TRY(zs_grad_accum(c, grads, f.n, f.dt, f.count, f.acc, e->micro == 0 ? 1 : 0, stream));
  } else {
    e->last.assign(grads, grads + f.n);
  }
  e->micro += 1;
  e->micro_total += 1;
  return ZS_OK;
}

zs_status zs_engine_step(zs_engine* e, int32_t* stepped, int32_t* overflow_out, float* scale_out,
                         float* grad_norm_out, cudaStream_t stream) {
  if (e == nullptr) return ZS_ERR_ARG;
  NvtxRange nvtx_("zs_engine_step");
  const zs_engine_config& f = e->cfg;
  if (stepped) *stepped = 0;
  if (e->micro < f.accum_steps) return ZS_OK;  // not at the accumulation boundary
  zs_adam_hparams hp = f.hp;
  if (f.has_schedule) hp.lr = host_lr_at(f.schedule, e->applied + 1);
  int32_t ovf = 0;
  float scale = 0.0f, norm = 0.0f;
  ZS_TRY(shard_step_impl(e->ctx, e->last.data(), f.n, f.dt, f.count, f.acc, f.accum_steps,
                         f.master, f.m, f.v, f.half_out, &hp, e->applied + 1, &e->cfg.scaler,
                         f.max_grad_norm > 0.0f ? f.max_grad_norm : 0.0f, &ovf, &scale, &norm,
                         stream));
  e->micro = 0;
  e->global_steps += 1;
  if (!ovf) e->applied += 1;
  if (stepped) *stepped = 1;
  if (overflow_out) *overflow_out = ovf;
  if (scale_out) *scale_out = scale;
  if (grad_norm_out) *grad_norm_out = norm;
  return ZS_OK;
}

zs_status zs_engine_state(const zs_engine* e, int64_t* global_steps, int64_t* applied_steps,
                          int64_t* micro_steps, zs_scaler* scaler) {
  if (e == nullptr) return ZS_ERR_ARG;
  if (global_steps) *global_steps = e->global_steps;
  if (applied_steps) *applied_steps = e->applied;
  if (micro_steps) *micro_steps = e->micro_total;
  if (scaler) *scaler = e->cfg.scaler;
  return ZS_OK;
}

zs_status zs_ctx_set_timing(zs_ctx* c, int32_t enable) {
  if (c == nullptr) return ZS_ERR_ARG;
  c->timing = enable != 0;
  return ZS_OK;
}

// Folds every pending record into the totals, waiting for each.  A record
// whose events cannot be read is dropped (its events destroyed) and reported
// after the rest have been folded.
static zs_status drain_timing(zs_ctx* c) {
  cudaError_t first = cudaSuccess;
  for (auto& r : c->pending) {
    float ms = 0.0f;
    cudaError_t e = cudaEventSynchronize(r.stop);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, r.start, r.stop);
    if (e != cudaSuccess) {
      if (first == cudaSuccess) first = e;
      (void)cudaGetLastError();
      cudaEventDestroy(r.start);
      cudaEventDestroy(r.stop);
      continue;
    }
    c->total_ms[r.kind] += ms;
    c->total_launches[r.kind] += 1;
    c->total_elements[r.kind] += r.elements;
    c->pool.push_back(r.start);
    c->pool.push_back(r.stop);
  }
  c->pending.clear();
  return first == cudaSuccess ? ZS_OK : cuda_fail(c, first, "timing events");
}

zs_status zs_ctx_timing(zs_ctx* c, int32_t kind, double* total_ms, int64_t* launches,
                        int64_t* elements) {
  if (c == nullptr || kind < 0 || kind >= ZS_KERNEL_KINDS) return ZS_ERR_ARG;
  ZS_TRY(drain_timing(c));
  if (total_ms) *total_ms = c->total_ms[kind];
  if (launches) *launches = c->total_launches[kind];
  if (elements) *elements = c->total_elements[kind];
  return ZS_OK;
}

zs_status zs_ctx_timing_reset(zs_ctx* c) {
  if (c == nullptr) return ZS_ERR_ARG;
  ZS_TRY(drain_timing(c));
  for (int k = 0; k < ZS_KERNEL_KINDS; ++k) {
    c->total_ms[k] = 0.0;
    c->total_launches[k] = 0;
    c->total_elements[k] = 0;
  }
  return ZS_OK;
}

zs_status zs_ctx_launch_count(const zs_ctx* c, int64_t* launches) {
  if (c == nullptr || launches == nullptr) return ZS_ERR_ARG;
  *launches = c->launches;
  return ZS_OK;
}

}  // extern "C"

// ---------------------------------------------------------------- allocation-free norm

// Scratch of zs_grad_sumsq_noalloc: one fp64 partial sum per CTA, in static
// device memory (each device that loads the library holds it until exit).
// In host code this name is only a stand-in; kernels get the device address
// looked up below.
static __device__ __align__(256) double zs_noalloc_partials[ZS_NOALLOC_MAX_PARTS];

namespace {

constexpr int kNoallocMaxDevices = 64;
std::mutex g_noalloc_mutex;
// Per device: the scratch's device address and the id of the CUDA context it
// was looked up in.  A device reset (cudaDeviceReset) ends that context and
// the array's address with it; a call under a newer context looks it up again.
struct NoallocSlot {
  double* scratch = nullptr;
  unsigned long long ctx_id = 0;
};
NoallocSlot g_noalloc[kNoallocMaxDevices];

typedef int (*CtxGetCurrentFn)(void** ctx);
typedef int (*CtxGetIdFn)(void* ctx, unsigned long long* id);

// Id of the calling thread's current CUDA context (0 if none), through the
// driver entry points the runtime hands out (no link against the driver).
unsigned long long current_ctx_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(f);
  });
  void* c = nullptr;
  unsigned long long id = 0;
  if (get_current == nullptr || get_id == nullptr || get_current(&c) != 0 || c == nullptr ||
      get_id(c, &id) != 0)
    return 0;
  return id;
}

template <int DT, bool HA, bool RC>
cudaError_t preload_sumsq() {
  cudaFuncAttributes a;
  return cudaFuncGetAttributes(&a, zs::k_sumsq<DT, HA, RC>);
}

// Set-up, once per device (and again after a device reset), with that device
// current: the static scratch's device address, and every kernel this entry
// point launches loaded now (under lazy module loading a kernel is otherwise
// loaded, taking device memory, at its first launch).
cudaError_t noalloc_scratch(double** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kNoallocMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  NoallocSlot& slot = g_noalloc[dev];
  if (slot.scratch == nullptr || slot.ctx_id != current_ctx_id()) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, zs_noalloc_partials);
    if (e != cudaSuccess) return e;
    const cudaError_t loads[] = {
        preload_sumsq<ZS_FP16, true, true>(), preload_sumsq<ZS_FP16, false, true>(),
        preload_sumsq<ZS_FP16, true, false>(), preload_sumsq<ZS_BF16, true, true>(),
        preload_sumsq<ZS_BF16, false, true>(), preload_sumsq<ZS_BF16, true, false>()};
    for (cudaError_t le : loads)
      if (le != cudaSuccess) return le;
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, zs::k_sumsq_finalize);
    if (e != cudaSuccess) return e;
    slot.scratch = static_cast<double*>(p);
    slot.ctx_id = current_ctx_id();  // the context the lookup ran in
  }
  *out = slot.scratch;
  return cudaSuccess;
}

template <int DT, bool HA, bool RC>
void launch_sumsq_noalloc(const zs::SlicePtrs& sp, int32_t n, const float* acc, int64_t count,
                          double* partials, int grid, cudaStream_t s) {
  zs::k_sumsq<DT, HA, RC><<<grid, zs::kThreads, 0, s>>>(sp, n, acc, count, partials);
}

}  // namespace

extern "C" zs_status zs_grad_sumsq_noalloc(const void* const* grads, int32_t n, zs_dtype dt,
                                           const float* acc, int64_t count, float grad_div,
                                           double* d_sumsq, cudaStream_t stream) {
  if (count < 0) return ZS_ERR_ARG;
  if (count > ZS_NOALLOC_MAX_COUNT) return ZS_ERR_LIMIT;
  if (dt != ZS_FP16 && dt != ZS_BF16) return ZS_ERR_DTYPE;
  if (d_sumsq == nullptr || !(grad_div > 0.0f) || !std::isfinite(grad_div)) return ZS_ERR_ARG;
  if (!aligned16(acc) || !aligned16(d_sumsq)) return ZS_ERR_ALIGN;
  zs::SlicePtrs sp;
  std::memset(&sp, 0, sizeof sp);
  const bool recompute = grads != nullptr;
  if (recompute) {
    if (n < 1 || n > ZS_MAX_RANKS) return ZS_ERR_ARG;
    for (int r = 0; r < n; ++r) {
      if (count > 0 && grads[r] == nullptr) return ZS_ERR_ARG;
      if (!aligned16(grads[r])) return ZS_ERR_ALIGN;
      sp.p[r] = static_cast<const uint4*>(grads[r]);
    }
  } else if (count > 0 && acc == nullptr) {
    return ZS_ERR_ARG;
  }
  // an error left pending by earlier work is the caller's: report it, leave it set
  if (cudaPeekAtLastError() != cudaSuccess) return ZS_ERR_CUDA;
  double* partials = nullptr;
  if (noalloc_scratch(&partials) != cudaSuccess) return ZS_ERR_CUDA;
  // one CTA (and one partial) per ZS_NOALLOC_ELEMS_PER_PART elements: each
  // thread takes ZS_NOALLOC_ELEMS_PER_PART / (8 * kThreads) vector units
  int64_t grid64 = (count + ZS_NOALLOC_ELEMS_PER_PART - 1) / ZS_NOALLOC_ELEMS_PER_PART;
  if (grid64 < 1) grid64 = 1;
  const int grid = (int)grid64;  // <= ZS_NOALLOC_MAX_PARTS by the count limit
  const int nn = recompute ? n : 0;
  const bool ha = acc != nullptr;
  if (dt == ZS_FP16) {
    if (recompute && ha) launch_sumsq_noalloc<ZS_FP16, true, true>(sp, nn, acc, count, partials, grid, stream);
    else if (recompute) launch_sumsq_noalloc<ZS_FP16, false, true>(sp, nn, acc, count, partials, grid, stream);
    else launch_sumsq_noalloc<ZS_FP16, true, false>(sp, nn, acc, count, partials, grid, stream);
  } else {
    if (recompute && ha) launch_sumsq_noalloc<ZS_BF16, true, true>(sp, nn, acc, count, partials, grid, stream);
    else if (recompute) launch_sumsq_noalloc<ZS_BF16, false, true>(sp, nn, acc, count, partials, grid, stream);
    else launch_sumsq_noalloc<ZS_BF16, true, false>(sp, nn, acc, count, partials, grid, stream);
  }
  const double div = (double)grad_div;
  zs::k_sumsq_finalize<<<1, zs::kThreads, 0, stream>>>(partials, grid, 1.0 / (div * div), d_sumsq);
  return cudaGetLastError() == cudaSuccess ? ZS_OK : ZS_ERR_CUDA;
}
