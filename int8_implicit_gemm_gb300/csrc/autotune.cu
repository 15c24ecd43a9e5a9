// Plan selection by measurement: times a fixed list of candidate plans of
// one convolution on the caller's own tensors and returns the options of the
// fastest.
//
// This is the search step of the "[BYOC] CUTLASS integration" pull request
// (apache/tvm #9261, the profiler renamed tune_cutlass_kernels in its review):
// candidate kernel configurations are built and timed on the device, the
// fastest is kept, and a default configuration remains available without
// tuning.  Here the default is i8c_plan_create's own choice (zeroed options),
// which is always the first candidate, so the result is never slower than
// the default on the measured inputs.  The torchao W4A8 issue's review
// (pytorch/ao #1406, on finding good configurations) notes that a sweep like
// this is what a cheap host-side selection rule is fitted to.
//
// Built only on the public entry points: i8c_plan_create / i8c_plan_run /
// i8c_plan_status / i8c_plan_destroy and CUDA events on the caller's stream.
#include <cuda_runtime.h>

#include <vector>

#include "i8conv.h"

namespace {

i8c_options make(int variant, int block_n, int tile_shape, int tile_px) {
  i8c_options o{};
  o.kernel_variant = variant;
  o.block_n = block_n;
  o.tile_shape = tile_shape;
  o.tile_px = tile_px;
  return o;
}

// The candidates, default first.  Options a shape cannot use (a halo that
// does not fit, transposed tiles on a strided layer, ...) fail in
// i8c_plan_create and are recorded as such.
std::vector<i8c_options> candidate_list() {
  std::vector<i8c_options> c;
  c.push_back(make(0, 0, 0, 0));  // i8c_plan_create's own choice
  c.push_back(make(1, 0, 0, 0));  // per-tap gather kernel
  for (int bn : {0, 64, 128, 256}) {
    c.push_back(make(2, bn, 1, 0));  // halo kernel, 16x8 patches
    c.push_back(make(2, bn, 2, 0));  // halo kernel, flat tiles
    c.push_back(make(3, bn, 0, 0));  // halo kernel on CTA pairs
  }
  for (int px : {0, 96, 128, 144, 160, 176, 192, 208, 224, 240, 256}) c.push_back(make(4, 0, 0, px));
  for (int px : {0, 128, 160, 192, 224, 240, 256}) c.push_back(make(5, 0, 0, px));
  return c;
}

i8c_status from_cuda(cudaError_t e) { return e == cudaSuccess ? I8C_OK : I8C_ERR_CUDA; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Mean device time of one run over `iters` runs after two warm-up runs.
i8c_status time_plan(const i8c_plan* plan, const int8_t* x, const int8_t* f, int8_t* y, float alpha, int iters,
                     cudaStream_t stream, cudaEvent_t e0, cudaEvent_t e1, float* us) {
  i8c_status st = I8C_OK;
  for (int i = 0; i < 2 && st == I8C_OK; ++i) st = i8c_plan_run(plan, x, f, y, alpha, stream);
  if (st != I8C_OK) return st;
  cudaError_t e = cudaEventRecord(e0, stream);
  if (e != cudaSuccess) return from_cuda(e);
  for (int i = 0; i < iters && st == I8C_OK; ++i) st = i8c_plan_run(plan, x, f, y, alpha, stream);
  if (st != I8C_OK) return st;
  e = cudaEventRecord(e1, stream);
  if (e == cudaSuccess) e = cudaEventSynchronize(e1);
  float ms = 0.0f;
  if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
  if (e != cudaSuccess) return from_cuda(e);
  // a bounded wait that ran out in any of the runs disqualifies the candidate
  st = i8c_plan_status(plan, stream);
  if (st != I8C_OK) return st;
  *us = ms * 1000.0f / static_cast<float>(iters);
  return I8C_OK;
}

}  // namespace

extern "C" i8c_status i8c_plan_autotune(const i8c_conv_shape* shape, const int8_t* x, const int8_t* f, int8_t* y,
                                        float alpha, int32_t iters, cudaStream_t stream, i8c_options* best,
                                        float* best_us, i8c_tune_entry* entries, int32_t max_entries,
                                        int32_t* num_entries) {
  if (shape == nullptr || x == nullptr || f == nullptr || y == nullptr || best == nullptr || best_us == nullptr)
    return I8C_ERR_INVALID_ARG;
  if (iters < 1 || max_entries < 0 || (max_entries > 0 && entries == nullptr)) return I8C_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(f) || !aligned16(y)) return I8C_ERR_MISALIGNED;
  i8c_status st = i8c_supported(shape);
  if (st != I8C_OK) return st;
  if (num_entries != nullptr) *num_entries = 0;

  cudaEvent_t e0 = nullptr, e1 = nullptr;
  cudaError_t e = cudaEventCreate(&e0);
  if (e == cudaSuccess) e = cudaEventCreate(&e1);
  if (e != cudaSuccess) {
    if (e0 != nullptr) cudaEventDestroy(e0);
    return from_cuda(e);
  }

  i8c_plan* kept = nullptr;  // the fastest plan so far, run once more at the end
  float kept_us = 0.0f;
  i8c_status first_status = I8C_OK;
  const std::vector<i8c_options> cands = candidate_list();
  int32_t n = 0;
  for (size_t i = 0; i < cands.size(); ++i) {
    i8c_plan* plan = nullptr;
    float us = 0.0f;
    st = i8c_plan_create(shape, &cands[i], &plan);
    if (st == I8C_OK) st = time_plan(plan, x, f, y, alpha, iters, stream, e0, e1, &us);
    if (i == 0) first_status = st;
    if (n < max_entries) entries[n] = i8c_tune_entry{cands[i], static_cast<int32_t>(st), st == I8C_OK ? us : 0.0f};
    ++n;
    if (st == I8C_OK && (kept == nullptr || us < kept_us)) {
      if (kept != nullptr) i8c_plan_destroy(kept);
      kept = plan;
      kept_us = us;
      *best = cands[i];
    } else if (plan != nullptr) {
      i8c_plan_destroy(plan);
    }
    // a CUDA error that the device reports again after a synchronisation
    // (a sticky one) leaves nothing to time: stop and report it
    if (st == I8C_ERR_CUDA) {
      cudaGetLastError();
      if (cudaDeviceSynchronize() != cudaSuccess) break;
      st = I8C_OK;
    }
  }
  if (num_entries != nullptr) *num_entries = n < max_entries ? n : max_entries;

  if (kept == nullptr) {
    st = st == I8C_ERR_CUDA ? st : first_status;
  } else if (st == I8C_ERR_CUDA) {
    i8c_plan_destroy(kept);
  } else {
    *best_us = kept_us;
    // y ends up holding the chosen plan's result
    st = i8c_plan_run(kept, x, f, y, alpha, stream);
    if (st == I8C_OK) st = i8c_plan_status(kept, stream);
    i8c_plan_destroy(kept);
  }
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  return st;
}
