// Instantiation, shared-memory set-up and launch of the transposed-tile
// kernel for one CTA-group size (included by one translation unit per size,
// so that the two sets of instantiations compile in parallel).
#pragma once

#include "conv_fprop_tr.cuh"
#include "halo_launch.cuh"

namespace i8c {

using TrKernel = void (*)(const CUtensorMap, const CUtensorMap, const HaloParams);

// Stages of 9 whole-row taps (a 3x3 channel block, three rows of a 1x3
// filter, a row of a 9-wide one) take the unrolled instantiation; MMAs of at
// most 192 columns the one with the larger producer register budget.
template <int CG>
TrKernel tr_kernel_for(int bgroup, int S, int mma_n) {
  const bool t9 = bgroup == 9 && 9 % S == 0;
  if (mma_n <= 192) return t9 ? conv_fprop_tr_kernel<9, 192, CG> : conv_fprop_tr_kernel<0, 192, CG>;
  return t9 ? conv_fprop_tr_kernel<9, 256, CG> : conv_fprop_tr_kernel<0, 256, CG>;
}

template <int CG>
cudaError_t tr_prepare_cg() {
  for (TrKernel k : {conv_fprop_tr_kernel<9, 192, CG>, conv_fprop_tr_kernel<0, 192, CG>,
                     conv_fprop_tr_kernel<9, 256, CG>, conv_fprop_tr_kernel<0, 256, CG>}) {
    const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynamicSmem);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// Launched like the halo kernel: single CTAs as programmatic dependents of
// the filter conversion (their prologue overlaps its tail), pairs as
// clusters of two.
template <int CG>
cudaError_t tr_launch_cg(const CUtensorMap& tmap, const CUtensorMap& tmap_x, const HaloParams& p, int smem,
                         int num_ctas, cudaStream_t stream) {
  cudaLaunchAttribute attr[2];
  const cudaLaunchConfig_t cfg = halo_launch_config<CG>(smem, num_ctas, stream, attr);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, tr_kernel_for<CG>(p.bgroup, p.c.S, CG * p.tile_px), tmap, tmap_x, p);
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace i8c
