// Transposed-tile kernel (output channels on the MMA's M, pixels on N):
// shared-memory set-up and launch.
#include "conv_fprop_tr.cuh"
#include "halo_launch.cuh"

namespace i8c {

using TrKernel = void (*)(const CUtensorMap, const HaloParams);

// Stages of 9 whole-row taps (a 3x3 channel block, three rows of a 1x3
// filter, a row of a 9-wide one) take the unrolled instantiation; tiles of
// at most 192 pixels the one with the larger producer register budget.
TrKernel tr_kernel_for(int bgroup, int S, int tile_px) {
  const bool t9 = bgroup == 9 && 9 % S == 0;
  if (tile_px <= 192) return t9 ? conv_fprop_tr_kernel<9, 192> : conv_fprop_tr_kernel<0, 192>;
  return t9 ? conv_fprop_tr_kernel<9, 256> : conv_fprop_tr_kernel<0, 256>;
}

cudaError_t tr_prepare() {
  for (TrKernel k : {conv_fprop_tr_kernel<9, 192>, conv_fprop_tr_kernel<0, 192>, conv_fprop_tr_kernel<9, 256>,
                     conv_fprop_tr_kernel<0, 256>}) {
    const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynamicSmem);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// Launched like the single-CTA halo kernel: a programmatic dependent of the
// filter conversion, whose tail its prologue overlaps.
cudaError_t tr_launch(const CUtensorMap& tmap, const HaloParams& p, int smem, int num_ctas, cudaStream_t stream) {
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t cfg = halo_launch_config<1>(smem, num_ctas, stream, attr);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, tr_kernel_for(p.bgroup, p.c.S, p.tile_px), tmap, p);
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace i8c
