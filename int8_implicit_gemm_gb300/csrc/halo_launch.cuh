// Instantiation, shared-memory set-up and launch of the halo kernel for one
// CTA-group size (included by one translation unit per size, so that the two
// sets of instantiations compile in parallel).
#pragma once

#include "internal.h"

namespace i8c {

using HaloKernel = void (*)(const CUtensorMap, const CUtensorMap, const HaloParams);

// Run lengths with an unrolled tap loop and precomputed tap offsets, for runs
// of whole filter rows (S divides the run length): 3 (a row of a 3x3
// filter) and 9 (a whole 3x3 channel block, or a row of a 9-wide filter);
// every other run takes the generic instantiation (GT = 0).
// 16x16 patches (subtiles 2; whole-row runs and BN <= 128 only) have
// instantiations of their own, so that the 16x8 kernels compile as before.
template <int BN, int CG>
HaloKernel halo_kernel_for(int bgroup, int S, int subtiles = 1) {
  if constexpr (BN <= 128) {
    if (subtiles == 2) {
      if (bgroup == 3 && 3 % S == 0) return conv_fprop_halo_kernel<BN, 3, CG, 2>;
      if (bgroup == 9 && 9 % S == 0) return conv_fprop_halo_kernel<BN, 9, CG, 2>;
    }
  }
  if (bgroup == 3 && 3 % S == 0) return conv_fprop_halo_kernel<BN, 3, CG>;
  if (bgroup == 9 && 9 % S == 0) return conv_fprop_halo_kernel<BN, 9, CG>;
  return conv_fprop_halo_kernel<BN, 0, CG>;
}

template <int BN, int CG>
cudaError_t halo_prepare_bn() {
  for (int sub : {1, 2})
    for (int g : {3, 9, 0}) {
      const cudaError_t e = cudaFuncSetAttribute(halo_kernel_for<BN, CG>(g, 1, sub),
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynamicSmem);
      if (e != cudaSuccess) return e;
    }
  return cudaSuccess;
}

// CTA pairs are launched as clusters of two.  Single CTAs that convert the
// filter themselves are launched cooperatively (all CTAs resident: their grid
// barrier cannot wait on a CTA that has not started).  Otherwise (pairs too)
// the kernel is a programmatic dependent of the filter conversion kernel,
// whose tail its prologue (barriers, tensor memory, halo loads) overlaps.
// attr: room for two attributes.
template <int CG>
cudaLaunchConfig_t halo_launch_config(int smem, int num_ctas, cudaStream_t stream, cudaLaunchAttribute* attr,
                                      bool cooperative = false) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(num_ctas));
  cfg.blockDim = dim3(kHaloThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  unsigned n = 0;
  if (CG == 2) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = 2;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  if (cooperative) {
    attr[n].id = cudaLaunchAttributeCooperative;
    attr[n].val.cooperative = 1;
  } else {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
  }
  ++n;
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cfg;
}

template <int BN, int CG>
cudaError_t halo_launch_bn(const CUtensorMap& tmap, const CUtensorMap& tmap_x, const HaloParams& p, int smem,
                           int num_ctas, cudaStream_t stream) {
  cudaLaunchAttribute attr[2];
  const cudaLaunchConfig_t cfg = halo_launch_config<CG>(smem, num_ctas, stream, attr, p.f_int8 != nullptr);
  const cudaError_t e =
      cudaLaunchKernelEx(&cfg, halo_kernel_for<BN, CG>(p.bgroup, p.c.S, p.subtiles), tmap, tmap_x, p);
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// Clusters of two that can be resident at once (0 if the query fails).
template <int BN>
int halo_max_clusters_bn(int bgroup, int S, int smem) {
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = halo_launch_config<2>(smem, 2, nullptr, attr);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void*>(halo_kernel_for<BN, 2>(bgroup, S)), &cfg) !=
      cudaSuccess)
    return 0;
  return n;
}

// CTAs of one kernel instance that fit on the GPU at once (0 if the query fails).
template <int BN>
int halo_max_ctas_bn(int bgroup, int S, int smem) {
  int per_sm = 0, dev = 0, sms = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, halo_kernel_for<BN, 1>(bgroup, S), kHaloThreads,
                                                    static_cast<size_t>(smem)) != cudaSuccess ||
      cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  return per_sm * sms;
}

}  // namespace i8c
