// Transposed-tile kernel on CTA pairs (M = 256 MMAs over two CTAs' 128
// output channels each, the N pixels split between their halos).
#include "tr_launch.cuh"

namespace i8c {

cudaError_t tr_prepare_pair() { return tr_prepare_cg<2>(); }

cudaError_t tr_launch_pair(const CUtensorMap& tmap, const CUtensorMap& tmap_x, const HaloParams& p, int smem, int num_ctas,
                           cudaStream_t stream) {
  return tr_launch_cg<2>(tmap, tmap_x, p, smem, num_ctas, stream);
}

// Clusters of two that can be resident at once (0 if the query fails).
int tr_pair_max_clusters(int bgroup, int S, int mma_n, int smem) {
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = halo_launch_config<2>(smem, 2, nullptr, attr);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void*>(tr_kernel_for<2>(bgroup, S, mma_n)), &cfg) !=
      cudaSuccess)
    return 0;
  return n;
}

}  // namespace i8c
