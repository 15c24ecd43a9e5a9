// Halo kernel on CTA pairs (clusters of two, M = 256 MMAs), tile widths 64-256.
#include "halo_launch.cuh"

namespace i8c {

cudaError_t halo_prepare_pair(int block_n) {
  switch (block_n) {
    case 64: return halo_prepare_bn<64, 2>();
    case 128: return halo_prepare_bn<128, 2>();
    case 256: return halo_prepare_bn<256, 2>();
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t halo_launch_pair(int block_n, const CUtensorMap& tmap, const CUtensorMap& tmap_x, const HaloParams& p, int smem, int num_ctas,
                             cudaStream_t stream) {
  switch (block_n) {
    case 64: return halo_launch_bn<64, 2>(tmap, tmap_x, p, smem, num_ctas, stream);
    case 128: return halo_launch_bn<128, 2>(tmap, tmap_x, p, smem, num_ctas, stream);
    case 256: return halo_launch_bn<256, 2>(tmap, tmap_x, p, smem, num_ctas, stream);
    default: return cudaErrorInvalidValue;
  }
}

int halo_pair_max_clusters(int block_n, int bgroup, int S, int smem) {
  switch (block_n) {
    case 64: return halo_max_clusters_bn<64>(bgroup, S, smem);
    case 128: return halo_max_clusters_bn<128>(bgroup, S, smem);
    case 256: return halo_max_clusters_bn<256>(bgroup, S, smem);
    default: return 0;
  }
}

}  // namespace i8c
