// Halo kernel on single CTAs (M = 128 MMAs), tile widths 32-256.
#include "halo_launch.cuh"

namespace i8c {

cudaError_t halo_prepare_single(int block_n) {
  switch (block_n) {
    case 32: return halo_prepare_bn<32, 1>();
    case 64: return halo_prepare_bn<64, 1>();
    case 128: return halo_prepare_bn<128, 1>();
    case 256: return halo_prepare_bn<256, 1>();
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t halo_launch_single(int block_n, const CUtensorMap& tmap, const CUtensorMap& tmap_x, const HaloParams& p, int smem, int num_ctas,
                               cudaStream_t stream) {
  switch (block_n) {
    case 32: return halo_launch_bn<32, 1>(tmap, tmap_x, p, smem, num_ctas, stream);
    case 64: return halo_launch_bn<64, 1>(tmap, tmap_x, p, smem, num_ctas, stream);
    case 128: return halo_launch_bn<128, 1>(tmap, tmap_x, p, smem, num_ctas, stream);
    case 256: return halo_launch_bn<256, 1>(tmap, tmap_x, p, smem, num_ctas, stream);
    default: return cudaErrorInvalidValue;
  }
}

int halo_single_max_ctas(int block_n, int bgroup, int S, int smem) {
  switch (block_n) {
    case 32: return halo_max_ctas_bn<32>(bgroup, S, smem);
    case 64: return halo_max_ctas_bn<64>(bgroup, S, smem);
    case 128: return halo_max_ctas_bn<128>(bgroup, S, smem);
    case 256: return halo_max_ctas_bn<256>(bgroup, S, smem);
    default: return 0;
  }
}

}  // namespace i8c
