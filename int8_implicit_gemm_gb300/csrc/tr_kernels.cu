// Transposed-tile kernel (output channels on the MMA's M, pixels on N) on
// single CTAs.
#include "tr_launch.cuh"

namespace i8c {

cudaError_t tr_prepare() { return tr_prepare_cg<1>(); }

cudaError_t tr_launch(const CUtensorMap& tmap, const CUtensorMap& tmap_x, const HaloParams& p, int smem, int num_ctas, cudaStream_t stream) {
  return tr_launch_cg<1>(tmap, tmap_x, p, smem, num_ctas, stream);
}

}  // namespace i8c
