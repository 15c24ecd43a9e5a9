// Instantiations and launch of the per-tap gather kernel per tile width.
#include "internal.h"

namespace i8c {

std::atomic<int64_t> g_launches{0};

int conv_smem_bytes(int block_n) {
  switch (block_n) {
    case 32: return TileCfg<32>::kSmemBytes;
    case 64: return TileCfg<64>::kSmemBytes;
    case 128: return TileCfg<128>::kSmemBytes;
    case 256: return TileCfg<256>::kSmemBytes;
    default: return -1;
  }
}

template <int BN>
static cudaError_t prepare_one() {
  return cudaFuncSetAttribute(conv_fprop_tc_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              TileCfg<BN>::kSmemBytes);
}

cudaError_t conv_prepare(int block_n) {
  switch (block_n) {
    case 32: return prepare_one<32>();
    case 64: return prepare_one<64>();
    case 128: return prepare_one<128>();
    case 256: return prepare_one<256>();
    default: return cudaErrorInvalidValue;
  }
}

template <int BN>
static cudaError_t launch_one(const CUtensorMap& tmap, const ConvParams& p, int num_ctas, cudaStream_t stream) {
  conv_fprop_tc_kernel<BN><<<num_ctas, TileCfg<BN>::kThreads, TileCfg<BN>::kSmemBytes, stream>>>(tmap, p);
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return cudaGetLastError();
}

cudaError_t launch_conv(int block_n, const CUtensorMap& tmap, const ConvParams& p, int num_ctas,
                        cudaStream_t stream) {
  switch (block_n) {
    case 32: return launch_one<32>(tmap, p, num_ctas, stream);
    case 64: return launch_one<64>(tmap, p, num_ctas, stream);
    case 128: return launch_one<128>(tmap, p, num_ctas, stream);
    case 256: return launch_one<256>(tmap, p, num_ctas, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace i8c
