// Internal interfaces between the library's translation units (not exported).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "conv_fprop_halo.cuh"
#include "conv_fprop_tc.cuh"

namespace i8c {

extern std::atomic<int64_t> g_launches;

// conv_kernels.cu
int conv_smem_bytes(int block_n);
cudaError_t conv_prepare(int block_n);  // raise the dynamic shared memory limit
cudaError_t launch_conv(int block_n, const CUtensorMap& tmap, const ConvParams& p, int num_ctas,
                        cudaStream_t stream);

// halo_kernels_single.cu / halo_kernels_pair.cu: the halo kernel on single
// CTAs and on CTA pairs (clusters of two); prepare allows the full dynamic
// shared memory, max_clusters is the number of pairs that fit at once.
cudaError_t halo_prepare_single(int block_n);
cudaError_t halo_launch_single(int block_n, const CUtensorMap& tmap, const CUtensorMap& tmap_x, const HaloParams& p,
                               int smem_bytes,
                               int num_ctas, cudaStream_t stream);
cudaError_t halo_prepare_pair(int block_n);
cudaError_t halo_launch_pair(int block_n, const CUtensorMap& tmap, const CUtensorMap& tmap_x, const HaloParams& p,
                             int smem_bytes,
                             int num_ctas, cudaStream_t stream);
int halo_pair_max_clusters(int block_n, int bgroup, int S, int smem_bytes);
int halo_single_max_ctas(int block_n, int bgroup, int S, int smem_bytes);  // resident at once

// tr_kernels.cu: the transposed-tile kernel (128 output channels x tile_px
// pixels per tile, stride-1 layers)
cudaError_t tr_prepare();
cudaError_t tr_launch(const CUtensorMap& tmap, const CUtensorMap& tmap_x, const HaloParams& p, int smem_bytes,
                      int num_ctas,
                      cudaStream_t stream);
// tr_kernels_pair.cu: the same on CTA pairs (clusters of two; tile_px is each
// CTA's half of the MMA's N); max_clusters is the number of pairs that fit
cudaError_t tr_prepare_pair();
cudaError_t tr_launch_pair(const CUtensorMap& tmap, const CUtensorMap& tmap_x, const HaloParams& p, int smem_bytes,
                           int num_ctas,
                           cudaStream_t stream);
int tr_pair_max_clusters(int bgroup, int S, int mma_n, int smem_bytes);
constexpr int kMaxDynamicSmem = 232448;

// stack_kernels.cu: the stacked-tap kernel for 64-output-channel layers (two
// filter taps per N = 128 MMA, CTA pairs) and its filter conversion into the
// stacked fp16 order
cudaError_t stack_prepare();
cudaError_t stack_launch(const CUtensorMap& tmap, const CUtensorMap& tmap_x, const HaloParams& p, int smem_bytes,
                         int num_ctas,
                         cudaStream_t stream);
int stack_max_clusters(int slots, int smem_bytes);
cudaError_t launch_filter_to_f16_stacked(const int8_t* f, uint16_t* f16, int CB, int R, int S, cudaStream_t stream);
constexpr int kStackXbufBytes = 2 * 8 * 8 * 32 * 4;  // the epilogue's shift buffers (two tiles)

// noalloc.cu: the no-allocation entry point's status word on device `dev`
// (synchronous; I8C_OK if that entry point has not run there), cleared once
// read; and the one-shot test hooks (debug flags, bounded-wait limit in us).
int noalloc_take_status(int dev);
void noalloc_set_debug(int debug_flags, int timeout_us);

// layout_kernels.cu
cudaError_t launch_filter_to_f16(const int8_t* f, uint16_t* f16, int64_t count, cudaStream_t stream);
cudaError_t launch_pack_act(const int8_t* src, int8_t* dst, int N, int C, int H, int W, bool to_interleaved,
                            cudaStream_t stream);
cudaError_t launch_pack_filter(const int8_t* src, int8_t* dst, int K, int C, int R, int S, bool to_interleaved,
                               cudaStream_t stream);

}  // namespace i8c
