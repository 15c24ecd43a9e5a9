// The stacked-tap kernel for 64-output-channel layers (conv_fprop_stack.cuh):
// its filter conversion, shared-memory set-up and launch.
#include <cuda_fp16.h>

#include "conv_fprop_stack.cuh"
#include "halo_launch.cuh"

namespace i8c {

// CxRSKx<32> int8 filter (K = 64) -> the stacked kernel's fp16 operand order
// [32-channel block cb][filter row r][rank][slot u][64 rows][32 channels]:
// rank 0's slot u holds tap s = 2u (its 64 output channels as rows), rank 1's
// slot u tap s = 2u + 1; for an odd last tap (2u + 1 = S) rank 1's slot holds
// that tap's output channels 32-63 in rows 0-31 and zeros below, so that the
// N = 64 MMA over both CTAs' first 32 rows sees all 64 channels.  One thread
// step converts one 16-channel half row.
__global__ void filter_to_f16_stacked_kernel(const int8_t* __restrict__ f, uint16_t* __restrict__ out, int R,
                                             int S, int U, int64_t vecs) {
  ptx::griddep_launch_dependents();
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < vecs;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int half = static_cast<int>(i & 1);
    int64_t rest = i >> 1;
    const int row = static_cast<int>(rest & 63);
    rest >>= 6;
    const int u = static_cast<int>(rest % U);
    rest /= U;
    const int rank = static_cast<int>(rest & 1);
    rest >>= 1;
    const int r = static_cast<int>(rest % R);
    const int64_t cb = rest / R;
    int s = 2 * u + rank, k = row;
    if (s >= S) {  // rank 1 of an odd last tap: channels 32-63 in the first 32 rows
      s = S - 1;
      k = row < 32 ? row + 32 : -1;
    }
    uint32_t w[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (k >= 0) {
      const int4 v = *reinterpret_cast<const int4*>(f + ((((cb * R + r) * S + s) * 64 + k) * 32 + half * 16));
      const int8_t* b = reinterpret_cast<const int8_t*>(&v);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const __half lo = __int2half_rn(b[2 * j]);
        const __half hi = __int2half_rn(b[2 * j + 1]);
        w[j] = static_cast<uint32_t>(__half_as_ushort(lo)) | (static_cast<uint32_t>(__half_as_ushort(hi)) << 16);
      }
    }
    int4* dst = reinterpret_cast<int4*>(out) + 2 * i;
    dst[0] = make_int4(w[0], w[1], w[2], w[3]);
    dst[1] = make_int4(w[4], w[5], w[6], w[7]);
  }
}

cudaError_t launch_filter_to_f16_stacked(const int8_t* f, uint16_t* f16, int CB, int R, int S, cudaStream_t stream) {
  const int U = (S + 1) / 2;
  const int64_t vecs = static_cast<int64_t>(CB) * R * 2 * U * 64 * 2;
  const int threads = 256;
  int64_t blocks = (vecs + threads - 1) / threads;
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) blocks = 1;
  filter_to_f16_stacked_kernel<<<static_cast<int>(blocks), threads, 0, stream>>>(f, f16, R, S, U, vecs);
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return cudaGetLastError();
}

using StackKernel = void (*)(const CUtensorMap, const CUtensorMap, const HaloParams);

// One instantiation per tap-pair count ceil(S/2) = 1 .. 8.
StackKernel stack_kernel_for(int slots) {
  switch (slots) {
    case 1: return conv_fprop_stack_kernel<1>;
    case 2: return conv_fprop_stack_kernel<2>;
    case 3: return conv_fprop_stack_kernel<3>;
    case 4: return conv_fprop_stack_kernel<4>;
    case 5: return conv_fprop_stack_kernel<5>;
    case 6: return conv_fprop_stack_kernel<6>;
    case 7: return conv_fprop_stack_kernel<7>;
    default: return conv_fprop_stack_kernel<8>;
  }
}

cudaError_t stack_prepare() {
  for (int u = 1; u <= kStackMaxSlots; ++u) {
    const cudaError_t e =
        cudaFuncSetAttribute(stack_kernel_for(u), cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynamicSmem);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// Launched like the halo kernel on pairs: clusters of two, a programmatic
// dependent of the filter conversion.
cudaError_t stack_launch(const CUtensorMap& tmap, const CUtensorMap& tmap_x, const HaloParams& p, int smem,
                         int num_ctas, cudaStream_t stream) {
  cudaLaunchAttribute attr[2];
  const cudaLaunchConfig_t cfg = halo_launch_config<2>(smem, num_ctas, stream, attr);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, stack_kernel_for(p.slots), tmap, tmap_x, p);
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return e != cudaSuccess ? e : cudaGetLastError();
}

int stack_max_clusters(int slots, int smem) {
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = halo_launch_config<2>(smem, 2, nullptr, attr);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void*>(stack_kernel_for(slots)), &cfg) !=
      cudaSuccess)
    return 0;
  return n;
}

}  // namespace i8c
