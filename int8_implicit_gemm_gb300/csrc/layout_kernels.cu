// Layout kernels: int8 filter -> fp16 operand copy (part of every run), and
// the NCHW <-> NCxHWx<32> / KCRS <-> CxRSKx<32> pack helpers (not timed).
#include <cuda_fp16.h>

#include "internal.h"

namespace i8c {

// CxRSKx<32> int8 -> the same layout in fp16 (the tensor-core operand type).
// 16 int8 in, 16 fp16 out per thread step; count is a multiple of 32.
__global__ void filter_to_f16_kernel(const int8_t* __restrict__ f, uint16_t* __restrict__ out, int64_t vecs) {
  // the convolution kernel that follows waits for this grid's completion
  // before it reads the converted filter; it may launch right away
  ptx::griddep_launch_dependents();
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < vecs;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int4 v = reinterpret_cast<const int4*>(f)[i];
    const int8_t* b = reinterpret_cast<const int8_t*>(&v);
    uint32_t w[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const __half lo = __int2half_rn(b[2 * j]);
      const __half hi = __int2half_rn(b[2 * j + 1]);
      w[j] = static_cast<uint32_t>(__half_as_ushort(lo)) | (static_cast<uint32_t>(__half_as_ushort(hi)) << 16);
    }
    int4* dst = reinterpret_cast<int4*>(out) + 2 * i;
    dst[0] = make_int4(w[0], w[1], w[2], w[3]);
    dst[1] = make_int4(w[4], w[5], w[6], w[7]);
  }
}

cudaError_t launch_filter_to_f16(const int8_t* f, uint16_t* f16, int64_t count, cudaStream_t stream) {
  const int64_t vecs = count / 16;
  const int threads = 256;
  int64_t blocks = (vecs + threads - 1) / threads;
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) blocks = 1;
  static const cudaError_t carveout = cudaFuncSetAttribute(
      filter_to_f16_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  (void)carveout;  // a preference only: the kernel runs either way
  filter_to_f16_kernel<<<static_cast<int>(blocks), threads, 0, stream>>>(f, f16, vecs);
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return cudaGetLastError();
}

// Activations.  Interleaved offset of (n, c, h, w):
//   (((n*C/32 + c/32)*H + h)*W + w)*32 + c%32.
__global__ void pack_act_kernel(const int8_t* __restrict__ src, int8_t* __restrict__ dst, int N, int C, int H, int W,
                                bool to_interleaved) {
  const int64_t total = static_cast<int64_t>(N) * C * H * W;
  const int64_t HW = static_cast<int64_t>(H) * W;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    // i enumerates the interleaved layout
    const int c32 = static_cast<int>(i & 31);
    int64_t t = i >> 5;
    const int64_t hw = t % HW;
    t /= HW;
    const int cb = static_cast<int>(t % (C / 32));
    const int64_t n = t / (C / 32);
    const int64_t plain = (n * C + cb * 32 + c32) * HW + hw;
    if (to_interleaved) dst[i] = src[plain];
    else dst[plain] = src[i];
  }
}

// Filters.  Interleaved offset of (k, c, r, s):
//   ((((c/32)*R + r)*S + s)*K + k)*32 + c%32.
__global__ void pack_filter_kernel(const int8_t* __restrict__ src, int8_t* __restrict__ dst, int K, int C, int R,
                                   int S, bool to_interleaved) {
  const int64_t total = static_cast<int64_t>(K) * C * R * S;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int c32 = static_cast<int>(i & 31);
    int64_t t = i >> 5;
    const int k = static_cast<int>(t % K);
    t /= K;
    const int s = static_cast<int>(t % S);
    t /= S;
    const int r = static_cast<int>(t % R);
    const int cb = static_cast<int>(t / R);
    const int64_t plain = ((static_cast<int64_t>(k) * C + cb * 32 + c32) * R + r) * S + s;
    if (to_interleaved) dst[i] = src[plain];
    else dst[plain] = src[i];
  }
}

static int grid_for(int64_t total) {
  int64_t b = (total + 255) / 256;
  if (b > 8192) b = 8192;
  if (b < 1) b = 1;
  return static_cast<int>(b);
}

cudaError_t launch_pack_act(const int8_t* src, int8_t* dst, int N, int C, int H, int W, bool to_interleaved,
                            cudaStream_t stream) {
  const int64_t total = static_cast<int64_t>(N) * C * H * W;
  pack_act_kernel<<<grid_for(total), 256, 0, stream>>>(src, dst, N, C, H, W, to_interleaved);
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return cudaGetLastError();
}

cudaError_t launch_pack_filter(const int8_t* src, int8_t* dst, int K, int C, int R, int S, bool to_interleaved,
                               cudaStream_t stream) {
  const int64_t total = static_cast<int64_t>(K) * C * R * S;
  pack_filter_kernel<<<grid_for(total), 256, 0, stream>>>(src, dst, K, C, R, S, to_interleaved);
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return cudaGetLastError();
}

}  // namespace i8c
