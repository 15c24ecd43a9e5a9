// Rates of the two engines the convolution does not use, measured the same
// way as the kind::f16 probe (probes.cu), for the engine choice:
//  - the warp-level integer MMA (mma.sync m16n8k32, s8 x s8 -> s32), the
//    tensor-core path of the Ampere kernels the CUTLASS and TensorRT
//    configurations describe;
//  - tcgen05.mma kind::f8f6f4 with e4m3 operands (M = 128, K = 32), the
//    engine an exact e4m3 nibble split of int8 operands would run on.
// Operands are zeros (finite, and the rates do not depend on the values).
// Not part of the convolution path.
#include "../../include/i8conv_probe.h"
#include "internal.h"

namespace i8c {

// kAcc independent accumulators per warp, so that consecutive MMAs do not
// wait for each other's results.
constexpr int kImmaAcc = 8;

__global__ void __launch_bounds__(512, 1) imma_rate_kernel(int iters, long long* out, int* sink) {
  uint32_t a[4] = {threadIdx.x & 0x7F7F7F7Fu, 0, 0, 0};  // one non-zero lane value keeps the loop live
  uint32_t b[2] = {0, 0};
  int32_t acc[kImmaAcc][4];
#pragma unroll
  for (int j = 0; j < kImmaAcc; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0;
  __syncthreads();
  const long long t0 = clock64();
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int j = 0; j < kImmaAcc; ++j)
      asm volatile(
          "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
          "{%0, %1, %2, %3};"
          : "+r"(acc[j][0]), "+r"(acc[j][1]), "+r"(acc[j][2]), "+r"(acc[j][3])
          : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
  }
  __syncthreads();
  const long long t1 = clock64();
  int s = 0;
#pragma unroll
  for (int j = 0; j < kImmaAcc; ++j) s += acc[j][0] + acc[j][1] + acc[j][2] + acc[j][3];
  if (s == 0x7fffffff) *sink = s;  // never true (b is zero): keeps the accumulators live
  if (threadIdx.x == 0) {
    out[3 * blockIdx.x + 0] = t1 - t0;
    out[3 * blockIdx.x + 1] = t1 - t0;
    out[3 * blockIdx.x + 2] = 1;
  }
}

// kind::f8f6f4 MMAs (e4m3 A and B, fp32 D) back to back from one thread, on
// zero operands resident in shared memory: A 128 rows, B N rows, 64-byte
// rows in the 64-byte-swizzled K-major layout (two K = 32 steps per row).
template <int N>
__global__ void __launch_bounds__(128, 1) f8_rate_kernel(int iters, long long* out) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int bytes = 128 * 64 + N * 64;
  for (int i = threadIdx.x * 16; i < bytes; i += blockDim.x * 16)
    *reinterpret_cast<uint4*>(smem + i) = make_uint4(0, 0, 0, 0);
  __shared__ uint64_t bar;
  __shared__ uint32_t slot;
  constexpr uint32_t cols = N <= 64 ? 64 : N <= 128 ? 128 : 256;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    ptx::fence_mbar_init();
  }
  ptx::fence_proxy_async_smem();
  if (threadIdx.x < 32) {
    ptx::tmem_alloc(&slot, cols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = slot;
  if (threadIdx.x == 0) {
    // e4m3 A and B (format code 0 in the A and B fields), fp32 D, K-major
    constexpr uint32_t idesc = ptx::idesc_f16_f32(128, N);
    const uint64_t ad = ptx::smem_desc_sw64_kmajor(ptx::smem_addr(smem));
    const uint64_t bd = ptx::smem_desc_sw64_kmajor(ptx::smem_addr(smem + 128 * 64));
    const long long t0 = clock64();
    for (int i = 0; i < iters; ++i) {
      const uint64_t k = static_cast<uint64_t>(i & 1) * 2;  // K = 0..31 or 32..63 of the 64-byte rows
      asm volatile(
          "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
          "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem),
          "l"(ad + k), "l"(bd + k), "r"(idesc), "r"(i > 0 ? 1u : 0u)
          : "memory");
    }
    const long long t1 = clock64();
    ptx::mma_commit(&bar);
    const bool done = ptx::mbar_wait(&bar, 0, 2000000000ull, nullptr);
    const long long t2 = clock64();
    out[3 * blockIdx.x + 0] = t1 - t0;
    out[3 * blockIdx.x + 1] = t2 - t0;
    out[3 * blockIdx.x + 2] = done ? 1 : 0;
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (threadIdx.x < 32) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, cols);
  }
}

static cudaError_t timed(void (*launch)(cudaStream_t), float* ms, cudaStream_t stream) {
  cudaEvent_t e0, e1;
  cudaError_t e = cudaEventCreate(&e0);
  if (e != cudaSuccess) return e;
  e = cudaEventCreate(&e1);
  if (e != cudaSuccess) {
    cudaEventDestroy(e0);
    return e;
  }
  cudaEventRecord(e0, stream);
  launch(stream);
  cudaEventRecord(e1, stream);
  e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaEventSynchronize(e1);
  if (e == cudaSuccess) e = cudaEventElapsedTime(ms, e0, e1);
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  return e;
}

}  // namespace i8c

namespace {
struct ImmaArgs {
  int ctas, warps, iters;
  long long* out;
  int* sink;
} g_imma;
struct F8Args {
  int ctas, iters, smem;
  long long* out;
} g_f8;
template <int N>
void launch_f8(cudaStream_t s) {
  i8c::f8_rate_kernel<N><<<g_f8.ctas, 128, g_f8.smem, s>>>(g_f8.iters, g_f8.out);
  i8c::g_launches.fetch_add(1, std::memory_order_relaxed);
}
void launch_imma(cudaStream_t s) {
  i8c::imma_rate_kernel<<<g_imma.ctas, 32 * g_imma.warps, 0, s>>>(g_imma.iters, g_imma.out, g_imma.sink);
  i8c::g_launches.fetch_add(1, std::memory_order_relaxed);
}
}  // namespace

extern "C" i8c_status i8c_probe_imma_s8(int32_t num_ctas, int32_t warps_per_cta, int32_t iters, long long* cycles,
                                        int* sink, float* elapsed_ms, cudaStream_t stream) {
  if (cycles == nullptr || sink == nullptr || elapsed_ms == nullptr || num_ctas < 1 || iters < 1 ||
      warps_per_cta < 1 || warps_per_cta > 16)
    return I8C_ERR_INVALID_ARG;
  g_imma = {num_ctas, warps_per_cta, iters, cycles, sink};
  return i8c::timed(launch_imma, elapsed_ms, stream) == cudaSuccess ? I8C_OK : I8C_ERR_CUDA;
}

extern "C" i8c_status i8c_probe_mma_f8(int32_t n, int32_t num_ctas, int32_t iters, long long* cycles,
                                       float* elapsed_ms, cudaStream_t stream) {
  if (cycles == nullptr || elapsed_ms == nullptr || num_ctas < 1 || iters < 1) return I8C_ERR_INVALID_ARG;
  const int smem = 128 * 64 + n * 64 + 1024;
  void (*launch)(cudaStream_t) = nullptr;
  const void* fn = nullptr;
  switch (n) {
    case 64: launch = launch_f8<64>; fn = reinterpret_cast<const void*>(i8c::f8_rate_kernel<64>); break;
    case 128: launch = launch_f8<128>; fn = reinterpret_cast<const void*>(i8c::f8_rate_kernel<128>); break;
    case 256: launch = launch_f8<256>; fn = reinterpret_cast<const void*>(i8c::f8_rate_kernel<256>); break;
    default: return I8C_ERR_INVALID_ARG;
  }
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return I8C_ERR_CUDA;
  g_f8 = {num_ctas, iters, smem, cycles};
  return i8c::timed(launch, elapsed_ms, stream) == cudaSuccess ? I8C_OK : I8C_ERR_CUDA;
}
