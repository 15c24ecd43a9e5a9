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

// L2 -> shared memory read rate of one SM.  Mode 0: one thread keeps
// kIngressBufs untiled bulk copies (TMA) of `chunk` bytes in flight into a
// ring of shared-memory buffers; mode 1: all threads load 16-byte vectors
// (ld.global.nc, kIngressVecs in flight per thread) and store them to shared
// memory.  Step i of CTA c reads chunk (c + i * gridDim.x) mod nchunks.
constexpr int kIngressBufs = 4;
constexpr int kIngressThreads = 512;
constexpr int kIngressVecs = 4;

__global__ void __launch_bounds__(kIngressThreads, 1)
    ingress_kernel(const uint8_t* __restrict__ src, int64_t nchunks, int chunk, int mode, int iters,
                   long long* out) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar[kIngressBufs];
  __shared__ uint64_t empty[kIngressBufs];  // mode 2: both CTAs of the cluster hold the buffer's chunk
  if (threadIdx.x == 0) {
    for (int b = 0; b < kIngressBufs; ++b) {
      ptx::mbar_init(&bar[b], 1);
      ptx::mbar_init(&empty[b], 2);
    }
    ptx::fence_mbar_init();
  }
  __syncthreads();
  if (mode == 2) ptx::cluster_sync();  // both CTAs' barriers exist before any multicast lands
  bool ok = true;
  const long long t0 = clock64();
  if (mode == 2) {
    // clusters of two: each CTA copies its half of every chunk into both
    // CTAs' buffer (multicast); a buffer is refilled only after both CTAs
    // have received its previous chunk whole
    if (threadIdx.x == 0) {
      const uint32_t rank = blockIdx.x & 1u;
      const int64_t cl = blockIdx.x >> 1, ncl = gridDim.x >> 1;
      const int half = chunk / 2;
      int issued = 0;
      for (int i = 0; i < iters && ok; ++i) {
        const int b = i % kIngressBufs;
        if (i >= kIngressBufs) {
          const uint32_t ph = ((i / kIngressBufs) - 1) & 1u;
          if (!ptx::mbar_wait(&bar[b], ph, 2000000000ull, nullptr)) {
            ok = false;
            break;
          }
          ptx::mbar_arrive(&empty[b]);
          ptx::mbar_arrive_remote(ptx::mapa(ptx::smem_addr(&empty[b]), rank ^ 1u), 1);
          if (!ptx::mbar_wait<true>(&empty[b], ph, 2000000000ull, nullptr)) {
            ok = false;
            break;
          }
        }
        const int64_t c = (cl + static_cast<int64_t>(i) * ncl) % nchunks;
        ptx::mbar_arrive_expect_tx(&bar[b], static_cast<uint32_t>(chunk));
        ptx::bulk_load_multicast(smem + static_cast<size_t>(b) * chunk + rank * half, src + c * chunk + rank * half,
                                 static_cast<uint32_t>(half), &bar[b], 3);
        issued = i + 1;
      }
      // every chunk issued into this CTA has landed (a step whose gate failed
      // was not issued); the peer's halves are covered by the same barriers
      const int first = issued > kIngressBufs ? issued - kIngressBufs : 0;
      for (int i = first; i < issued; ++i)
        if (!ptx::mbar_wait(&bar[i % kIngressBufs], (i / kIngressBufs) & 1u, 2000000000ull, nullptr)) ok = false;
    }
  } else if (mode == 0) {
    if (threadIdx.x == 0) {
      int issued = 0;
      for (int i = 0; i < iters && ok; ++i) {
        const int b = i % kIngressBufs;
        // the buffer's previous copy (kIngressBufs steps ago) has landed
        if (i >= kIngressBufs && !ptx::mbar_wait(&bar[b], ((i / kIngressBufs) - 1) & 1u, 2000000000ull, nullptr)) {
          ok = false;
          break;
        }
        const int64_t c = (blockIdx.x + static_cast<int64_t>(i) * gridDim.x) % nchunks;
        ptx::mbar_arrive_expect_tx(&bar[b], static_cast<uint32_t>(chunk));
        ptx::bulk_load(smem + static_cast<size_t>(b) * chunk, src + c * chunk, static_cast<uint32_t>(chunk), &bar[b]);
        issued = i + 1;
      }
      // the copies still in flight
      const int first = issued > kIngressBufs ? issued - kIngressBufs : 0;
      for (int i = first; i < issued; ++i)
        if (!ptx::mbar_wait(&bar[i % kIngressBufs], (i / kIngressBufs) & 1u, 2000000000ull, nullptr)) ok = false;
    }
  } else if (mode == 3) {
    // every thread copies its 16-byte pieces of each chunk with cp.async
    // (global -> shared, no registers), one commit group per chunk, at most
    // kIngressBufs - 1 groups in flight
    const int vecs = chunk / 16;
    const uint32_t base = ptx::smem_addr(smem);
    for (int i = 0; i < iters; ++i) {
      const int64_t c = (blockIdx.x + static_cast<int64_t>(i) * gridDim.x) % nchunks;
      const uint8_t* s = src + c * chunk;
      const uint32_t d = base + static_cast<uint32_t>((i % kIngressBufs) * chunk);
      for (int v = threadIdx.x; v < vecs; v += kIngressThreads) ptx::cp_async_16_cg(d + v * 16, s + v * 16);
      ptx::cp_async_commit();
      ptx::cp_async_wait<kIngressBufs - 1>();
    }
    ptx::cp_async_wait_all();
  } else {
    const int vecs = chunk / 16;  // a multiple of kIngressThreads * kIngressVecs
    for (int i = 0; i < iters; ++i) {
      const int64_t c = (blockIdx.x + static_cast<int64_t>(i) * gridDim.x) % nchunks;
      const uint4* s = reinterpret_cast<const uint4*>(src + c * chunk);
      uint4* d = reinterpret_cast<uint4*>(smem + static_cast<size_t>(i % kIngressBufs) * chunk);
      for (int v0 = 0; v0 < vecs; v0 += kIngressThreads * kIngressVecs) {
        uint4 v[kIngressVecs];
#pragma unroll
        for (int q = 0; q < kIngressVecs; ++q) v[q] = ptx::ldg16_or_zero(s + v0 + q * kIngressThreads + threadIdx.x, true);
#pragma unroll
        for (int q = 0; q < kIngressVecs; ++q) d[v0 + q * kIngressThreads + threadIdx.x] = v[q];
      }
    }
  }
  __syncthreads();
  const long long t1 = clock64();
  // the peer may still be delivering into this CTA (mode 2): leave together
  if (mode == 2) ptx::cluster_sync();
  if (threadIdx.x == 0) {
    out[3 * blockIdx.x + 0] = t1 - t0;
    out[3 * blockIdx.x + 1] = static_cast<long long>(iters) * chunk;
    out[3 * blockIdx.x + 2] = ok ? 1 : 0;
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
struct IngressArgs {
  const uint8_t* src;
  int64_t nchunks;
  int chunk, mode, ctas, iters, smem;
  long long* out;
} g_ingress;
void launch_ingress(cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(static_cast<unsigned>(g_ingress.ctas));
  cfg.blockDim = dim3(i8c::kIngressThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(g_ingress.smem);
  cfg.stream = s;
  if (g_ingress.mode == 2) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  cudaLaunchKernelEx(&cfg, i8c::ingress_kernel, g_ingress.src, g_ingress.nchunks, g_ingress.chunk, g_ingress.mode,
                     g_ingress.iters, g_ingress.out);
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

extern "C" i8c_status i8c_probe_l2_ingress(const void* src, int64_t region_bytes, int32_t chunk_bytes, int32_t mode,
                                           int32_t num_ctas, int32_t iters, long long* cycles, float* elapsed_ms,
                                           cudaStream_t stream) {
  if (src == nullptr || cycles == nullptr || elapsed_ms == nullptr || num_ctas < 1 || iters < 1 ||
      mode < 0 || mode > 3 || chunk_bytes < 16 || chunk_bytes > 49152 || chunk_bytes % 16 != 0 ||
      (mode == 2 && (chunk_bytes % 32 != 0 || num_ctas % 2 != 0)) ||
      (mode == 1 && chunk_bytes % (16 * i8c::kIngressThreads * i8c::kIngressVecs) != 0) ||
      region_bytes < chunk_bytes || region_bytes % chunk_bytes != 0 || (reinterpret_cast<uintptr_t>(src) & 15u))
    return I8C_ERR_INVALID_ARG;
  const int smem = i8c::kIngressBufs * chunk_bytes + 1024;
  if (cudaFuncSetAttribute(reinterpret_cast<const void*>(i8c::ingress_kernel),
                           cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return I8C_ERR_CUDA;
  g_ingress = {static_cast<const uint8_t*>(src), region_bytes / chunk_bytes, chunk_bytes, mode, num_ctas, iters,
               smem, cycles};
  return i8c::timed(launch_ingress, elapsed_ms, stream) == cudaSuccess ? I8C_OK : I8C_ERR_CUDA;
}
