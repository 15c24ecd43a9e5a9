// Engine microbenchmarks: tensor-core issue cost and throughput of
// tcgen05.mma kind::f16 (the engine of the convolution kernels) for the
// operand layouts and tile widths they use.  One CTA per SM; lane 0 of warp 0
// issues `iters` MMAs (M = 128, N = n, K = 16) back to back on operands that
// stay resident in shared memory, then waits for their completion.  Not part
// of the convolution path.
#include "../../include/i8conv_probe.h"
#include "internal.h"

namespace i8c {

template <int N>
__global__ void __launch_bounds__(384, 1) mma_rate_kernel(int iters, int a_swizzled, int loop_mode, long long* out) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // A: 128 rows x 32 fp16 (8 KB), B: 4 K-slices of N rows x 32 fp16; all zero (finite operands)
  const int bytes = 8192 + 4 * N * 64;
  for (int i = threadIdx.x * 16; i < bytes; i += blockDim.x * 16)
    *reinterpret_cast<uint4*>(smem + i) = make_uint4(0, 0, 0, 0);
  __shared__ uint64_t bar;
  __shared__ uint32_t slot;
  constexpr uint32_t cols = N <= 32 ? 32 : N <= 64 ? 64 : N <= 128 ? 128 : 256;  // a power of two
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
  __shared__ uint64_t never;
  __shared__ volatile int stop;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&never, 1);
    stop = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5;
  if (loop_mode == 10 && warp >= 4 && warp < 8) {
    // four warps storing 16-byte vectors to a separate 8 KB scratch area as
    // fast as they can (shared-memory write traffic next to the MMAs)
    uint8_t* scratch = smem + 8192 + 4 * N * 64;
    const uint64_t t0 = ptx::globaltimer_ns();
    uint32_t v = threadIdx.x;
    int it = 0;
    while (!stop && ptx::globaltimer_ns() - t0 < 1000000000ull) {
      for (int k = 0; k < 16; ++k) {
        const uint32_t addr =
            ptx::smem_addr(scratch + (((threadIdx.x - 128) * 16 + (it & 3) * 2048) & 8191));
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v), "r"(v + 1), "r"(v + 2),
                     "r"(v + 3)
                     : "memory");
        ++it;
        v += 7;
      }
    }
  }
  if (loop_mode >= 6 && loop_mode < 8 && (warp == 4 || warp == 8)) {
    // a warp waiting on a barrier that never completes, as the producer and
    // epilogue warps wait while the MMA warp runs: sleeping (mode 6) or plain
    // polling (mode 7); leaves when warp 0 sets `stop` (bounded by 1 s)
    const uint64_t t0 = ptx::globaltimer_ns();
    while (!stop && ptx::globaltimer_ns() - t0 < 1000000000ull) {
      if (loop_mode == 6) ptx::mbar_try_wait_sleep(&never, 0, 20000u);
      else ptx::mbar_try_wait(&never, 0);
    }
  }
  // modes 19/20: a four-stage ring of full/empty barriers between the MMA
  // warp (mode 8's run loop, waiting on `full`, committing to `empty`) and a
  // producer warp that, per run, waits for the stage to be released and
  // arrives on its `full` barrier (no data moves): the kernel's handshake
  // without its loads.  19: the producer sleeps in its waits; 20: it spins.
  __shared__ uint64_t pfull[4], pempty[4];
  if (threadIdx.x == 0) {
    for (int i = 0; i < 4; ++i) {
      ptx::mbar_init(&pfull[i], 1);
      ptx::mbar_init(&pempty[i], 1);
    }
    ptx::fence_mbar_init();
  }
  __syncthreads();
  const int runs = iters / 6;
  if ((loop_mode == 19 || loop_mode == 20) && warp == 4) {
    for (int r = 0; r < runs; ++r) {
      const int st = r & 3;
      const uint32_t ph = static_cast<uint32_t>(r >> 2) & 1u;
      bool got;
      if (loop_mode == 19) {
        got = ptx::mbar_wait(&pempty[st], ph ^ 1u, 1000000000ull, nullptr);
      } else {
        const uint64_t t0 = ptx::globaltimer_ns();
        got = false;
        while (!(got = ptx::mbar_try_wait(&pempty[st], ph ^ 1u)) && ptx::globaltimer_ns() - t0 < 1000000000ull) {
        }
      }
      if (!__all_sync(0xffffffffu, got)) break;
      if (ptx::elect_one()) ptx::mbar_arrive(&pfull[st]);
      __syncwarp();
    }
  }
  if (loop_mode >= 4 && threadIdx.x < 32) {
    // The same per-K-slice pattern issued from a warp in uniform control
    // flow: the A offset comes from loop counters (mode 4) or from the
    // shared-memory table (mode 5); one elected lane issues.
    __shared__ uint32_t tbl2[16];
    __shared__ uint64_t sink2;
    if (threadIdx.x == 0) {
      for (int i = 0; i < 16; ++i) tbl2[i] = static_cast<uint32_t>(i & 7) * 2u;
      ptx::mbar_init(&bar, 1);
      ptx::mbar_init(&sink2, 1);
      ptx::fence_mbar_init();
    }
    __syncwarp();
    constexpr uint32_t idesc = ptx::idesc_f16_f32(128, N);
    const uint32_t a = ptx::smem_addr(smem);
    const uint32_t b = ptx::smem_addr(smem + 8192);
    const uint64_t ad = ptx::smem_desc_noswizzle_kmajor(a, 2560, 160);
    const uint64_t bd = ptx::smem_desc_sw64_kmajor(b);
    if (loop_mode >= 11 && loop_mode <= 14) {
      // queue-depth test: 6 MMAs, then busy-wait D cycles (D = 0, 200, 400,
      // 800 for modes 11..14), repeated
      const long long D = loop_mode == 11 ? 0 : loop_mode == 12 ? 200 : loop_mode == 13 ? 400 : 800;
      const long long t0 = clock64();
      for (int i = 0; i < iters; i += 6) {
        if (ptx::elect_one()) {
          for (int k = 0; k < 6; ++k) ptx::mma_f16_ss(tmem, ad, bd + (k & 1) * 2, idesc, (i + k) > 0 ? 1u : 0u);
        }
        __syncwarp();
        const long long w0 = clock64();
        while (clock64() - w0 < D) {
        }
      }
      const long long t1 = clock64();
      stop = 1;
      if (ptx::elect_one()) ptx::mma_commit(&bar);
      __syncwarp();
      const bool done = ptx::mbar_wait(&bar, 0, 2000000000ull, nullptr);
      const long long t2 = clock64();
      if (threadIdx.x == 0) {
        out[3 * blockIdx.x + 0] = t1 - t0;
        out[3 * blockIdx.x + 1] = t2 - t0;
        out[3 * blockIdx.x + 2] = done ? 1 : 0;
      }
    } else if (loop_mode == 19 || loop_mode == 20) {
      const uint64_t a_desc0 = ad & ~static_cast<uint64_t>(0x3FFF);
      const uint64_t b_desc0 = bd & ~static_cast<uint64_t>(0x3FFF);
      const uint32_t h_stage = static_cast<uint32_t>(ad & 0x3FFF), b_lo0 = static_cast<uint32_t>(bd & 0x3FFF);
      const uint32_t chunk2_lo = 2560 >> 4, slice_lo = (N * 64) >> 4;
      uint32_t acc_flag = 0;
      const long long t0 = clock64();
      for (int r = 0; r < runs; ++r) {
        const int st = r & 3;
        const uint32_t ph = static_cast<uint32_t>(r >> 2) & 1u;
        if (!__all_sync(0xffffffffu, ptx::mbar_wait(&pfull[st], ph, 1000000000ull, nullptr))) break;
        ptx::tc_fence_after();
        uint32_t b_cur = b_lo0 + static_cast<uint32_t>(r & 1) * slice_lo;
        for (int t = 0; t < 3; ++t) {
          const uint32_t a_cur = h_stage + static_cast<uint32_t>((r % 3) * 10 + t);
          const uint64_t ad0 = a_desc0 | static_cast<uint64_t>(a_cur & 0x3FFFu);
          const uint64_t ad1 = a_desc0 | static_cast<uint64_t>((a_cur + chunk2_lo) & 0x3FFFu);
          const uint64_t bdd = b_desc0 | static_cast<uint64_t>(b_cur & 0x3FFFu);
          if (ptx::elect_one()) {
            ptx::mma_f16_ss(tmem, ad0, bdd, idesc, acc_flag);
            ptx::mma_f16_ss(tmem, ad1, bdd + 2, idesc, 1u);
          }
          __syncwarp();
          acc_flag = 1;
          b_cur += slice_lo;
        }
        if (ptx::elect_one()) ptx::mma_commit(&pempty[st]);
        __syncwarp();
      }
      const long long t1 = clock64();
      stop = 1;
      if (ptx::elect_one()) ptx::mma_commit(&bar);
      __syncwarp();
      const bool done = ptx::mbar_wait(&bar, 0, 2000000000ull, nullptr);
      const long long t2 = clock64();
      if (threadIdx.x == 0) {
        out[3 * blockIdx.x + 0] = t1 - t0;
        out[3 * blockIdx.x + 1] = t2 - t0;
        out[3 * blockIdx.x + 2] = done ? 1 : 0;
      }
    } else if (loop_mode == 8 || loop_mode == 9 || (loop_mode >= 15 && loop_mode <= 18)) {
      // mode 8: the convolution kernel's run loop verbatim (runs of 3 K-slices,
      // a completed-barrier wait + fence before each run, column-phase
      // arithmetic, a commit after each run); mode 9: the same with the tap
      // address advanced by a constant.  Modes 15-18 take parts away: 15 no
      // commit, 16 no barrier wait, 17 one elected block per run (all six
      // MMAs and the commit), 18 as 17 without wait and commit.
      const bool do_commit = loop_mode != 15 && loop_mode != 18;
      const bool do_wait = loop_mode != 16 && loop_mode != 18;
      const bool per_run = loop_mode == 17 || loop_mode == 18;
      __shared__ uint64_t full3;
      if (threadIdx.x == 0) {
        ptx::mbar_init(&full3, 1);
        ptx::fence_mbar_init();
        ptx::mbar_arrive(&full3);
      }
      __syncwarp();
      // geometry from the (runtime) iteration count so the compiler cannot fold it
      const int rt = iters >> 30;  // 0 for any real iteration count
      const int G = 3, S = 3 + rt, sw = 2 + rt, dw_mod = 1 + rt, dw_div = rt, cw_q = 5 + rt, cw_r = rt;
      const uint64_t a_desc0 = ad & ~static_cast<uint64_t>(0x3FFF);
      const uint64_t b_desc0 = bd & ~static_cast<uint64_t>(0x3FFF);
      const uint32_t h_stage = static_cast<uint32_t>(ad & 0x3FFF), b_lo0 = static_cast<uint32_t>(bd & 0x3FFF);
      const uint32_t chunk2_lo = 2560 >> 4, slice_lo = (N * 64) >> 4;
      uint32_t acc_flag = 0;
      const long long t0 = clock64();
      for (int run = 0; run < iters / (2 * G); ++run) {
        if (do_wait) {
          if (!__all_sync(0xffffffffu, ptx::mbar_wait(&full3, 0, 1000000000ull, nullptr))) break;
          ptx::tc_fence_after();
        }
        uint32_t b_cur = b_lo0 + static_cast<uint32_t>(run & 1) * slice_lo;
        int fph = 0, idx = 0;
        const int rowpos = (run % S) * (10 + rt);
        if (per_run) {
          uint64_t a0[3], a1[3], bq[3];
#pragma unroll
          for (int t = 0; t < 3; ++t) {
            const uint32_t a_cur = h_stage + static_cast<uint32_t>(rowpos + fph * cw_q + min(fph, cw_r) + idx);
            a0[t] = a_desc0 | static_cast<uint64_t>(a_cur & 0x3FFFu);
            a1[t] = a_desc0 | static_cast<uint64_t>((a_cur + chunk2_lo) & 0x3FFFu);
            bq[t] = b_desc0 | static_cast<uint64_t>(b_cur & 0x3FFFu);
            b_cur += slice_lo;
            fph += dw_mod;
            const int carry = fph >= sw ? 1 : 0;
            fph -= carry * sw;
            idx += dw_div + carry;
          }
          if (ptx::elect_one()) {
#pragma unroll
            for (int t = 0; t < 3; ++t) {
              ptx::mma_f16_ss(tmem, a0[t], bq[t], idesc, acc_flag | static_cast<uint32_t>(t));
              ptx::mma_f16_ss(tmem, a1[t], bq[t] + 2, idesc, 1u);
            }
            if (do_commit) ptx::mma_commit(&sink2);
          }
          __syncwarp();
          acc_flag = 1;
          continue;
        }
        for (int t = 0; t < G; ++t) {
          const uint32_t a_cur = loop_mode == 8
                                     ? h_stage + static_cast<uint32_t>(rowpos + fph * cw_q + min(fph, cw_r) + idx)
                                     : h_stage + static_cast<uint32_t>(rowpos + t);
          const uint64_t ad0 = a_desc0 | static_cast<uint64_t>(a_cur & 0x3FFFu);
          const uint64_t ad1 = a_desc0 | static_cast<uint64_t>((a_cur + chunk2_lo) & 0x3FFFu);
          const uint64_t bdd = b_desc0 | static_cast<uint64_t>(b_cur & 0x3FFFu);
          if (ptx::elect_one()) {
            ptx::mma_f16_ss(tmem, ad0, bdd, idesc, acc_flag);
            ptx::mma_f16_ss(tmem, ad1, bdd + 2, idesc, 1u);
          }
          __syncwarp();
          acc_flag = 1;
          b_cur += slice_lo;
          fph += dw_mod;
          const int carry = fph >= sw ? 1 : 0;
          fph -= carry * sw;
          idx += dw_div + carry;
        }
        if (do_commit) {
          if (ptx::elect_one()) ptx::mma_commit(&sink2);
          __syncwarp();
        }
        (void)S;
      }
      const long long t1 = clock64();
      stop = 1;
      if (ptx::elect_one()) ptx::mma_commit(&bar);
      __syncwarp();
      const bool done = ptx::mbar_wait(&bar, 0, 2000000000ull, nullptr);
      const long long t2 = clock64();
      if (threadIdx.x == 0) {
        out[3 * blockIdx.x + 0] = t1 - t0;
        out[3 * blockIdx.x + 1] = t2 - t0;
        out[3 * blockIdx.x + 2] = done ? 1 : 0;
      }
    } else {
    const long long t0 = clock64();
    int r = 0, s = 0;
    for (int i = 0; i < iters; i += 2) {
      const int sl = i >> 1;
      const uint32_t aoff = (loop_mode == 4 || loop_mode == 10) ? static_cast<uint32_t>(r * 10 + s) : tbl2[sl & 15];
      const uint64_t a_lo = ad + aoff;
      const uint64_t b_lo = bd + static_cast<uint64_t>((sl & 3) * N * 4);
      if (ptx::elect_one()) {
        ptx::mma_f16_ss(tmem, a_lo, b_lo, idesc, i > 0 ? 1u : 0u);
        ptx::mma_f16_ss(tmem, a_lo + 2, b_lo + 2, idesc, 1u);
        if ((sl & 3) == 3) ptx::mma_commit(&sink2);
      }
      __syncwarp();
      if (++s == 3) {
        s = 0;
        if (++r == 3) r = 0;
      }
    }
    const long long t1 = clock64();
    stop = 1;
    if (ptx::elect_one()) ptx::mma_commit(&bar);
    __syncwarp();
    const bool done = ptx::mbar_wait(&bar, 0, 2000000000ull, nullptr);
    const long long t2 = clock64();
    if (threadIdx.x == 0) {
      out[3 * blockIdx.x + 0] = t1 - t0;
      out[3 * blockIdx.x + 1] = t2 - t0;
      out[3 * blockIdx.x + 2] = done ? 1 : 0;
    }
    }
  } else if (loop_mode < 4 && threadIdx.x == 0) {
    constexpr uint32_t idesc = ptx::idesc_f16_f32(128, N);
    const uint32_t a = ptx::smem_addr(smem);
    const uint32_t b = ptx::smem_addr(smem + 8192);
    // a_layout: 0 no-swizzle, core matrices contiguous (SBO 128, LBO 2048); 1 64-byte swizzle;
    // 2 no-swizzle with 8-row groups 160 bytes apart (a 10-entry halo row) and LBO 2560;
    // 3 as 2 but starting 16 bytes in (a shifted filter tap)
    // 4, 5: transposed operands -- A 64-byte swizzled (128 filter rows), B
    // without swizzle, N pixel rows in 8-channel planes of N*16 bytes, 8-row
    // groups 128 bytes apart; 5 starts B 48 bytes in (a tap shift: core
    // matrices straddle 128-byte lines)
    const bool transposed = a_swizzled == 4 || a_swizzled == 5;
    uint64_t ad, bd;
    if (a_swizzled == 1 || transposed) ad = ptx::smem_desc_sw64_kmajor(a);
    else if (a_swizzled == 0) ad = ptx::smem_desc_noswizzle_kmajor(a, 2048, 128);
    else ad = ptx::smem_desc_noswizzle_kmajor(a + (a_swizzled == 3 ? 16 : 0), 2560, 160);
    if (transposed) bd = ptx::smem_desc_noswizzle_kmajor(b + (a_swizzled == 5 ? 48 : 0), N * 16, 128);
    else bd = ptx::smem_desc_sw64_kmajor(b);
    const uint64_t b_khalf = transposed ? static_cast<uint64_t>(2 * N) : 2u;  // K = 16..31: 2 planes, or 32 bytes
    long long t0, t1;
    if (loop_mode == 0) {
      t0 = clock64();
      for (int i = 0; i < iters; ++i)
        ptx::mma_f16_ss(tmem, ad + (a_swizzled == 1 || transposed ? (i & 1) * 2 : 0), bd + (i & 1) * b_khalf, idesc,
                        i > 0 ? 1u : 0u);
      t1 = clock64();
    } else {
      // The convolution's per-K-slice pattern: two MMAs (K = 16 each) per
      // slice, the A start taken from a per-tap offset table in shared
      // memory, a barrier check every 4 slices (mode >= 2, on a barrier whose
      // phase has completed) and a commit every 4 slices (mode >= 3).
      __shared__ uint32_t tbl[16];
      __shared__ uint64_t ready, sink;
      for (int i = 0; i < 16; ++i) tbl[i] = static_cast<uint32_t>(i & 7) * 2u;
      ptx::mbar_init(&ready, 1);
      ptx::mbar_init(&sink, 1);
      ptx::fence_mbar_init();
      ptx::mbar_arrive(&ready);
      t0 = clock64();
      for (int i = 0; i < iters; i += 2) {
        const int sl = i >> 1;
        if (loop_mode >= 2 && (sl & 3) == 0) {
          if (!ptx::mbar_wait(&ready, 0, 1000000000ull, nullptr)) break;
          ptx::tc_fence_after();
        }
        const uint64_t a_lo = ad + (loop_mode >= 1 && a_swizzled != 1 ? tbl[sl & 15] : 0u);
        // B slice (sl & 3) of the 4-slice B region: +N*64 bytes = +N*4 in the >>4 address field
        const uint64_t b_lo = bd + static_cast<uint64_t>((sl & 3) * N * 4);
        ptx::mma_f16_ss(tmem, a_lo, b_lo, idesc, i > 0 ? 1u : 0u);
        ptx::mma_f16_ss(tmem, a_lo + 2, b_lo + 2, idesc, 1u);
        if (loop_mode >= 3 && (sl & 3) == 3) ptx::mma_commit(&sink);
      }
      t1 = clock64();
    }
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

template <int N>
static cudaError_t run_rate(int ctas, int iters, int swz, int mode, long long* out, float* ms, cudaStream_t stream) {
  const int smem = 8192 + 4 * N * 64 + 8192 + 1024;
  cudaError_t e = cudaFuncSetAttribute(mma_rate_kernel<N>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaEvent_t e0, e1;
  cudaEventCreate(&e0);
  cudaEventCreate(&e1);
  cudaEventRecord(e0, stream);
  mma_rate_kernel<N><<<ctas, 384, smem, stream>>>(iters, swz, mode, out);
  g_launches.fetch_add(1, std::memory_order_relaxed);
  cudaEventRecord(e1, stream);
  e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaEventSynchronize(e1);
  if (e == cudaSuccess) e = cudaEventElapsedTime(ms, e0, e1);
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  return e;
}

}  // namespace i8c

extern "C" i8c_status i8c_probe_mma_f16(int32_t n, int32_t a_swizzled, int32_t loop_mode, int32_t num_ctas, int32_t iters,
                                        long long* cycles, float* elapsed_ms, cudaStream_t stream) {
  if (cycles == nullptr || elapsed_ms == nullptr || num_ctas < 1 || iters < 1) return I8C_ERR_INVALID_ARG;
  cudaError_t e;
  switch (n) {
    case 32: e = i8c::run_rate<32>(num_ctas, iters, a_swizzled, loop_mode, cycles, elapsed_ms, stream); break;
    case 64: e = i8c::run_rate<64>(num_ctas, iters, a_swizzled, loop_mode, cycles, elapsed_ms, stream); break;
    case 128: e = i8c::run_rate<128>(num_ctas, iters, a_swizzled, loop_mode, cycles, elapsed_ms, stream); break;
    case 256: e = i8c::run_rate<256>(num_ctas, iters, a_swizzled, loop_mode, cycles, elapsed_ms, stream); break;
    case 176: e = i8c::run_rate<176>(num_ctas, iters, a_swizzled, loop_mode, cycles, elapsed_ms, stream); break;
    case 224: e = i8c::run_rate<224>(num_ctas, iters, a_swizzled, loop_mode, cycles, elapsed_ms, stream); break;
    default: return I8C_ERR_INVALID_ARG;
  }
  return e == cudaSuccess ? I8C_OK : I8C_ERR_CUDA;
}
