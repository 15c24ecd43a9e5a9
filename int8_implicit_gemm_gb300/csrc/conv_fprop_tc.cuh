// INT8 NCxHWx<32> Conv2d fprop as an implicit GEMM on the sm_103a tensor cores.
//
// GEMM view (the CUTLASS fprop configuration of the "int8 fprop2d kernel with
// NCxHWx interleaved layout" issue, and the implicit-GEMM paragraph of the
// POPCORNBENCH l1_p80 trace):  rows m = (n, p, q) output pixels (M = N*P*Q),
// columns = output channels (K), reduction = (c, r, s) (C*R*S).  One K-slice
// is one filter tap (r, s) of one 32-channel block cb: exactly one 32-byte
// NCxHWx<32> vector per output pixel and one 32-byte CxRSKx<32> row per
// output channel.
//
// sm_103a has no tcgen05 int8 MMA, so the contraction runs as kind::f16 with
// fp16 operands (every int8 value is exact in fp16, every product |x*f| <=
// 2^14 is exact in fp32) accumulating in fp32 tensor memory.  A partial sum
// stays exact while its magnitude is at most 2^24, which holds for any data
// when a chunk covers at most 1024 reduction elements (32 slices).  After each
// chunk the epilogue warps convert the fp32 accumulator to int32 (exact) and
// add it into an int32 running sum kept in tensor memory, so the final
// accumulator is the exact int32 sum for every input.
//
// Persistent CTAs, one per SM, walk tiles of 128 pixels x BN channels.  Warp
// roles (384 threads):
//   warp 0      tensor-memory allocation; lane 0 issues the MMAs
//   warp 1      lane 0 streams fp16 filter tiles with TMA
//   warps 4-7   activation producers: cp.async gather of the 32-byte vectors
//               (zero-filled outside the image), int8 -> fp16 conversion into
//               the 64-byte-swizzled K-major operand layout
//   warps 8-11  epilogue: tensor memory -> registers, chunk flush, then
//               clamp(rint(alpha * float(acc))) and 32-byte NCxHWx<32> stores
// Every barrier wait is bounded; on expiry the CTA records I8C_ERR_TIMEOUT in
// the status word, stops all roles, waits for its copies and MMAs in flight
// and frees its tensor memory before returning.
#pragma once

#include <climits>
#include <cstdint>

#include "ptx.cuh"

namespace i8c {

struct ConvParams {
  const int8_t* x;
  int8_t* y;       // int8 output (out_mode 0)
  int32_t* acc;    // int32 accumulators (out_mode 1)
  int* status;     // device status word (0 = ok)
  float alpha;
  // per-output-channel epilogue (null / 0: the scalar alpha, no bias, no ReLU)
  const float* alpha_k;  // K scales, 16-byte aligned
  const float* bias_k;   // K biases added after the scale, 16-byte aligned
  int relu;              // 1: max(v, 0) before the clamp
  int H, W, K;
  int pad_h, pad_w, stride_h, stride_w, dil_h, dil_w;
  int R, S;
  int P, Q, PQ;
  int M;           // N*P*Q
  int CB, KB;      // C/32, K/32
  int num_slices;  // CB*R*S
  int chunk_slices;
  int num_chunks;
  int num_n_tiles;
  int num_tiles;
  int acc_buffers;  // 1 or 2
  uint32_t tmem_cols;
  int64_t img_stride;  // bytes per input image: CB*H*W*32
  uint64_t timeout_ns;
  int out_mode;
  int debug_flags;
  long long* trace;  // optional clock64 trace of CTA 0 (null = off), kTraceSlots per role
};

// Trace layout (CTA 0 only): role r, event e, index i ->
// trace[(r * 4 + e) * kTraceSlots + i].  Roles: 0 MMA, 1 filter TMA,
// 2 activation producer thread 0, 3 epilogue thread 0.
constexpr int kTraceSlots = 512;
constexpr int kTraceRows = 32;  // rows 0-15: role x event; 16-31: pipeline analysis build
__device__ __forceinline__ void trace_mark(const ConvParams& p, int role, int ev, uint32_t i) {
  if (p.trace != nullptr && blockIdx.x == 0 && i < static_cast<uint32_t>(kTraceSlots))
    p.trace[(role * 4 + ev) * kTraceSlots + i] = clock64();
}

constexpr int kStatusTimeout = 6;  // I8C_ERR_TIMEOUT

template <int BN>
struct TileCfg {
  static constexpr int BM = 128;
  static constexpr int kThreads = 384;
  static constexpr int kAStage = BM * 64;  // 128 rows x 32 fp16
  static constexpr int kBStage = BN * 64;  // BN rows x 32 fp16
  static constexpr int kStages = BN >= 256 ? 6 : (BN >= 128 ? 8 : 10);
  static constexpr int kStg = BN >= 256 ? 8 : (BN >= 128 ? 12 : 16);  // int8 staging slots
  static constexpr int kLook = kStg - 1;                              // slices of cp.async lookahead
  static constexpr int kStgBytes = BM * 32;
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + kStages * kAStage;
  static constexpr int kOffStg = kOffB + kStages * kBStage;
  static constexpr int kOffBar = kOffStg + kStg * kStgBytes;
  // full_a[S], full_b[S], empty[S], acc_full[2], acc_empty[2], drain
  static constexpr int kNumBars = 3 * kStages + 5;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + slack to align the base to 1024
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(kOffB % 1024 == 0 && kOffStg % 1024 == 0, "operand tiles must stay 1024-byte aligned");
};

// 4 int8 (one 32-bit word) -> 4 fp16 as two fp16x2 words, exactly: bias each
// byte to unsigned (b + 128), place it in the mantissa of 1024.0 (fp16 bits
// 0x6400 | byte), subtract 1152.0.
__device__ __forceinline__ void i8x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  uint32_t a, b;
  asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(a) : "r"(u), "r"(0x64646464u));
  asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(b) : "r"(u), "r"(0x64646464u));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(0x64806480u));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(0x64806480u));
}

__device__ __forceinline__ void raise_timeout(const ConvParams& p, volatile int* abort_flag) {
  atomicCAS(p.status, 0, kStatusTimeout);
  *abort_flag = 1;
}

// Epilogue arithmetic of the LinearCombinationClamp / alpha-only configuration:
// int32 -> fp32 (round to nearest even), one fp32 multiply, round half to even
// to int32.  The clamp to the int8 range is left to the saturating packs
// below: both bounds are integers, so clamping before rounding and saturating
// after it give the same byte (a float -> int32 conversion itself saturates,
// so no product is out of reach of the clamp).
__device__ __forceinline__ int requant_rn(int a, float alpha) {
  return __float2int_rn(__fmul_rn(__int2float_rn(a), alpha));
}

// The per-output-channel epilogue: one fp32 multiply by the channel's scale
// and one fp32 add of its bias, each rounded to nearest even and never fused
// (a fused multiply-add rounds once and can land on the other side of a .5),
// round half to even, then ReLU as a lower bound of 0 (lo = 0, else lo =
// INT_MIN, no bound); the clamp to [-128, 127] again in the pack.  max(rint(v),
// 0) = rint(max(v, 0)) because 0 is an integer.  With scale = alpha, bias = 0
// and no ReLU it equals requant_rn(): adding 0 changes at most the sign of a
// zero.
__device__ __forceinline__ int requant_ch(int a, float scale, float bias, int lo) {
  return max(__float2int_rn(__fadd_rn(__fmul_rn(__int2float_rn(a), scale), bias)), lo);
}

// Saturating packs of int32 values into int8 bytes (the packed-conversion
// instruction: each source clamped to [-128, 127]); a is the lowest byte.
__device__ __forceinline__ uint32_t pack4_sat_s8(int a, int b, int c, int d) {
  uint32_t hi, r;
  asm("cvt.pack.sat.s8.s32.b32 %0, %1, %2, 0;" : "=r"(hi) : "r"(d), "r"(c));
  asm("cvt.pack.sat.s8.s32.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(b), "r"(a), "r"(hi));
  return r;
}
__device__ __forceinline__ uint32_t sat_s8(int a) {
  uint32_t r;
  asm("cvt.pack.sat.s8.s32.b32 %0, 0, %1, 0;" : "=r"(r) : "r"(a));
  return r;
}

// One pixel's 32 consecutive output channels k0 .. k0 + 31 (a(i) the
// accumulator of channel k0 + i) requantised into eight packed words, with
// the channels' scales and biases, or the scalar alpha and no bias.
template <typename Acc>
__device__ __forceinline__ void requant32(const ConvParams& p, int k0, Acc&& a, uint32_t (&o)[8]) {
  if (p.alpha_k == nullptr && p.bias_k == nullptr && !p.relu) {  // one scale, no bias: no loads
#pragma unroll
    for (int i = 0; i < 8; ++i)
      o[i] = pack4_sat_s8(requant_rn(a(4 * i), p.alpha), requant_rn(a(4 * i + 1), p.alpha),
                          requant_rn(a(4 * i + 2), p.alpha), requant_rn(a(4 * i + 3), p.alpha));
    return;
  }
  // per-channel scales or biases, loaded channel by channel where they are
  // used (every lane of the warp reads the same addresses): volatile loads
  // the compiler keeps in place, so the 256-wide kernels' epilogue (128
  // running sums per thread) stays within its register budget
  const int lo = p.relu ? 0 : INT_MIN;
  const float* sa = p.alpha_k != nullptr ? p.alpha_k + k0 : nullptr;
  const float* sb = p.bias_k != nullptr ? p.bias_k + k0 : nullptr;
  auto ld = [](const float* q) {
    float v;
    asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(q));
    return v;
  };
  auto ch = [&](int i) {
    const float sc = sa != nullptr ? ld(sa + i) : p.alpha;
    const float bi = sb != nullptr ? ld(sb + i) : 0.0f;
    return requant_ch(a(i), sc, bi, lo);
  };
#pragma unroll
  for (int i = 0; i < 8; ++i) o[i] = pack4_sat_s8(ch(4 * i), ch(4 * i + 1), ch(4 * i + 2), ch(4 * i + 3));
}

template <int BN>
__global__ void __launch_bounds__(TileCfg<BN>::kThreads, 1)
    conv_fprop_tc_kernel(const __grid_constant__ CUtensorMap tmap_f, const ConvParams p) {
  using Cfg = TileCfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::kOffBar);
  uint64_t* full_a = bars;
  uint64_t* full_b = bars + Cfg::kStages;
  uint64_t* empty = bars + 2 * Cfg::kStages;
  uint64_t* acc_full = bars + 3 * Cfg::kStages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_full + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::kOffMisc + 4);

  const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x) >> 5, 0);
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < Cfg::kStages; ++i) {
      ptx::mbar_init(&full_a[i], 128);
      ptx::mbar_init(&full_b[i], 1);
      ptx::mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&acc_full[i], 1);
      ptx::mbar_init(&acc_empty[i], 128);
    }
    ptx::mbar_init(drain, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1 && lane == 0) ptx::prefetch_tensormap(&tmap_f);
  if (warp == 0) {
    ptx::tmem_alloc(tmem_slot, p.tmem_cols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const uint32_t nb = static_cast<uint32_t>(p.acc_buffers);

  if (warp == 0) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = ptx::idesc_f16_f32(128, BN);
      const uint32_t a_base = ptx::smem_addr(smem + Cfg::kOffA);
      const uint32_t b_base = ptx::smem_addr(smem + Cfg::kOffB);
      uint32_t g = 0, u = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
        for (int c = 0; ok && c < p.num_chunks; ++c, ++u) {
          const int s0 = c * p.chunk_slices;
          const int s1 = min(s0 + p.chunk_slices, p.num_slices);
          const uint32_t buf = u % nb;
          if (!ptx::mbar_wait(&acc_empty[buf], ((u / nb) & 1u) ^ 1u, p.timeout_ns, abort_flag)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t d_tmem = tmem_base + buf * BN;
          for (int kk = s0; kk < s1; ++kk, ++g) {
            const uint32_t st = g % Cfg::kStages;
            const uint32_t ph = (g / Cfg::kStages) & 1u;
            if (!ptx::mbar_wait(&full_a[st], ph, p.timeout_ns, abort_flag) ||
                !ptx::mbar_wait(&full_b[st], ph, p.timeout_ns, abort_flag)) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            const uint64_t ad = ptx::smem_desc_sw64_kmajor(a_base + st * Cfg::kAStage);
            const uint64_t bd = ptx::smem_desc_sw64_kmajor(b_base + st * Cfg::kBStage);
            // two K=16 steps cover the 32 channels of the slice (+32 bytes each)
            ptx::mma_f16_ss(d_tmem, ad, bd, idesc, kk > s0 ? 1u : 0u);
            ptx::mma_f16_ss(d_tmem, ad + 2, bd + 2, idesc, 1u);
            ptx::mma_commit(&empty[st]);
          }
          if (!ok) break;
          ptx::mma_commit(&acc_full[buf]);
        }
      }
      if (!ok) raise_timeout(p, abort_flag);
      // every MMA issued by this thread has completed before TMEM is freed
      ptx::mma_commit(drain);
      if (!ptx::mbar_wait(drain, 0, p.timeout_ns, nullptr)) raise_timeout(p, abort_flag);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ filter TMA producer
    if (lane == 0) {
      uint32_t g = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
        const int n0 = (tile % p.num_n_tiles) * BN;
        for (int kk = 0; kk < p.num_slices; ++kk, ++g) {
          const uint32_t st = g % Cfg::kStages;
          if (!ptx::mbar_wait(&empty[st], ((g / Cfg::kStages) & 1u) ^ 1u, p.timeout_ns, abort_flag)) {
            ok = false;
            break;
          }
          ptx::mbar_arrive_expect_tx(&full_b[st], Cfg::kBStage);
          ptx::tma_load_3d(smem + Cfg::kOffB + st * Cfg::kBStage, &tmap_f, &full_b[st], 0, n0, kk);
        }
      }
      if (!ok) raise_timeout(p, abort_flag);
      // wait for the loads still in flight (at most one per stage)
      const uint32_t first = g > static_cast<uint32_t>(Cfg::kStages) ? g - Cfg::kStages : 0u;
      for (uint32_t i = first; i < g; ++i) {
        if (!ptx::mbar_wait(&full_b[i % Cfg::kStages], (i / Cfg::kStages) & 1u, p.timeout_ns, nullptr)) {
          raise_timeout(p, abort_flag);
          break;
        }
      }
    }
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ activation producers
    const int pt = threadIdx.x - 128;
    const int wp = pt >> 5;
    const int half = lane & 1;
    int row[2];
    row[0] = 32 * wp + (lane >> 1);
    row[1] = row[0] + 16;

    // load cursor (runs kLook slices ahead of the convert cursor)
    int l_tile = blockIdx.x, l_kk = 0, l_cb = 0, l_r = 0, l_s = 0;
    int64_t l_img[2];
    int l_h0[2], l_w0[2];
    bool l_valid[2];
    auto set_tile = [&](int tile) {
      const int m0 = (tile / p.num_n_tiles) * Cfg::BM;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int m = m0 + row[j];
        l_valid[j] = m < p.M;
        const int mm = l_valid[j] ? m : 0;
        const int n = mm / p.PQ;
        const int pq = mm - n * p.PQ;
        const int pp = pq / p.Q;
        const int qq = pq - pp * p.Q;
        l_img[j] = static_cast<int64_t>(n) * p.img_stride;
        l_h0[j] = pp * p.stride_h - p.pad_h;
        l_w0[j] = qq * p.stride_w - p.pad_w;
      }
    };
    if (l_tile < p.num_tiles) set_tile(l_tile);
    const uint32_t stg_base = ptx::smem_addr(smem + Cfg::kOffStg);
    const int HW32 = p.H * p.W * 32;

    auto issue_load = [&](uint32_t slot) {
      if (l_tile < p.num_tiles) {
        const int dh = l_r * p.dil_h, dw = l_s * p.dil_w;
        const int cb_off = l_cb * HW32;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int h = l_h0[j] + dh, w = l_w0[j] + dw;
          const bool in = l_valid[j] && h >= 0 && h < p.H && w >= 0 && w < p.W;
          const int8_t* src = in ? p.x + l_img[j] + cb_off + (h * p.W + w) * 32 + half * 16 : p.x;
          ptx::cp_async_16_ca(stg_base + slot * Cfg::kStgBytes + row[j] * 32 + half * 16, src, in ? 16u : 0u);
        }
        // advance (cb, r, s) with s fastest; wrap into the next tile of this CTA
        if (++l_s == p.S) {
          l_s = 0;
          if (++l_r == p.R) {
            l_r = 0;
            ++l_cb;
          }
        }
        if (++l_kk == p.num_slices) {
          l_kk = 0;
          l_cb = 0;
          l_tile += gridDim.x;
          if (l_tile < p.num_tiles) set_tile(l_tile);
        }
      }
      ptx::cp_async_commit();
    };

    const uint32_t total = static_cast<uint32_t>((p.num_tiles - static_cast<int>(blockIdx.x) + gridDim.x - 1) /
                                                 gridDim.x) *
                           static_cast<uint32_t>(p.num_slices);
    for (int i = 0; i < Cfg::kLook; ++i) issue_load(static_cast<uint32_t>(i % Cfg::kStg));
    bool ok = true;
    for (uint32_t g = 0; g < total; ++g) {
      issue_load((g + Cfg::kLook) % Cfg::kStg);
      ptx::cp_async_wait<Cfg::kLook>();
      const uint32_t st = g % Cfg::kStages;
      if (!ptx::mbar_wait(&empty[st], ((g / Cfg::kStages) & 1u) ^ 1u, p.timeout_ns, abort_flag)) {
        ok = false;
        break;
      }
      const uint8_t* stg = smem + Cfg::kOffStg + (g % Cfg::kStg) * Cfg::kStgBytes;
      uint8_t* a_tile = smem + Cfg::kOffA + st * Cfg::kAStage;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const uint4 v = *reinterpret_cast<const uint4*>(stg + row[j] * 32 + half * 16);
        uint4 c0, c1;
        i8x4_to_f16x4(v.x, c0.x, c0.y);
        i8x4_to_f16x4(v.y, c0.z, c0.w);
        i8x4_to_f16x4(v.z, c1.x, c1.y);
        i8x4_to_f16x4(v.w, c1.z, c1.w);
        uint8_t* arow = a_tile + row[j] * 64;
        const int sw = (row[j] >> 1) & 3;
        *reinterpret_cast<uint4*>(arow + (((2 * half) ^ sw) << 4)) = c0;
        *reinterpret_cast<uint4*>(arow + (((2 * half + 1) ^ sw) << 4)) = c1;
      }
      ptx::fence_proxy_async_smem();
      if (!((p.debug_flags & 1) && g == 0 && pt == 0)) ptx::mbar_arrive(&full_a[st]);
    }
    if (!ok) raise_timeout(p, abort_flag);
    ptx::cp_async_wait_all();
  } else if (warp >= 8) {
    // ------------------------------------------------------------ epilogue
    const int qd = warp & 3;  // tensor-memory lane quarter of this warp
    const int row = 32 * qd + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(32 * qd) << 16;
    uint32_t u = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
      const int mt = tile / p.num_n_tiles, nt = tile % p.num_n_tiles;
      const int m = mt * Cfg::BM + row;
      const bool valid = m < p.M;
      const int mm = valid ? m : 0;
      const int n_img = mm / p.PQ;
      const int pq = mm - n_img * p.PQ;
      for (int c = 0; c < p.num_chunks; ++c, ++u) {
        const uint32_t buf = u % nb;
        // the tcgen05.ld below is warp-collective: decide as one warp
        const bool got = ptx::mbar_wait(&acc_full[buf], (u / nb) & 1u, p.timeout_ns, abort_flag);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t t_acc = tmem_base + lane_addr + buf * BN;
        const uint32_t t_run = tmem_base + lane_addr + nb * BN;
        const bool first = c == 0, last = c + 1 == p.num_chunks;
#pragma unroll 1
        for (int g32 = 0; g32 < BN / 32; ++g32) {
          const int k0 = nt * BN + g32 * 32;
          if (k0 >= p.K) break;
          uint32_t v[32];
          ptx::tmem_ld_32x32b_x32(t_acc + g32 * 32, v);
          ptx::tmem_wait_ld();
          int a[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) a[i] = __float2int_rn(__uint_as_float(v[i]));
          if (!first) {
            uint32_t rsum[32];
            ptx::tmem_ld_32x32b_x32(t_run + g32 * 32, rsum);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) a[i] += static_cast<int>(rsum[i]);
          }
          if (!last) {
            uint32_t w[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) w[i] = static_cast<uint32_t>(a[i]);
            ptx::tmem_st_32x32b_x32(t_run + g32 * 32, w);
          } else if (valid) {
            const int kb = k0 >> 5;
            const int64_t off = (static_cast<int64_t>(n_img) * p.KB + kb) * p.PQ + pq;
            if (p.out_mode == 0) {
              uint32_t o[8];
              requant32(p, k0, [&](int i) { return a[i]; }, o);
              uint4* dst = reinterpret_cast<uint4*>(p.y + off * 32);
              dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
              dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
            } else {
              int4* dst = reinterpret_cast<int4*>(p.acc + off * 32);
#pragma unroll
              for (int i = 0; i < 8; ++i) dst[i] = make_int4(a[4 * i], a[4 * i + 1], a[4 * i + 2], a[4 * i + 3]);
            }
          }
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(&acc_empty[buf]);
      }
    }
    if (!ok) raise_timeout(p, abort_flag);
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, p.tmem_cols);
  }
}

}  // namespace i8c
