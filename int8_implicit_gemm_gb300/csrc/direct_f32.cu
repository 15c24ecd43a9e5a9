// fp32 direct convolution on the SIMT cores: the second workload of the
// POPCORNBENCH kernel-benchmark trace (problem l1_p80: nn.Conv2d on fp32 NCHW
// input, KCRS weight and an optional bias, with per-axis stride, padding and
// dilation), where the result must match the framework's own convolution to
// atol = rtol = 1e-4.  Every product and sum is an IEEE fp32 fused
// multiply-add in a fixed order (input channel, filter row, filter column),
// so the result is within the fp32 summation bound of the exact sum; the
// tensor cores are not used (TF32 operands would round each input to 11
// significant bits, far outside that tolerance).
//
// Tiling: a CTA of 256 threads computes 64 output channels x 8 output rows x
// 32 output columns of one image.  Warp w owns channels 8w .. 8w + 7 of the
// tile and lane l output column l; each thread keeps 8 channels x 8 rows = 64
// accumulators in registers.  Per step of CS input channels the CTA stages in
// shared memory (double-buffered, cp.async):
//   - the input region its taps read, TH x TW floats per channel (zeros
//     outside the image), read by the lanes of a warp as consecutive columns;
//   - the weights of its 64 channels, R*S rows of 64 floats per channel, from
//     a copy of the weight transposed once per call to [C][R*S][Kpad] (read
//     as two broadcast 16-byte loads per tap).
// One tap is 8 input loads, 2 weight loads and 32 paired FMAs (64 FMAs) per
// thread.
#include <cuda_runtime.h>

#include <array>
#include <cstdint>
#include <map>
#include <mutex>

#include "i8conv.h"
#include "internal.h"

namespace i8c {
namespace {

constexpr int kThreads = 256;
constexpr int kTileP = 8;    // output rows per thread (and per tile)
constexpr int kTileQ = 32;   // output columns per tile: one per lane
constexpr int kTileK = 64;   // output channels per tile: 8 per warp
constexpr int kMaxSmem = 113 * 1024;  // two CTAs per SM

struct F32Params {
  const float* x;
  const float* wt;    // [C][R*S][Kpad]
  const float* bias;  // K floats or null
  float* y;
  int N, C, H, W, K, R, S, ph, pw, sh, sw, dh, dw, P, Q;
  int tiles_q, TH, TW, CS, Kpad;
  int in_floats;      // input floats per stage, rounded up to a multiple of 4
  int stage_floats;   // input + weights per stage
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

// w [K][C][R*S] -> wt [C][R*S][Kpad], zeros for k >= K.
__global__ void weight_transpose_kernel(const float* __restrict__ w, float* __restrict__ wt, int K, int C, int RS,
                                        int Kpad) {
  const int64_t total = static_cast<int64_t>(C) * RS * Kpad;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int k = static_cast<int>(i % Kpad);
    const int64_t crs = i / Kpad;  // c * RS + rs
    const int c = static_cast<int>(crs / RS);
    const int rs = static_cast<int>(crs - static_cast<int64_t>(c) * RS);
    wt[i] = k < K ? w[(static_cast<int64_t>(k) * C + c) * RS + rs] : 0.0f;
  }
}

__global__ void __launch_bounds__(kThreads, 2) conv_f32_direct_kernel(const F32Params p) {
  extern __shared__ __align__(16) float sm[];
  const int RS = p.R * p.S;
  const int tq = static_cast<int>(blockIdx.x) % p.tiles_q;
  const int tp = static_cast<int>(blockIdx.x) / p.tiles_q;
  const int n = blockIdx.y;
  const int kt = blockIdx.z;
  const int q0 = tq * kTileQ, p0 = tp * kTileP;
  const int h0 = p0 * p.sh - p.ph, w0 = q0 * p.sw - p.pw;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* xn = p.x + static_cast<int64_t>(n) * p.C * p.H * p.W;
  const float* wk = p.wt + kt * kTileK;
  const int thw = p.TH * p.TW;

  // Stage channels c0 .. c0 + CS - 1 into buffer buf (channels past C read as zeros).
  auto load_stage = [&](int c0, int buf) {
    float* si = sm + buf * p.stage_floats;
    float* sw = si + p.in_floats;
    for (int i = threadIdx.x; i < p.CS * thw; i += kThreads) {
      const int cc = i / thw;
      const int rem = i - cc * thw;
      const int row = rem / p.TW;
      const int col = rem - row * p.TW;
      const int c = c0 + cc, h = h0 + row, w = w0 + col;
      const bool in = c < p.C && h >= 0 && h < p.H && w >= 0 && w < p.W;
      const float* src = in ? xn + (static_cast<int64_t>(c) * p.H + h) * p.W + w : p.x;
      cp_async_4(smem_u32(si + i), src, in ? 4u : 0u);
    }
    for (int i = threadIdx.x; i < p.CS * RS * (kTileK / 4); i += kThreads) {
      const int row = i >> 4, part = i & 15;  // a row of 64 floats: 16 chunks of 16 bytes
      const int cc = row / RS;
      const int c = c0 + cc;
      const bool in = c < p.C;
      const float* src = in ? wk + (static_cast<int64_t>(c) * RS + (row - cc * RS)) * p.Kpad + part * 4 : p.wt;
      cp_async_16(smem_u32(sw + row * kTileK + part * 4), src, in ? 16u : 0u);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };

  // acc[k][j]: channel k, output rows 2j and 2j + 1 (one packed pair, so that
  // one paired fp32 FMA instruction updates both)
  float2 acc[8][kTileP / 2];
#pragma unroll
  for (int k = 0; k < 8; ++k)
#pragma unroll
    for (int j = 0; j < kTileP / 2; ++j) acc[k][j] = make_float2(0.0f, 0.0f);

  const int nst = (p.C + p.CS - 1) / p.CS;
  const int row_step = p.sh * p.TW;  // between the input rows of consecutive output rows
  load_stage(0, 0);
  for (int st = 0; st < nst; ++st) {
    if (st + 1 < nst) {
      load_stage((st + 1) * p.CS, (st + 1) & 1);
      asm volatile("cp.async.wait_group 1;" ::: "memory");
    } else {
      asm volatile("cp.async.wait_group 0;" ::: "memory");
    }
    __syncthreads();
    const float* si = sm + (st & 1) * p.stage_floats;
    const float* swt = si + p.in_floats;
    for (int cc = 0; cc < p.CS; ++cc) {
      for (int r = 0; r < p.R; ++r) {
        const float* irow = si + cc * thw + r * p.dh * p.TW + lane * p.sw;
        const float* wrow = swt + (cc * RS + r * p.S) * kTileK + warp * 8;
        for (int s = 0; s < p.S; ++s) {
          const float4 wa = *reinterpret_cast<const float4*>(wrow + s * kTileK);
          const float4 wb = *reinterpret_cast<const float4*>(wrow + s * kTileK + 4);
          const float wv[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
          const float* xc = irow + s * p.dw;
          float2 xv[kTileP / 2];
#pragma unroll
          for (int j = 0; j < kTileP / 2; ++j) xv[j] = make_float2(xc[2 * j * row_step], xc[(2 * j + 1) * row_step]);
          // each lane of the paired FMA is one IEEE fp32 fused multiply-add
          // (round to nearest), as __fmaf_rn on each row would be
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float2 w2 = make_float2(wv[k], wv[k]);
#pragma unroll
            for (int j = 0; j < kTileP / 2; ++j) acc[k][j] = __ffma2_rn(w2, xv[j], acc[k][j]);
          }
        }
      }
    }
    __syncthreads();  // the buffer is refilled by the next step's loads
  }

  const int q = q0 + lane;
  if (q >= p.Q) return;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int kk = kt * kTileK + warp * 8 + k;
    if (kk >= p.K) break;
    const float b = p.bias != nullptr ? p.bias[kk] : 0.0f;
    float* yk = p.y + (static_cast<int64_t>(n) * p.K + kk) * p.P * p.Q;
#pragma unroll
    for (int i = 0; i < kTileP; ++i) {
      const int pp = p0 + i;
      const float a = (i & 1) ? acc[k][i >> 1].y : acc[k][i >> 1].x;
      if (pp < p.P) yk[static_cast<int64_t>(pp) * p.Q + q] = __fadd_rn(a, b);
    }
  }
}

// The transposed weight copy, one per (device, K, C, R, S), kept until exit.
std::mutex g_wt_mu;
std::map<std::array<int, 5>, float*> g_wt;

}  // namespace
}  // namespace i8c

extern "C" i8c_status i8c_conv2d_fprop_f32(const float* x, const float* w, const float* bias, float* y,
                                           const i8c_conv_shape* shape, cudaStream_t stream) {
  using namespace i8c;
  if (x == nullptr || w == nullptr || y == nullptr || shape == nullptr) return I8C_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(w) | reinterpret_cast<uintptr_t>(y) |
       reinterpret_cast<uintptr_t>(bias)) & 3u)
    return I8C_ERR_MISALIGNED;
  const i8c_conv_shape& s = *shape;
  int32_t P = 0, Q = 0;
  i8c_status st = i8c_output_size(shape, &P, &Q);
  if (st != I8C_OK) return st;
  if (s.N > 65535 || (s.K + kTileK - 1) / kTileK > 65535) return I8C_ERR_UNSUPPORTED;
  const int64_t img = static_cast<int64_t>(s.C) * s.H * s.W, out_img = static_cast<int64_t>(s.K) * P * Q;
  if (img >= (int64_t{1} << 31) || out_img >= (int64_t{1} << 31)) return I8C_ERR_OVERFLOW_RISK;
  const int RS = s.R * s.S;
  F32Params p{};
  p.x = x;
  p.bias = bias;
  p.y = y;
  p.N = s.N; p.C = s.C; p.H = s.H; p.W = s.W; p.K = s.K; p.R = s.R; p.S = s.S;
  p.ph = s.pad_h; p.pw = s.pad_w; p.sh = s.stride_h; p.sw = s.stride_w; p.dh = s.dil_h; p.dw = s.dil_w;
  p.P = P; p.Q = Q;
  p.tiles_q = (Q + kTileQ - 1) / kTileQ;
  const int64_t tiles = static_cast<int64_t>(p.tiles_q) * ((P + kTileP - 1) / kTileP);
  if (tiles > 0x7fffffff) return I8C_ERR_OVERFLOW_RISK;
  const int64_t TH = static_cast<int64_t>(kTileP - 1) * s.stride_h + static_cast<int64_t>(s.R - 1) * s.dil_h + 1;
  const int64_t TW = static_cast<int64_t>(kTileQ - 1) * s.stride_w + static_cast<int64_t>(s.S - 1) * s.dil_w + 1;
  p.Kpad = (s.K + kTileK - 1) / kTileK * kTileK;
  // channels per step: two when two steps fit two CTAs per SM, else one
  int cs = 2;
  int64_t stage = 0;
  for (; cs >= 1; --cs) {
    const int64_t in_f = (cs * TH * TW + 3) / 4 * 4;
    stage = in_f + static_cast<int64_t>(cs) * RS * kTileK;
    if (2 * stage * 4 <= kMaxSmem) break;
  }
  if (cs < 1) return I8C_ERR_UNSUPPORTED;  // one channel's input region and weights do not fit
  if (cs > s.C) cs = s.C;
  p.CS = cs;
  p.TH = static_cast<int>(TH);
  p.TW = static_cast<int>(TW);
  p.in_floats = static_cast<int>((cs * TH * TW + 3) / 4 * 4);
  p.stage_floats = p.in_floats + cs * RS * kTileK;
  const int smem = 2 * p.stage_floats * static_cast<int>(sizeof(float));

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return I8C_ERR_CUDA;
  cudaDeviceProp prop;
  e = cudaGetDeviceProperties(&prop, dev);
  if (e != cudaSuccess) return I8C_ERR_CUDA;
  if (prop.major != 10 || prop.minor != 3) return I8C_ERR_NO_DEVICE;
  float* wt = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_wt_mu);
    const std::array<int, 5> key{dev, s.K, s.C, s.R, s.S};
    auto it = g_wt.find(key);
    if (it != g_wt.end()) {
      wt = it->second;
    } else {
      e = cudaMalloc(&wt, sizeof(float) * static_cast<size_t>(p.Kpad) * s.C * RS);
      if (e != cudaSuccess) return I8C_ERR_CUDA;
      g_wt[key] = wt;
    }
  }
  p.wt = wt;
  // per device: set on every call (a host-side attribute write)
  if (cudaFuncSetAttribute(conv_f32_direct_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem) !=
      cudaSuccess)
    return I8C_ERR_CUDA;

  const int64_t wt_elems = static_cast<int64_t>(p.Kpad) * s.C * RS;
  int64_t blocks = (wt_elems + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  weight_transpose_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(w, wt, s.K, s.C, RS, p.Kpad);
  g_launches.fetch_add(1, std::memory_order_relaxed);
  e = cudaGetLastError();
  if (e != cudaSuccess) return I8C_ERR_CUDA;
  const dim3 grid(static_cast<unsigned>(tiles), static_cast<unsigned>(s.N),
                  static_cast<unsigned>((s.K + kTileK - 1) / kTileK));
  conv_f32_direct_kernel<<<grid, kThreads, smem, stream>>>(p);
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return cudaGetLastError() == cudaSuccess ? I8C_OK : I8C_ERR_CUDA;
}
