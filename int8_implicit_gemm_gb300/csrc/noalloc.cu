// i8c_conv2d_fprop_noalloc: the convolution for callers that must not
// allocate device memory.
//
// The regular entry points keep the fp16 copy of the filter and the device
// status word in memory that a plan allocates with cudaMalloc.  Some callers
// cannot allow that: code running where the allocator is owned by someone
// else (a framework's caching allocator, a memory-pool budget fixed at start
// up), real-time paths where cudaMalloc's implicit device synchronisation is
// not acceptable, or plug-ins that are handed buffers and forbidden to grow
// the process footprint.  This entry point instead uses one fixed scratch
// array compiled into the library (static __device__ storage, reserved on
// every GPU that loads the library until the process exits) and calls no
// allocating routine at all.
#include <cudaTypedefs.h>

#include <mutex>

#include "../../include/i8conv.h"
#include "internal.h"

namespace {

// Scratch layout: [0, 256) device status word (zeroed by every call),
// [256, end) fp16 copy of the filter, [C/32][R][S][K][32].
constexpr size_t kScratchBytes = size_t(8) << 20;
constexpr size_t kStatusBytes = 256;
constexpr int64_t kMaxFilterElems = static_cast<int64_t>((kScratchBytes - kStatusBytes) / 2);

}  // namespace

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

namespace {

constexpr int kMaxDevices = 64;

struct DeviceSetup {
  bool ready = false;
  unsigned char* scratch = nullptr;  // device address of g_noalloc_scratch on this device
  int num_sms = 0;
};

std::mutex g_setup_mu;
DeviceSetup g_setup[kMaxDevices];

using EncodeTiled = PFN_cuTensorMapEncodeTiled_v12000;

EncodeTiled encode_fn() {
  static EncodeTiled fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(p);
  });
  return fn;
}

i8c_status status_of(cudaError_t e) {
  if (e == cudaSuccess) return I8C_OK;
  if (e == cudaErrorNoDevice || e == cudaErrorInsufficientDriver) return I8C_ERR_NO_DEVICE;
  return I8C_ERR_CUDA;
}

// Once per device, with that device current: look up the device address of
// the scratch array (the host-side name is only a stand-in) and prepare the
// kernels.  Nothing here allocates.
i8c_status setup_device(int dev, DeviceSetup* out) {
  if (dev < 0 || dev >= kMaxDevices) return I8C_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  DeviceSetup& s = g_setup[dev];
  if (!s.ready) {
    int major = 0, minor = 0, sms = 0;
    cudaError_t e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return status_of(e);
    if (major != 10 || minor != 3) return I8C_ERR_NO_DEVICE;
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) return e != cudaSuccess ? status_of(e) : I8C_ERR_CUDA;
    for (int bn : {32, 64, 128, 256}) {
      e = i8c::conv_prepare(bn);
      if (e != cudaSuccess) return status_of(e);
    }
    s.scratch = static_cast<unsigned char*>(p);
    s.num_sms = sms;
    s.ready = true;
  }
  *out = s;
  return I8C_OK;
}

bool aligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" i8c_status i8c_conv2d_fprop_noalloc(const int8_t* x, const int8_t* f, int8_t* y,
                                               const i8c_conv_shape* shape, float alpha, cudaStream_t stream) {
  if (x == nullptr || f == nullptr || y == nullptr || shape == nullptr) return I8C_ERR_INVALID_ARG;
  if (!aligned(x) || !aligned(f) || !aligned(y)) return I8C_ERR_MISALIGNED;
  i8c_status st = i8c_supported(shape);
  if (st != I8C_OK) return st;
  int32_t P = 0, Q = 0;
  st = i8c_output_size(shape, &P, &Q);
  if (st != I8C_OK) return st;
  const i8c_conv_shape& s = *shape;
  const int64_t filter_elems = static_cast<int64_t>(s.K) * s.C * s.R * s.S;
  if (filter_elems > kMaxFilterElems) return I8C_ERR_UNSUPPORTED;  // does not fit the static scratch

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return status_of(e);
  DeviceSetup ds;
  st = setup_device(dev, &ds);
  if (st != I8C_OK) return st;
  EncodeTiled encode = encode_fn();
  if (encode == nullptr) return I8C_ERR_CUDA;

  // The same schedule as a default plan.
  const int bn = s.K <= 32 ? 32 : (s.K <= 64 ? 64 : (s.K <= 128 ? 128 : 256));
  const int64_t M = static_cast<int64_t>(s.N) * P * Q;
  const int num_n_tiles = (s.K + bn - 1) / bn;
  const int64_t tiles = ((M + 127) / 128) * num_n_tiles;
  if (tiles > 2147483647LL) return I8C_ERR_OVERFLOW_RISK;
  const int num_slices = (s.C / 32) * s.R * s.S;
  const int num_chunks = (num_slices + 31) / 32;
  const int chunk_slices = (num_slices + num_chunks - 1) / num_chunks;
  const int run_cols = num_chunks > 1 ? bn : 0;
  const int acc_buffers = (2 * bn + run_cols <= 512) ? 2 : 1;
  int tmem_cols = 32;
  while (tmem_cols < acc_buffers * bn + run_cols) tmem_cols <<= 1;

  int* status = reinterpret_cast<int*>(ds.scratch);
  uint16_t* f16 = reinterpret_cast<uint16_t*>(ds.scratch + kStatusBytes);

  cuuint64_t dims[3] = {32, static_cast<cuuint64_t>(s.K), static_cast<cuuint64_t>(num_slices)};
  cuuint64_t strides[2] = {64, static_cast<cuuint64_t>(s.K) * 64};
  cuuint32_t box[3] = {32, static_cast<cuuint32_t>(bn), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUtensorMap tmap;
  if (encode(&tmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, f16, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return I8C_ERR_CUDA;

  // the status word must start at zero; the fp16 filter is fully rewritten
  e = cudaMemsetAsync(status, 0, sizeof(int), stream);
  if (e != cudaSuccess) return status_of(e);
  e = i8c::launch_filter_to_f16(f, f16, filter_elems, stream);
  if (e != cudaSuccess) return status_of(e);

  i8c::ConvParams p{};
  p.x = x;
  p.y = y;
  p.acc = nullptr;
  p.status = status;
  p.alpha = alpha;
  p.H = s.H;
  p.W = s.W;
  p.K = s.K;
  p.pad_h = s.pad_h;
  p.pad_w = s.pad_w;
  p.stride_h = s.stride_h;
  p.stride_w = s.stride_w;
  p.dil_h = s.dil_h;
  p.dil_w = s.dil_w;
  p.R = s.R;
  p.S = s.S;
  p.P = P;
  p.Q = Q;
  p.PQ = P * Q;
  p.M = static_cast<int>(M);
  p.CB = s.C / 32;
  p.KB = s.K / 32;
  p.num_slices = num_slices;
  p.chunk_slices = chunk_slices;
  p.num_chunks = num_chunks;
  p.num_n_tiles = num_n_tiles;
  p.num_tiles = static_cast<int>(tiles);
  p.acc_buffers = acc_buffers;
  p.tmem_cols = static_cast<uint32_t>(tmem_cols);
  p.img_stride = static_cast<int64_t>(s.C) * s.H * s.W;
  p.timeout_ns = 2000000000ull;
  p.out_mode = 0;
  p.debug_flags = 0;
  const int ctas = ds.num_sms < p.num_tiles ? ds.num_sms : p.num_tiles;
  return status_of(i8c::launch_conv(bn, tmap, p, ctas, stream));
}
