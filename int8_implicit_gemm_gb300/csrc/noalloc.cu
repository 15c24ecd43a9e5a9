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

// Per device: whether it was checked to be an sm_103 device, its SM count,
// and whether this entry point has run there (so its status word means
// something).  The scratch array's device address and the kernels' shared
// memory limit are looked up again on every call, since a device reset
// (cudaDeviceReset, or a torn-down primary context) invalidates both.
struct DeviceSetup {
  bool checked = false;
  bool used = false;
  int num_sms = 0;
};

std::mutex g_setup_mu;
DeviceSetup g_setup[kMaxDevices];
int g_debug_flags = 0;       // test hooks (i8c_debug_set_oneshot)
int g_timeout_us = 0;        // 0: 2 s

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

// With device `dev` current: check it once, then (every call) look up the
// device address of the scratch array -- the host-side name is only a
// stand-in -- and raise the kernels' shared-memory limit.  Nothing here
// allocates.
i8c_status setup_device(int dev, unsigned char** scratch, int* num_sms) {
  if (dev < 0 || dev >= kMaxDevices) return I8C_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  DeviceSetup& s = g_setup[dev];
  if (!s.checked) {
    int major = 0, minor = 0, sms = 0;
    cudaError_t e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return status_of(e);
    if (major != 10 || minor != 3) return I8C_ERR_NO_DEVICE;
    s.num_sms = sms;
    s.checked = true;
  }
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess || p == nullptr) return e != cudaSuccess ? status_of(e) : I8C_ERR_CUDA;
  for (int bn : {32, 64, 128, 256}) {
    e = i8c::conv_prepare(bn);
    if (e != cudaSuccess) return status_of(e);
  }
  s.used = true;
  *scratch = static_cast<unsigned char*>(p);
  *num_sms = s.num_sms;
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
  unsigned char* scratch = nullptr;
  int num_sms = 0;
  st = setup_device(dev, &scratch, &num_sms);
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

  int* status = reinterpret_cast<int*>(scratch);
  uint16_t* f16 = reinterpret_cast<uint16_t*>(scratch + kStatusBytes);

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
  int debug_flags = 0, timeout_us = 0;
  {
    std::lock_guard<std::mutex> lock(g_setup_mu);
    debug_flags = g_debug_flags;
    timeout_us = g_timeout_us;
  }
  p.timeout_ns = static_cast<uint64_t>(timeout_us > 0 ? timeout_us : 2000000) * 1000ull;
  p.out_mode = 0;
  p.debug_flags = debug_flags;
  const int ctas = num_sms < p.num_tiles ? num_sms : p.num_tiles;
  return status_of(i8c::launch_conv(bn, tmap, p, ctas, stream));
}

namespace i8c {

int noalloc_take_status(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return I8C_OK;
  {
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (!g_setup[dev].used) return I8C_OK;
  }
  int h = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&h, g_noalloc_scratch, sizeof(int), 0, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return status_of(e);
  if (h != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_noalloc_scratch, &zero, sizeof(int), 0, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return status_of(e);
  }
  return h;
}

void noalloc_set_debug(int debug_flags, int timeout_us) {
  std::lock_guard<std::mutex> lock(g_setup_mu);
  g_debug_flags = debug_flags;
  g_timeout_us = timeout_us;
}

}  // namespace i8c
