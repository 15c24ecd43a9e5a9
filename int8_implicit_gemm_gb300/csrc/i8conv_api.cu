// Host side of the C-ABI: argument checks, plans, the filter tensor map, and
// launches.  See include/i8conv.h for the contract of each entry point.
#include <cudaTypedefs.h>

#include <array>
#include <cstring>
#include <map>
#include <mutex>
#include <new>
#include <utility>
#include <vector>

#include "../../include/i8conv.h"
#include "internal.h"

using i8c::ConvParams;

struct i8c_plan {
  i8c_conv_shape shape;
  int P, Q;
  int64_t M;
  int device;
  int kernel_variant;  // 1 = per-tap gather kernel, 2 = halo kernel, 3 = halo kernel on CTA pairs
  int cta_group;       // CTAs per MMA tile: 2 for variant 3, else 1
  int split_tiles;     // halo kernel: tiles of the last wave split along the channel blocks
  int block_n, num_n_tiles, num_m_tiles, num_tiles, num_ctas;
  i8c::HaloParams halo;  // geometry and shared-memory layout of the halo kernel
  int num_slices, chunk_slices, num_chunks, acc_buffers;
  uint32_t tmem_cols;
  int smem_bytes;
  uint64_t timeout_ns;
  int debug_flags;
  uint16_t* f16;   // fp16 copy of the filter, [C/32][R][S][K][32]
  int* status;     // device status word
  long long* trace;  // clock64 trace of CTA 0 (debug flag I8C_DEBUG_TRACE), kTraceRows * kTraceSlots entries
  CUtensorMap tmap;
  // TMA-fed halos: the activations' tensor map, encoded for the x pointer of
  // the last run (a run with another x encodes it again)
  mutable CUtensorMap tmap_x;
  mutable const int8_t* tmap_x_ptr;
  int8_t *stage_x, *stage_f, *stage_y;  // device staging for host-buffer runs (optional)
  // host_staging = 2: a second staging set and the pipelined host-buffer
  // runs' copy streams and ordering events (set b: in_done, run_done, out_done)
  int8_t *stage_x2, *stage_f2, *stage_y2;
  cudaStream_t s_in, s_out;
  cudaEvent_t ev_begin, ev_in[2], ev_run[2], ev_out[2];
  uint32_t* gbar;        // halo kernel converting the filter itself: grid barrier {arrivals, generation}
  int* split_count;      // halo kernel, split tail tiles: arrivals per tile and CTA rank
  int32_t* split_part;   // halo kernel, split tail tiles: int32 partial sums
  size_t x_bytes, f_bytes, y_bytes;
  size_t f16_bytes;  // the fp16 filter copy
  int64_t workspace_bytes;
  // optional per-launch timing of the convolution kernel
  std::vector<cudaEvent_t> ev_start, ev_end;
  mutable int64_t ev_recorded = 0;
  // i8c_plan_set_filter was called: f16 holds the operand copy (or, for a
  // kernel that writes its resident filter itself, an int8 copy of f)
  mutable bool prepacked = false;
  // set_filter's conversion (or copy) may be the kernel launched just before
  // the next prepacked run, which must then wait for it before reading
  mutable bool filter_fresh = false;
};

namespace {

constexpr int64_t kMaxI32 = 2147483647LL;
// Whether the automatic plan takes the stacked-tap kernel for the 64-channel
// layers it suits (with a resident filter).
constexpr bool kStackAuto = false;

i8c_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return I8C_OK;
  if (e == cudaErrorNoDevice || e == cudaErrorInsufficientDriver) return I8C_ERR_NO_DEVICE;
  return I8C_ERR_CUDA;
}

int64_t extent(int64_t in, int64_t pad, int64_t dil, int64_t k, int64_t stride) {
  const int64_t num = in + 2 * pad - dil * (k - 1) - 1;
  if (num < 0) return 0;
  return num / stride + 1;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

i8c_status check_shape(const i8c_conv_shape* s, int64_t* P, int64_t* Q) {
  if (s == nullptr) return I8C_ERR_INVALID_ARG;
  if (s->N < 1 || s->C < 1 || s->H < 1 || s->W < 1 || s->K < 1 || s->R < 1 || s->S < 1) return I8C_ERR_INVALID_ARG;
  if (s->pad_h < 0 || s->pad_w < 0 || s->stride_h < 1 || s->stride_w < 1 || s->dil_h < 1 || s->dil_w < 1)
    return I8C_ERR_INVALID_ARG;
  *P = extent(s->H, s->pad_h, s->dil_h, s->R, s->stride_h);
  *Q = extent(s->W, s->pad_w, s->dil_w, s->S, s->stride_w);
  if (*P < 1 || *Q < 1) return I8C_ERR_UNSUPPORTED;
  return I8C_OK;
}

i8c_status check_supported(const i8c_conv_shape* s, int64_t* P, int64_t* Q) {
  i8c_status st = check_shape(s, P, Q);
  if (st != I8C_OK) return st;
  if (s->C % 32 != 0 || s->K % 32 != 0) return I8C_ERR_UNSUPPORTED;
  // |acc| <= C*R*S*128*128 must fit int32
  if (static_cast<int64_t>(s->C) * s->R * s->S * 16384 > kMaxI32) return I8C_ERR_OVERFLOW_RISK;
  // 32-bit element offsets inside one image, 32-bit GEMM row count
  const int64_t img = static_cast<int64_t>(s->C) * s->H * s->W;
  const int64_t out_img = static_cast<int64_t>(s->K) * (*P) * (*Q);
  const int64_t M = static_cast<int64_t>(s->N) * (*P) * (*Q);
  if (img > kMaxI32 || out_img > kMaxI32 || M > kMaxI32 - 256) return I8C_ERR_OVERFLOW_RISK;
  return I8C_OK;
}

using EncodeTiled = PFN_cuTensorMapEncodeTiled_v12000;

EncodeTiled get_encode_tiled() {
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

int next_pow2(int v) {
  int p = 32;
  while (p < v) p <<= 1;
  return p;
}

double wave_efficiency(int64_t tiles, int ctas) {
  const int64_t waves = (tiles + ctas - 1) / ctas;
  return static_cast<double>(tiles) / static_cast<double>(waves * ctas);
}

// The TMA box that carries one channel block of a tile's halo into shared
// memory (int8, 32 bytes per position): for 2-D patches the halo region
// itself (CW columns x HR rows, natural column order); for flat tiles the
// whole zero-padded input rows (W + 2*pad_w wide) that the run of
// `positions` padded positions can span, from any starting column.  TMA
// boxes are at most 256 elements per dimension.  Returns false when the box
// does not fit that limit.
bool tma_halo_box(const i8c_conv_shape& s, const i8c::HaloParams& h, i8c::HaloParams* out) {
  const int64_t bw = h.CW;
  const int64_t bh = h.flat ? (h.CW - 1 + static_cast<int64_t>(h.positions) + h.CW - 1) / h.CW : h.HR;
  if (bw > 256 || bh > 256 || bw < 1 || bh < 1) return false;
  if (h.flat && h.CW != s.W + 2 * s.pad_w) return false;
  out->box_w = static_cast<int>(bw);
  out->box_h = static_cast<int>(bh);
  out->x8_box = static_cast<uint32_t>(32 * bw * bh);
  out->x8_bytes = (out->x8_box + 1023) / 1024 * 1024;
  return true;
}

// Halo geometry and shared-memory layout of the halo kernel for tile width bn
// on cg CTAs (each CTA of a pair stages bn/2 filter rows): two fp16 halo
// stages, the int8 staging ring (if any), the filter stages, the barriers.
// loads: 0 = auto, 1 = staging ring only, 2 = register loads only.  Returns
// false when the halo does not fit with at least three filter stages.
bool halo_layout(const i8c_conv_shape& s, int P, int Q, int bn, int cg, int loads, bool flat, i8c::HaloParams* h,
                 int* smem_bytes, bool wide = false) {
  if (s.stride_w > 8) return false;
  if (flat && (s.stride_h != 1 || s.stride_w != 1)) return false;
  // 16x16 patches (two 16x8 sub-tiles on one halo): 2-D patches, at most 128
  // channels per tile, register or staged halo loads, whole filter rows per
  // filter stage (checked by the caller)
  if (wide && (flat || bn > 128 || loads == 3)) return false;
  *h = i8c::HaloParams{};
  h->flat = flat ? 1 : 0;
  h->subtiles = wide ? 2 : 1;
  const int pw_out = wide ? 16 : 8;  // output columns per patch
  int64_t HR, CW, npos, patches;
  if (flat) {
    // flat tiles: 128 consecutive pixels of the output laid out with the
    // padded input's row width; their taps read one contiguous run
    CW = static_cast<int64_t>(s.W) + 2LL * s.pad_w;
    npos = 128 + static_cast<int64_t>(s.R - 1) * s.dil_h * CW + static_cast<int64_t>(s.S - 1) * s.dil_w;
    HR = (npos + CW - 1) / CW;
    const int64_t tpi = (static_cast<int64_t>(P) * CW + 127) / 128;
    if (tpi > kMaxI32) return false;
    h->tpi = static_cast<int>(tpi);
    h->tile_px = 128;
    patches = static_cast<int64_t>(s.N) * tpi;
  } else {
    h->TPH = (P + 15) / 16;
    h->TQW = (Q + pw_out - 1) / pw_out;
    patches = static_cast<int64_t>(s.N) * h->TPH * h->TQW;
    HR = 15LL * s.stride_h + static_cast<int64_t>(s.R - 1) * s.dil_h + 1;
    CW = static_cast<int64_t>(pw_out - 1) * s.stride_w + static_cast<int64_t>(s.S - 1) * s.dil_w + 1;
    npos = HR * CW;
  }
  if (patches > kMaxI32) return false;
  h->num_patches = static_cast<int>(patches);
  if (npos > 65536 || CW > 65536) return false;
  h->HR = static_cast<int>(HR);
  h->CW = static_cast<int>(CW);
  h->positions = static_cast<int>(npos);
  const uint32_t pos = static_cast<uint32_t>(npos);
  h->plane_bytes = (pos * 16 + 127) / 128 * 128;
  h->halo_bytes = 4 * h->plane_bytes;
  h->stg_bytes = (pos * 32 + 127) / 128 * 128;
  int off = 0;
  for (int f = 0; f < s.stride_w; ++f) {
    h->phase_off[f] = off;
    off += static_cast<int>((CW - f + s.stride_w - 1) / s.stride_w);
  }
  h->phase_off[s.stride_w] = off;
  // Filter stages of G K-slices each: a run of taps of one channel block,
  // either part of a filter row (G divides S) or whole rows (S divides G, G
  // divides R*S).  Longer stages need fewer barrier waits per MMA, so the
  // largest G is taken that leaves at least three stages (two for whole-row
  // stages, which are long enough to double-buffer) beside the halo.  The
  // producers load into registers unless the staging ring (three slots, else
  // two) is asked for: measured on the 3x3 layers, the ring's deeper prefetch
  // gains nothing and costs filter stages.
  const int budget = i8c::kMaxDynamicSmem - 1024 - i8c::kHaloBarBytes;
  static const int kSlots[3] = {3, 2, 0};
  const int first = loads == 1 ? 0 : 2, last = loads == 1 ? 1 : 2;
  const int RS = s.R * s.S;
  // TMA-fed halos (loads == 3): one to three int8 slots of one box each; the
  // most that leave the filter enough stages, and one where more would cost
  // the filter its residency (one output-channel tile whose every stage fits)
  const bool tma = loads == 3;
  if (tma && !tma_halo_box(s, *h, h)) return false;
  const int n_tiles = (s.K + bn - 1) / bn;
  for (int G = RS; G >= 1; --G) {
    const bool part_row = s.S % G == 0;
    const bool whole_rows = G % s.S == 0 && RS % G == 0;
    if (!(part_row || whole_rows) || G > 32) continue;
    const int min_stages = part_row ? 3 : 2;
    // a stage that holds a whole channel block leaves the producers one
    // stage of slack with two halo stages: give them a third when it fits.
    // With the staging ring, a single fp16 halo stage is allowed as a last
    // resort: the ring already holds the next channel blocks' loads, and only
    // the shared-memory conversion of each block waits for the MMAs.
    for (int nhs = G == RS ? 3 : 2; nhs >= (loads == 1 ? 1 : 2); --nhs)
    for (int k = first; k <= last; ++k) {
      const int nstg = tma ? 0 : kSlots[k];
      const int64_t stage = static_cast<int64_t>(G) * (bn / cg) * 64;
      const int64_t need_resident = (s.C / 32) * RS / G;
      int64_t off_x8 = 0, off_b = 0, nbs = 0;
      int nxs = 0;
      for (int nx = tma ? 3 : 0; nx >= 0; --nx) {  // TMA: three slots, else fewer; no TMA: none
        const int64_t off_stg = static_cast<int64_t>(nhs) * h->halo_bytes;
        const int64_t ox = (off_stg + static_cast<int64_t>(nstg) * h->stg_bytes + 1023) / 1024 * 1024;
        const int64_t ob = (ox + static_cast<int64_t>(nx) * h->x8_bytes + 1023) / 1024 * 1024;
        int64_t n = (budget - ob) / stage;
        if (n > i8c::kMaxBStages) n = i8c::kMaxBStages;
        if (n < min_stages) {
          if (tma && nx > 1) continue;
          break;
        }
        if (tma && nx >= 2 && n_tiles == 1 && n < need_resident) {
          // would one slot keep the filter resident?
          const int64_t ob1 = (ox + h->x8_bytes + 1023) / 1024 * 1024;
          const int64_t n1 = (budget - ob1) / stage;
          if (n1 >= need_resident && need_resident <= i8c::kMaxBStages) continue;
        }
        off_x8 = ox;
        off_b = ob;
        nbs = n;
        nxs = nx;
        break;
      }
      if (nbs < min_stages || (tma && nxs < 1)) continue;
      h->bgroup = G;
      h->nhs = nhs;
      h->nstg = nstg;
      h->nbs = static_cast<int>(nbs);
      h->tma_halo = tma ? 1 : 0;
      h->nxs = nxs;
      h->off_x8 = static_cast<uint32_t>(off_x8);
      h->off_stg = static_cast<uint32_t>(static_cast<int64_t>(nhs) * h->halo_bytes);
      h->off_b = static_cast<uint32_t>(off_b);
      h->off_bar = static_cast<uint32_t>(off_b + nbs * stage);
      *smem_bytes = static_cast<int>(h->off_bar) + i8c::kHaloBarBytes + 1024;
      return true;
    }
  }
  return false;
}

// Layout of the transposed-tile kernel for np output pixels per CTA and cg
// CTAs per MMA tile (stride 1 only): the flat halo of np + (R-1)*dh*CW +
// (S-1)*dw padded input positions per channel block, two or three halo
// stages and at least two filter stages of G K-slices x 128 output channels,
// and the epilogue's output staging rows (the MMA's cg * np pixels x 128
// channels, int8).  G is want_g if given,
// else the longest divisor of R*S that fits.  nstg > 0: an int8 staging ring
// of nstg slots that cp.async fills nstg - 1 channel blocks ahead.  Returns
// false when nothing fits.
bool tr_layout(const i8c_conv_shape& s, int P, int np, int cg, int want_g, int nstg, i8c::HaloParams* h,
               int* smem_bytes, bool tma = false) {
  if (s.stride_h != 1 || s.stride_w != 1) return false;
  const int mma_n = cg * np;
  if (mma_n < 16 || mma_n > 256 || mma_n % 16 != 0 || np % 8 != 0) return false;
  *h = i8c::HaloParams{};
  h->flat = 1;
  h->tile_px = np;
  const int64_t CW = static_cast<int64_t>(s.W) + 2LL * s.pad_w;
  const int64_t npos = np + static_cast<int64_t>(s.R - 1) * s.dil_h * CW + static_cast<int64_t>(s.S - 1) * s.dil_w;
  const int64_t tpi = (static_cast<int64_t>(P) * CW + np - 1) / np;
  const int64_t patches = static_cast<int64_t>(s.N) * tpi;
  if (tpi > kMaxI32 || patches > kMaxI32 || npos > 65536 || CW > 65536) return false;
  h->tpi = static_cast<int>(tpi);
  h->num_patches = static_cast<int>(patches);
  h->HR = static_cast<int>((npos + CW - 1) / CW);
  h->CW = static_cast<int>(CW);
  h->positions = static_cast<int>(npos);
  h->plane_bytes = (static_cast<uint32_t>(npos) * 16 + 127) / 128 * 128;
  h->halo_bytes = 4 * h->plane_bytes;
  h->stg_bytes = (static_cast<uint32_t>(npos) * 32 + 127) / 128 * 128;
  h->phase_off[0] = 0;
  h->phase_off[1] = static_cast<int>(CW);
  const int budget = i8c::kMaxDynamicSmem - 1024 - i8c::kHaloBarBytes;
  const int RS = s.R * s.S;
  const int64_t stage_unit = 128 * 64;  // one K-slice of 128 output channels, fp16
  const int64_t out_bytes = static_cast<int64_t>(mma_n) * 128;
  if (tma) {
    if (!tma_halo_box(s, *h, h)) return false;
    nstg = 0;
  }
  for (int G = RS < 32 ? RS : 32; G >= 1; --G) {
    if (RS % G != 0 || (want_g != 0 && G != want_g)) continue;
    const int64_t stage = G * stage_unit;
    // halo stages (2 or 3) and TMA slots (2 or 1; none without TMA): the
    // first combination in this order that leaves two filter stages; a third
    // halo stage only when it costs no filter stage
    int nhs = 0, nxs = 0;
    int64_t nbs = 0, off_x8 = 0, off_b = 0;
    const int64_t stg = static_cast<int64_t>(nstg) * h->stg_bytes;
    auto fit = [&](int nh, int nx, int64_t* ox, int64_t* ob) {
      *ox = (static_cast<int64_t>(nh) * h->halo_bytes + stg + 1023) / 1024 * 1024;
      *ob = (*ox + static_cast<int64_t>(nx) * h->x8_bytes + 1023) / 1024 * 1024;
      const int64_t n = (budget - *ob - out_bytes) / stage;
      return n > i8c::kMaxBStages ? static_cast<int64_t>(i8c::kMaxBStages) : n;
    };
    for (int nx = tma ? 2 : 0; nx >= (tma ? 1 : 0) && nbs < 2; --nx) {
      int64_t ox3, ob3, ox2, ob2;
      const int64_t n3 = fit(3, nx, &ox3, &ob3), n2 = fit(2, nx, &ox2, &ob2);
      if (n3 >= 2 && n3 >= n2) {
        nhs = 3, nxs = nx, nbs = n3, off_x8 = ox3, off_b = ob3;
      } else if (n2 >= 2) {
        nhs = 2, nxs = nx, nbs = n2, off_x8 = ox2, off_b = ob2;
      }
    }
    if (nbs < 2) continue;
    h->bgroup = G;
    h->nhs = nhs;
    h->nstg = nstg;
    h->nbs = static_cast<int>(nbs);
    h->tma_halo = tma ? 1 : 0;
    h->nxs = nxs;
    h->off_x8 = static_cast<uint32_t>(off_x8);
    h->off_stg = static_cast<uint32_t>(nhs * h->halo_bytes);
    h->off_b = static_cast<uint32_t>(off_b);
    h->off_out = static_cast<uint32_t>(off_b + nbs * stage);
    h->off_bar = static_cast<uint32_t>(h->off_out + out_bytes);
    *smem_bytes = static_cast<int>(h->off_bar) + i8c::kHaloBarBytes + 1024;
    return true;
  }
  return false;
}

// Layout of the stacked-tap kernel (64 output channels, stride 1, CTA
// pairs): per 32-channel block a halo of R segments of L = 128 + (S-1)*dw
// input positions (one per filter row), two or three halo stages, the
// epilogue's shift buffers, and filter stages of one filter row's U = ceil(S/2)
// slots of 64 fp16 rows per CTA.  The filter is kept resident when all
// (C/32)*R stages fit: three halo stages when that still holds, else two.
// Returns false when the shape does not suit the kernel or nothing fits.
bool stack_layout(const i8c_conv_shape& s, int P, int Q, i8c::HaloParams* h, int* smem_bytes) {
  if (s.K != 64 || s.stride_h != 1 || s.stride_w != 1 || s.S < 2 || s.S > 16 || s.dil_w > 8) return false;
  *h = i8c::HaloParams{};
  const int U = (s.S + 1) / 2;
  const int64_t L = 128 + static_cast<int64_t>(s.S - 1) * s.dil_w;
  const int64_t npos = static_cast<int64_t>(s.R) * L;
  const int vq = 128 - s.dil_w;
  const int64_t tq = (static_cast<int64_t>(Q) + vq - 1) / vq;
  const int64_t tiles = static_cast<int64_t>(s.N) * P * tq;
  if (npos > 65536 || tiles > kMaxI32 - 1) return false;
  h->seg_len = static_cast<int>(L);
  h->vq = vq;
  h->tq = static_cast<int>(tq);
  h->slots = U;
  h->num_patches = static_cast<int>(tiles);
  h->HR = s.R;
  h->CW = static_cast<int>(L);
  h->positions = static_cast<int>(npos);
  h->plane_bytes = (static_cast<uint32_t>(npos) * 16 + 127) / 128 * 128;
  h->halo_bytes = 4 * h->plane_bytes;
  h->phase_off[0] = 0;
  h->phase_off[1] = static_cast<int>(L);
  h->bgroup = U;
  const int budget = i8c::kMaxDynamicSmem - 1024 - i8c::kHaloBarBytes;
  const int64_t stage = static_cast<int64_t>(U) * 64 * 64;
  const int stages = (s.C / 32) * s.R;
  int64_t nbs_for[4] = {0, 0, 0, 0}, off_b_for[4] = {0, 0, 0, 0};
  for (int nhs = 2; nhs <= 3; ++nhs) {
    off_b_for[nhs] = (static_cast<int64_t>(nhs) * h->halo_bytes + i8c::kStackXbufBytes + 1023) / 1024 * 1024;
    const int64_t n = (budget - off_b_for[nhs]) / stage;
    nbs_for[nhs] = n > i8c::kMaxBStages ? i8c::kMaxBStages : n;
  }
  int nhs = nbs_for[3] >= stages ? 3 : 2;
  if (nbs_for[nhs] < (stages < 2 ? stages : 2)) return false;
  h->nhs = nhs;
  h->nstg = 0;
  h->resident = nbs_for[nhs] >= stages ? 1 : 0;
  h->nbs = static_cast<int>(h->resident ? stages : nbs_for[nhs]);
  h->off_stg = static_cast<uint32_t>(nhs * h->halo_bytes);
  h->off_out = h->off_stg;
  h->off_b = static_cast<uint32_t>(off_b_for[nhs]);
  h->off_bar = static_cast<uint32_t>(off_b_for[nhs] + static_cast<int64_t>(h->nbs) * stage);
  *smem_bytes = static_cast<int>(h->off_bar) + i8c::kHaloBarBytes + 1024;
  return true;
}

void free_plan_memory(i8c_plan* p) {
  for (cudaEvent_t e : p->ev_start) cudaEventDestroy(e);
  for (cudaEvent_t e : p->ev_end) cudaEventDestroy(e);
  p->ev_start.clear();
  p->ev_end.clear();
  if (p->f16) cudaFree(p->f16);
  if (p->status) cudaFree(p->status);
  if (p->trace) cudaFree(p->trace);
  if (p->stage_x) cudaFree(p->stage_x);
  if (p->stage_f) cudaFree(p->stage_f);
  if (p->stage_y) cudaFree(p->stage_y);
  if (p->split_count) cudaFree(p->split_count);
  if (p->gbar) cudaFree(p->gbar);
  if (p->split_part) cudaFree(p->split_part);
  if (p->stage_x2) cudaFree(p->stage_x2);
  if (p->stage_f2) cudaFree(p->stage_f2);
  if (p->stage_y2) cudaFree(p->stage_y2);
  for (cudaEvent_t e : {p->ev_begin, p->ev_in[0], p->ev_in[1], p->ev_run[0], p->ev_run[1], p->ev_out[0], p->ev_out[1]})
    if (e) cudaEventDestroy(e);
  if (p->s_in) cudaStreamDestroy(p->s_in);
  if (p->s_out) cudaStreamDestroy(p->s_out);
}

ConvParams make_params(const i8c_plan* pl, const int8_t* x, float alpha) {
  const i8c_conv_shape& s = pl->shape;
  ConvParams p{};
  p.x = x;
  p.status = pl->status;
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
  p.P = pl->P;
  p.Q = pl->Q;
  p.PQ = pl->P * pl->Q;
  p.M = static_cast<int>(pl->M);
  p.CB = s.C / 32;
  p.KB = s.K / 32;
  p.num_slices = pl->num_slices;
  p.chunk_slices = pl->chunk_slices;
  p.num_chunks = pl->num_chunks;
  p.num_n_tiles = pl->num_n_tiles;
  p.num_tiles = pl->num_tiles;
  p.acc_buffers = pl->acc_buffers;
  p.tmem_cols = pl->tmem_cols;
  p.img_stride = static_cast<int64_t>(s.C) * s.H * s.W;
  p.timeout_ns = pl->timeout_ns;
  p.debug_flags = pl->debug_flags;
  p.trace = pl->trace;
  return p;
}

// The filter operand transform of a plan: the stacked order for the
// stacked-tap kernel, else the fp16 copy in the CxRSKx<32> order; nothing
// for the kernels that convert the filter themselves.
cudaError_t convert_filter(const i8c_plan* pl, const int8_t* f, cudaStream_t stream) {
  const i8c_conv_shape& s = pl->shape;
  if (pl->kernel_variant == 6) return i8c::launch_filter_to_f16_stacked(f, pl->f16, s.C / 32, s.R, s.S, stream);
  return i8c::launch_filter_to_f16(f, pl->f16, static_cast<int64_t>(s.K) * s.C * s.R * s.S, stream);
}

bool converts_in_kernel(const i8c_plan* pl) {
  return pl->gbar != nullptr || (pl->kernel_variant >= 2 && pl->kernel_variant <= 3 && pl->halo.f_smem);
}

// prepacked: the filter was converted by i8c_plan_set_filter; f is unused
// (the kernels that write their resident filter themselves read the plan's
// int8 copy instead)
i8c_status run_plan(const i8c_plan* pl, const int8_t* x, const int8_t* f, int8_t* y, int32_t* acc, float alpha,
                    cudaStream_t stream, const i8c_epilogue* ep = nullptr, bool prepacked = false) {
  const i8c_conv_shape& s = pl->shape;
  cudaError_t e = cudaSuccess;
  if (prepacked) {
    f = reinterpret_cast<const int8_t*>(pl->f16);
  } else {
    pl->prepacked = false;  // a run with its own filter replaces the prepacked copy
  }
  if (prepacked) {
  } else if (pl->kernel_variant == 6 || !converts_in_kernel(pl)) {
    e = convert_filter(pl, f, stream);
    if (e != cudaSuccess) return from_cuda(e);
  }
  ConvParams p = make_params(pl, x, alpha);
  p.y = y;
  p.acc = acc;
  p.out_mode = acc != nullptr ? 1 : 0;
  if (ep != nullptr) {
    p.alpha_k = ep->alpha;
    p.bias_k = ep->bias;
    p.relu = ep->relu != 0 ? 1 : 0;
  }
  const size_t nev = pl->ev_start.size();
  if (nev > 0) {
    e = cudaEventRecord(pl->ev_start[pl->ev_recorded % nev], stream);
    if (e != cudaSuccess) return from_cuda(e);
  }
  if (pl->kernel_variant >= 2) {
    i8c::HaloParams hp = pl->halo;
    hp.c = p;
    if (hp.tma_halo && pl->tmap_x_ptr != x) {
      // the activations as {32 channel bytes, W, H, N*C/32}; one box is one
      // channel block of a tile's halo (zeros outside the image)
      EncodeTiled encode = get_encode_tiled();
      if (encode == nullptr) return I8C_ERR_CUDA;
      cuuint64_t dims[4] = {32, static_cast<cuuint64_t>(s.W), static_cast<cuuint64_t>(s.H),
                            static_cast<cuuint64_t>(s.N) * (s.C / 32)};
      cuuint64_t strides[3] = {32, static_cast<cuuint64_t>(s.W) * 32, static_cast<cuuint64_t>(s.W) * s.H * 32};
      cuuint32_t box[4] = {32, static_cast<cuuint32_t>(hp.box_w), static_cast<cuuint32_t>(hp.box_h), 1};
      cuuint32_t estr[4] = {1, 1, 1, 1};
      if (encode(&pl->tmap_x, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<int8_t*>(x), dims, strides, box, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return I8C_ERR_CUDA;
      pl->tmap_x_ptr = x;
    }
    hp.f_src = f;  // read only when the kernel writes its resident filter itself
    hp.filter_ready = prepacked && !pl->filter_fresh ? 1 : 0;
    if (prepacked) pl->filter_fresh = false;
    if (pl->gbar != nullptr && !prepacked) {  // prepacked: the TMA reads the converted copy
      hp.f_int8 = f;
      hp.f16 = pl->f16;
      hp.f_vecs = static_cast<int64_t>(s.K) * s.C * s.R * s.S / 16;
      hp.gbar = pl->gbar;
    }
    const CUtensorMap& tx = pl->tmap_x;  // read only by TMA-fed halos
    e = pl->kernel_variant == 6   ? i8c::stack_launch(pl->tmap, tx, hp, pl->smem_bytes, pl->num_ctas, stream)
        : pl->kernel_variant == 5 ? i8c::tr_launch_pair(pl->tmap, tx, hp, pl->smem_bytes, pl->num_ctas, stream)
        : pl->kernel_variant == 4 ? i8c::tr_launch(pl->tmap, tx, hp, pl->smem_bytes, pl->num_ctas, stream)
        : pl->kernel_variant == 3 ? i8c::halo_launch_pair(pl->block_n, pl->tmap, tx, hp, pl->smem_bytes,
                                                          pl->num_ctas, stream)
                                  : i8c::halo_launch_single(pl->block_n, pl->tmap, tx, hp, pl->smem_bytes,
                                                            pl->num_ctas, stream);
  } else {
    e = i8c::launch_conv(pl->block_n, pl->tmap, p, pl->num_ctas, stream);
  }
  if (e != cudaSuccess) return from_cuda(e);
  if (nev > 0) {
    e = cudaEventRecord(pl->ev_end[pl->ev_recorded % nev], stream);
    ++pl->ev_recorded;
  }
  return from_cuda(e);
}

// Plans behind the one-shot entry points, one per (device, stream, shape),
// at most kMaxCachedPlans of them: the least recently used plan is destroyed
// when a new one would exceed the bound (a caller that creates streams call
// after call cannot grow the cache without limit).
constexpr size_t kMaxCachedPlans = 64;
using CacheKey = std::array<int64_t, 15>;
struct CacheEntry {
  i8c_plan* plan;
  uint64_t last_use;
};
std::mutex g_cache_mu;
std::map<CacheKey, CacheEntry> g_cache;
uint64_t g_cache_clock = 0;
// Test hooks for the one-shot and no-allocation entry points
// (i8c_debug_set_oneshot): debug flags and the bounded-wait limit.
int32_t g_oneshot_debug_flags = 0;
int32_t g_oneshot_timeout_us = 0;

i8c_status cached_plan(const i8c_conv_shape* s, cudaStream_t stream, i8c_plan** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return from_cuda(e);
  CacheKey key{dev, static_cast<int64_t>(reinterpret_cast<uintptr_t>(stream)),
               s->N, s->C, s->H, s->W, s->K, s->R, s->S, s->pad_h, s->pad_w,
               s->stride_h, s->stride_w, s->dil_h * 65536LL + s->dil_w, 0};
  std::lock_guard<std::mutex> lock(g_cache_mu);
  auto it = g_cache.find(key);
  if (it != g_cache.end()) {
    it->second.last_use = ++g_cache_clock;
    *out = it->second.plan;
    return I8C_OK;
  }
  i8c_options o{};
  o.debug_flags = g_oneshot_debug_flags;
  o.wait_timeout_us = g_oneshot_timeout_us;
  i8c_plan* p = nullptr;
  i8c_status st = i8c_plan_create(s, &o, &p);
  if (st != I8C_OK) return st;
  if (g_cache.size() >= kMaxCachedPlans) {
    auto lru = g_cache.begin();
    for (auto jt = g_cache.begin(); jt != g_cache.end(); ++jt)
      if (jt->second.last_use < lru->second.last_use) lru = jt;
    i8c_plan_destroy(lru->second.plan);  // synchronises the device first
    g_cache.erase(lru);
  }
  g_cache[key] = CacheEntry{p, ++g_cache_clock};
  *out = p;
  return I8C_OK;
}

bool options_valid(const i8c_options& o) {
  if (o.block_n != 0 && o.block_n != 32 && o.block_n != 64 && o.block_n != 128 && o.block_n != 256) return false;
  return !(o.num_ctas < 0 || o.max_chunk_slices < 0 || o.max_chunk_slices > 32 || o.wait_timeout_us < 0 ||
           o.timing_events < 0 || o.timing_events > 65536 || o.host_staging < 0 || o.host_staging > 2 ||
           o.kernel_variant < 0 || o.kernel_variant > 6 || o.halo_loads < 0 || o.halo_loads > 3 ||
           o.tail_split < 0 || o.tail_split > 3 || o.tile_shape < 0 || o.tile_shape > 3 || o.fused_filter < 0 ||
           o.fused_filter > 3 || o.filter_run < 0 || o.filter_run > 32 ||
           (o.tile_px != 0 && (o.tile_px < 16 || o.tile_px > 256 || o.tile_px % 16 != 0)));
}

// The planner: kernel form, tile shape, persistent schedule, exact-fp32
// chunking and shared-memory layout of shape `s` (P, Q already checked) on
// `ctas` SMs, into `p`.  host_only: no device call at all -- CTA pairs are
// assumed to fit one per two SMs -- so that the layout can be inspected
// without a GPU (i8c_plan_layout).  *split_bytes_out: the int32 partial-sum
// workspace the schedule needs.
i8c_status plan_geometry(const i8c_conv_shape& s, const i8c_options& o, int64_t P, int64_t Q, int ctas,
                         bool host_only, i8c_plan* p, int64_t* split_bytes_out) {
  p->shape = s;
  p->P = static_cast<int>(P);
  p->Q = static_cast<int>(Q);
  p->M = static_cast<int64_t>(s.N) * P * Q;
  if (o.kernel_variant == 6 ||
      (kStackAuto && o.kernel_variant == 0 && o.block_n == 0 && o.halo_loads == 0 && o.tile_shape == 0 &&
       o.tail_split == 0 && (o.fused_filter == 0 || o.fused_filter == 3) && o.tile_px == 0 && o.filter_run == 0)) {
    // The stacked-tap kernel: two taps per N = 128 MMA on CTA pairs.
    int smem = 0;
    if (!stack_layout(s, p->P, p->Q, &p->halo, &smem) || (o.kernel_variant == 0 && !p->halo.resident)) {
      if (o.kernel_variant == 6) return I8C_ERR_UNSUPPORTED;
      p->halo = i8c::HaloParams{};
    } else {
      p->kernel_variant = 6;
      p->cta_group = 2;
      p->block_n = 64;
      p->num_n_tiles = 1;
      const int64_t units = (static_cast<int64_t>(p->halo.num_patches) + 1) / 2;
      p->num_m_tiles = static_cast<int>(units);
      p->num_tiles = static_cast<int>(units);
      p->halo.ksplit = 1;
      p->halo.nsplit = 1;
      p->halo.full_units = p->num_tiles;
      p->halo.num_units = p->num_tiles;
      p->split_tiles = 0;
      int g = ctas / 2;
      if (!host_only) {
        if (i8c::stack_prepare() != cudaSuccess) return I8C_ERR_CUDA;
        const int fit = i8c::stack_max_clusters(p->halo.slots, smem);
        if (fit < 1) return I8C_ERR_UNSUPPORTED;
        if (g > fit) g = fit;
      }
      if (g < 1) g = 1;
      p->num_ctas = 2 * (g < p->num_tiles ? g : p->num_tiles);
      // chunks of whole filter rows: a column gathers at most U taps x 32
      // channels per row, so 32 / U rows stay within 1024 products
      const int U = p->halo.slots;
      int rows = 32 / U;
      if (o.max_chunk_slices > 0) rows = o.max_chunk_slices / U < rows ? o.max_chunk_slices / U : rows;
      if (rows < 1) rows = 1;
      p->num_slices = (s.C / 32) * s.R * s.S;
      p->chunk_slices = rows;  // filter rows per chunk for this kernel
      p->num_chunks = ((s.C / 32) * s.R + rows - 1) / rows;
      p->acc_buffers = 2;
      p->tmem_cols = 256;
      p->smem_bytes = smem;
      return o.fused_filter == 2 ? I8C_ERR_UNSUPPORTED : I8C_OK;  // its filter order has its own conversion
    }
  }
  // Kernel and tile width.  The halo kernel (16x8 output patches) is preferred
  // whenever its halo fits in shared memory; its tile width is the one with
  // the best wave efficiency (ties go to the wider tile).  Variant 3 runs it
  // on CTA pairs (clusters of two): one M = 256 MMA per K-step for two
  // patches, each CTA staging half of the filter tile.
  int bn = 0, halo_smem = 0, groups = 0;
  p->kernel_variant = 1;
  p->cta_group = 1;
  // Transposed tiles on cg CTAs per MMA tile: the MMA width (pixels per
  // tile, cg halves of tile_px each) whose tile count fills the waves best.
  // Model (measured on the 3x3 layers): a K-slice of a tile costs its width
  // in tensor-core cycles plus a fixed issue, wait and halo overhead, and a
  // launch takes as many tile times as its fullest SM (pair) runs tiles.
  // Returns the width (0: nothing fits), its cost in cycles per K-slice of
  // the launch and the concurrent CTA groups.
  const int tr_stg = o.halo_loads == 1 ? 3 : 0;  // staging ring on request
  auto pick_tr = [&](int cg, double* cost_out, int* groups_out) -> int {
    const int n_tiles = (s.K + 128 * cg - 1) / (128 * cg);
    // a pair's MMA queue hides more of the per-stage waits, but both CTAs'
    // producers gate every channel block (measured: 2 x 144 K-slices of 240
    // pixels on the 64x512x28x28 layer at ~310 cycles each)
    const double overhead = cg == 2 ? 80.0 : 130.0;
    double best = 0.0;
    int best_n = 0;
    for (int n = 256; n >= 16; n -= 16) {
      if (o.tile_px != 0 && n != o.tile_px) continue;
      i8c::HaloParams h;
      int sm = 0;
      if (!tr_layout(s, p->P, n / cg, cg, o.filter_run, tr_stg, &h, &sm, o.halo_loads == 3)) continue;
      // A pair's CTA builds the halo of n / 2 pixels plus the filter's overhang
      // for every channel block; when the overhang outweighs the pixels the
      // producers, not the tensor core, set the pace (8x256x56x56 layer: 88
      // pixels + 118 positions, 34.5 us on pairs against 31.3 us on single CTAs).
      if (cg == 2 && o.kernel_variant != 5 && h.positions > 1.6 * (n / 2)) continue;
      int g = ctas / cg;
      if (cg == 2) {
        if (!host_only && i8c::tr_prepare_pair() != cudaSuccess) continue;
        const int fit = host_only ? g : i8c::tr_pair_max_clusters(h.bgroup, s.S, n, sm);
        if (fit < 1) continue;
        if (g > fit) g = fit;
      }
      const int64_t t = (static_cast<int64_t>(h.num_patches) + cg - 1) / cg * n_tiles;
      const int64_t waves = (t + g - 1) / g;
      const double cost = static_cast<double>(waves) * (n + overhead);
      if (best_n == 0 || cost < best * 0.999) {
        best = cost;
        best_n = n;
        *groups_out = g;
      }
    }
    *cost_out = best;
    return best_n;
  };
  if (o.kernel_variant == 4 || o.kernel_variant == 5) {
    const int cg = o.kernel_variant == 5 ? 2 : 1;
    double cost = 0.0;
    const int n = pick_tr(cg, &cost, &groups);
    if (n == 0) {
      return I8C_ERR_UNSUPPORTED;
    }
    tr_layout(s, p->P, n / cg, cg, o.filter_run, tr_stg, &p->halo, &halo_smem, o.halo_loads == 3);
    p->kernel_variant = o.kernel_variant;
    p->cta_group = cg;
    bn = 128 * cg;
  } else if (o.kernel_variant != 1) {
    // best tile width on cg CTAs per tile: {width, groups} (width 0: none fits)
    // best {width, groups, flat} on cg CTAs per tile (width 0: none fits);
    // tile shapes: 16x8 patches, and flat tiles for stride 1 unless forced
    struct Choice {
      int bn, groups;
      bool flat, wide;
    };
    auto search = [&](int cg, int only_bn) -> Choice {
      Choice bestc{0, 0, false, false};
      double best = -1.0;
      for (int geo = 0; geo < 3; ++geo)
      for (int cand : {256, 128, 64, 32}) {
        const bool flat = geo == 1, wide = geo == 2;
        // tile_shape 3: 16x16 patches only; auto considers them too (below)
        if (o.tile_shape == 3 && !wide) continue;
        if (wide && o.tile_shape != 3 && o.tile_shape != 0) continue;
        if ((flat && o.tile_shape == 1) || (!flat && o.tile_shape == 2)) continue;
        if (o.block_n != 0 && cand != o.block_n) continue;
        if (only_bn != 0 && cand != only_bn) continue;
        if (cg == 2 && cand < 64) continue;
        if (o.block_n == 0 && cand > 32 * cg && cand / 2 >= s.K) continue;  // half the tile would be empty
        i8c::HaloParams h;
        int sm = 0;
        if (!halo_layout(s, p->P, p->Q, cand, cg, o.halo_loads, flat, &h, &sm, wide)) continue;
        // 16x16 patches issue through the whole-row run path only; auto takes
        // them only where the filter stays resident beside their larger halo
        // (one output-channel tile, every filter stage in the ring)
        if (wide && !((h.bgroup == 3 || h.bgroup == 9) && h.bgroup % s.S == 0)) continue;
        if (wide && o.tile_shape == 0 &&
            !((s.K + cand - 1) / cand == 1 && (s.C / 32) * s.R * s.S / h.bgroup <= h.nbs))
          continue;
        // 128-wide 16x16 patches only when asked for: their larger halos pace
        // the producers (stride-2 112x112 layer: 115 against 63 us; 8x256x56x56
        // layer: 36 against 26 us)
        if (wide && o.tile_shape == 0 && cand > 64) continue;
        int g = ctas / cg;
        if (cg == 2) {
          // pairs that fit on the GPU at once (clusters need both SMs free)
          if (!host_only && i8c::halo_prepare_pair(cand) != cudaSuccess) continue;
          const int fit = host_only ? g : i8c::halo_pair_max_clusters(cand, h.bgroup, s.S, sm);
          if (fit < 1) continue;
          if (g > fit) g = fit;
          if (g < 1) g = 1;
        }
        const int nt = (s.K + cand - 1) / cand;
        const int64_t t = (static_cast<int64_t>(h.num_patches) + cg - 1) / cg * nt;
        // narrower MMAs leave the issuing warp's per-slice overhead exposed (the
        // tensor core queues only about two MMAs); measured relative rates
        double width_eff = cand == 256 ? 1.0 : cand == 128 ? 0.62 : cand == 64 ? 0.45 : 0.3;
        // runs of one K-slice (no room for longer filter stages) issue poorly
        if (h.bgroup == 1 && s.S > 1) width_eff *= 0.6;
        // 16x16 patches: twice the MMAs per tile boundary and per run, and a
        // third fewer halo loads per pixel (measured on the dilated 5x9 layer
        // on CTA pairs: 259.8 against 291 us)
        if (wide) width_eff *= 1.12;
        // share of a tile's 128 rows that are real output pixels
        const double m_util =
            static_cast<double>(p->P) * p->Q /
            (flat ? 128.0 * h.tpi : 128.0 * h.subtiles * h.TPH * h.TQW);
        const double score = wave_efficiency(t, g) * m_util * width_eff * static_cast<double>(s.K) /
                             (static_cast<double>(nt) * cand);
        if (score > best * 1.02) {
          best = score;
          bestc = {cand, g, flat, wide};
        }
      }
      return bestc;
    };
    int cg = o.kernel_variant == 3 ? 2 : 1;
    Choice best = search(cg, 0);
    if (o.kernel_variant == 0 && best.bn == 64) {
      // 64-wide tiles issue MMAs at the tensor core's per-instruction floor; a
      // CTA pair's M = 256 MMAs halve the instructions per SM (measured on the
      // dilated 5x9 layer: 1042 against 889 TOPS).  At 256 columns single
      // CTAs are faster.
      const Choice pair = search(2, 64);
      if (pair.bn != 0) {
        cg = 2;
        best = pair;
      }
    }
    // Auto: transposed tiles instead of 256-wide single-CTA halo tiles when
    // the model says they fill the waves enough better (a K-slice of a
    // 128-pixel x 256-channel halo tile costs about 345 cycles).  E.g. the
    // 8x256x56x56 layer: 224 halo tiles on 152 SMs take two tile times
    // (2 x 345); 304 transposed tiles of 176 pixels fill two waves exactly
    // (2 x 306).
    bool use_tr = false;
    if (o.kernel_variant == 0 && o.block_n == 0 && o.halo_loads == 0 && o.tile_shape == 0 && o.tail_split == 0 &&
        (o.fused_filter == 0 || o.fused_filter == 3) && best.bn == 256 && cg == 1) {
      i8c::HaloParams h;
      int sm = 0;
      if (halo_layout(s, p->P, p->Q, 256, 1, 0, best.flat, &h, &sm)) {
        const int64_t t = static_cast<int64_t>(h.num_patches) * ((s.K + 255) / 256);
        const double halo_cost = static_cast<double>((t + ctas - 1) / ctas) * 345.0;
        double tr_cost = 0.0, pair_cost = 0.0;
        int tr_groups = 0, pair_groups = 0;
        int n1 = pick_tr(1, &tr_cost, &tr_groups);
        int n2 = pick_tr(2, &pair_cost, &pair_groups);
        const bool pair = n2 != 0 && (n1 == 0 || pair_cost < tr_cost);
        const double cost = pair ? pair_cost : tr_cost;
        // Halo tiles on CTA pairs (256 pixels x 256 channels per pair): a
        // K-slice costs about 256 + 53 cycles, fitted to the 64x512x28x28
        // layer (143 us against 148 us for transposed pairs), provided the
        // halo stays close to its 128 pixels per CTA -- on strided layers the
        // producers set the pace (stride-2 112x112 layer: 82 us on pairs
        // against 69 us on single CTAs).  Taken when at least 2% cheaper than
        // both other choices.
        if (s.stride_h == 1 && s.stride_w == 1) {
          const Choice hc = search(2, 256);
          i8c::HaloParams h2;
          int sm2 = 0;
          if (hc.bn == 256 && halo_layout(s, p->P, p->Q, 256, 2, 0, hc.flat, &h2, &sm2) &&
              h2.positions <= 1.6 * 128) {
            const int64_t t2 = (static_cast<int64_t>(h2.num_patches) + 1) / 2 * ((s.K + 255) / 256);
            const double hp_cost = static_cast<double>((t2 + hc.groups - 1) / hc.groups) * (256.0 + 53.0);
            const double other = (n1 != 0 || n2 != 0) && cost < halo_cost ? cost : halo_cost;
            if (hp_cost < 0.98 * other) {
              cg = 2;
              best = hc;
              n1 = n2 = 0;  // keep the halo kernel
            }
          }
        }
        if ((n1 != 0 || n2 != 0) && cost < 0.97 * halo_cost) {
          const int cgt = pair ? 2 : 1;
          const int n = pair ? n2 : n1;
          tr_layout(s, p->P, n / cgt, cgt, o.filter_run, tr_stg, &p->halo, &halo_smem, o.halo_loads == 3);
          p->kernel_variant = pair ? 5 : 4;
          p->cta_group = cgt;
          groups = pair ? pair_groups : tr_groups;
          bn = 128 * cgt;
          use_tr = true;
        }
      }
    }
    if (use_tr) {
      // chosen above
    } else if (best.bn != 0) {
      bn = best.bn;
      groups = best.groups;
      p->kernel_variant = cg == 2 ? 3 : 2;
      p->cta_group = cg;
      halo_layout(s, p->P, p->Q, bn, cg, o.halo_loads, best.flat, &p->halo, &halo_smem, best.wide);
    } else if (o.kernel_variant >= 2) {
      return I8C_ERR_UNSUPPORTED;
    }
  }
  if (bn == 0) {
    bn = o.block_n;
    if (bn == 0) bn = s.K <= 32 ? 32 : (s.K <= 64 ? 64 : (s.K <= 128 ? 128 : 256));
  }
  p->block_n = bn;
  p->num_n_tiles = (s.K + bn - 1) / bn;
  const int64_t m_tiles = p->kernel_variant >= 2
                              ? (static_cast<int64_t>(p->halo.num_patches) + p->cta_group - 1) / p->cta_group
                              : (p->M + 127) / 128;
  const int64_t tiles = m_tiles * p->num_n_tiles;
  if (tiles > kMaxI32) {
    return I8C_ERR_OVERFLOW_RISK;
  }
  p->num_m_tiles = static_cast<int>(m_tiles);
  p->num_tiles = static_cast<int>(tiles);
  int64_t& split_bytes = *split_bytes_out;
  split_bytes = 0;
  if (p->kernel_variant >= 4) {
    // one unit per tile, no split tail
    p->halo.ksplit = 1;
    p->halo.nsplit = 1;
    p->halo.full_units = p->num_tiles;
    p->halo.num_units = p->num_tiles;
    p->split_tiles = 0;
    const int g = p->kernel_variant == 5 ? groups : ctas;
    p->num_ctas = p->cta_group * (g < p->num_tiles ? g : p->num_tiles);
  } else if (p->kernel_variant >= 2) {
    // The last wave is partial when the tile count is not a multiple of the
    // persistent CTAs (pairs): its tiles are split along the channel blocks
    // into ksplit units each, so that the wave's units fill the GPU and take
    // 1/ksplit of a tile's time.
    const int g = p->cta_group == 2 ? groups : ctas;
    const int rem = p->num_tiles % g;
    int ksplit = 1, nsplit = 1;
    // Halving the last wave's tiles along the output channels needs no
    // partial sums (disjoint outputs), but a K-slice costs the MMA warp about
    // as long at N = BN/2 as at BN (barrier waits and issue work dominate), so
    // a half unit takes nearly a whole tile's time: measured no faster on the
    // 8x256x56x56 layer, hence only on request.
    if (rem > 0 && p->cta_group == 1 && bn >= 128 && 2 * rem <= g && o.tail_split == 3) nsplit = 2;
    if (nsplit == 1 && rem > 0 && o.tail_split != 1 && o.tail_split != 3 && p->halo.subtiles != 2) {
      ksplit = g / rem;
      if (ksplit > s.C / 32) ksplit = s.C / 32;
      if (ksplit < 2) ksplit = 1;
    }
    if (ksplit > 1 && o.tail_split == 0) {
      // Auto: split only when the time saved in the last wave clearly exceeds
      // the cost of the partial sums, which all split units write (and half
      // read back) at nearly the same moment.  Estimates: a K-slice takes
      // about BN + 100 cycles at ~1.9 GHz; the partials move at ~8 TB/s
      // through L2, plus ~2 us for the burst to drain.
      const double tile_us = static_cast<double>((s.C / 32) * s.R * s.S) * (bn + 100) / 1900.0;
      const double saved_us = tile_us * (1.0 - 1.0 / ksplit);
      const double bytes = static_cast<double>(rem) * ksplit * p->cta_group * 128.0 * bn * 4.0 * 1.5;
      const double cost_us = bytes / 8.0e6 + 2.0;
      if (saved_us < 1.5 * cost_us) ksplit = 1;
    }
    p->halo.ksplit = ksplit;
    p->halo.nsplit = nsplit;
    // Resident filter: with one output-channel tile and whole-tile units,
    // every unit streams the same filter stages in the same order; when all
    // of them fit in the stage ring, they are loaded once and kept, and the
    // MMA warp stops waiting for and releasing filter stages after the first
    // unit (e.g. the 64-channel 5x9 layer: five 9-slice stages per tile).
    const int unit_stages = (s.C / 32) * s.R * s.S / p->halo.bgroup;
    if (p->num_n_tiles == 1 && ksplit == 1 && nsplit == 1 && unit_stages <= p->halo.nbs) {
      p->halo.nbs = unit_stages;
      p->halo.resident = 1;
      // the stages beyond the filter's own are not needed: the barriers move down
      p->halo.off_bar = p->halo.off_b + static_cast<uint32_t>(unit_stages * p->halo.bgroup * (bn / p->cta_group) * 64);
      halo_smem = static_cast<int>(p->halo.off_bar) + i8c::kHaloBarBytes + 1024;
    }
    // fused_filter = 2, and auto: a resident filter is converted by the
    // kernel itself into its stages (no fp16 copy, no conversion launch).
    // Measured on the 64-channel 5x9 layer: 318.3-319.0 us per run against
    // 318.9-319.3 with the conversion kernel; on the 32-channel 16x16 layer
    // 6.5 against 8.4 us.
    if (o.fused_filter == 2 || (o.fused_filter == 0 && p->halo.resident)) {
      if (!p->halo.resident) return I8C_ERR_UNSUPPORTED;
      p->halo.f_smem = 1;
    }
    p->halo.full_units = ksplit > 1 || nsplit > 1 ? p->num_tiles - rem : p->num_tiles;
    p->halo.num_units = p->halo.full_units + (ksplit > 1 ? rem * ksplit : 0) + (nsplit > 1 ? rem * 2 : 0);
    if (ksplit > 1)
      split_bytes = static_cast<int64_t>(rem) * ksplit * p->cta_group * 128 * bn * static_cast<int64_t>(sizeof(int32_t));
    p->split_tiles = ksplit > 1 ? rem : 0;
    p->num_ctas = p->cta_group * (g < p->halo.num_units ? g : p->halo.num_units);
  } else {
    p->num_ctas = ctas < p->num_tiles ? ctas : p->num_tiles;
  }
  p->num_slices = (s.C / 32) * s.R * s.S;
  int max_chunk = o.max_chunk_slices > 0 ? o.max_chunk_slices : 32;
  if (p->kernel_variant >= 2) {
    // the halo kernel switches accumulators only between filter stages
    const int G = p->halo.bgroup;
    max_chunk = max_chunk / G * G;
    if (max_chunk < G) max_chunk = G;
  }
  p->num_chunks = (p->num_slices + max_chunk - 1) / max_chunk;
  p->chunk_slices = (p->num_slices + p->num_chunks - 1) / p->num_chunks;
  if (p->kernel_variant >= 2) {
    p->chunk_slices = (p->chunk_slices + p->halo.bgroup - 1) / p->halo.bgroup * p->halo.bgroup;
    p->num_chunks = (p->num_slices + p->chunk_slices - 1) / p->chunk_slices;
  }
  if (p->kernel_variant >= 2) {
    // halo kernel: two fp32 chunk accumulators; running sums live in registers
    p->acc_buffers = 2;
    p->tmem_cols = static_cast<uint32_t>(
        next_pow2(2 * (p->kernel_variant >= 4 ? p->cta_group * p->halo.tile_px
                                              : bn * (p->halo.subtiles == 2 ? 2 : 1))));
  } else {
    const int run_cols = p->num_chunks > 1 ? bn : 0;
    p->acc_buffers = (2 * bn + run_cols <= 512) ? 2 : 1;
    p->tmem_cols = static_cast<uint32_t>(next_pow2(p->acc_buffers * bn + run_cols));
  }
  p->smem_bytes = p->kernel_variant >= 2 ? halo_smem : i8c::conv_smem_bytes(bn);
  // the in-kernel resident filter exists for the halo kernels (single and pairs) only
  if (o.fused_filter == 2 && !((p->kernel_variant == 2 || p->kernel_variant == 3) && p->halo.f_smem))
    return I8C_ERR_UNSUPPORTED;
  return I8C_OK;
}

}  // namespace

extern "C" {

const char* i8c_status_string(i8c_status status) {
  switch (status) {
    case I8C_OK: return "ok";
    case I8C_ERR_INVALID_ARG: return "invalid argument";
    case I8C_ERR_UNSUPPORTED: return "unsupported shape";
    case I8C_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case I8C_ERR_OVERFLOW_RISK: return "int32 accumulator or index overflow possible";
    case I8C_ERR_CUDA: return "CUDA error";
    case I8C_ERR_TIMEOUT: return "device-side wait timed out";
    case I8C_ERR_NO_DEVICE: return "no usable sm_103 CUDA device";
  }
  return "unknown status";
}

int64_t i8c_launch_count(void) { return i8c::g_launches.load(std::memory_order_relaxed); }

i8c_status i8c_output_size(const i8c_conv_shape* shape, int32_t* P, int32_t* Q) {
  if (P == nullptr || Q == nullptr) return I8C_ERR_INVALID_ARG;
  int64_t p = 0, q = 0;
  i8c_status st = check_shape(shape, &p, &q);
  if (st != I8C_OK) return st;
  if (p > kMaxI32 || q > kMaxI32) return I8C_ERR_OVERFLOW_RISK;
  *P = static_cast<int32_t>(p);
  *Q = static_cast<int32_t>(q);
  return I8C_OK;
}

i8c_status i8c_supported(const i8c_conv_shape* shape) {
  int64_t p = 0, q = 0;
  return check_supported(shape, &p, &q);
}

i8c_status i8c_plan_create(const i8c_conv_shape* shape, const i8c_options* opts, i8c_plan** out) {
  if (out == nullptr) return I8C_ERR_INVALID_ARG;
  *out = nullptr;
  int64_t P = 0, Q = 0;
  i8c_status st = check_supported(shape, &P, &Q);
  if (st != I8C_OK) return st;
  i8c_options o{};
  if (opts) o = *opts;
  if (!options_valid(o)) return I8C_ERR_INVALID_ARG;

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return from_cuda(e);
  cudaDeviceProp prop;
  e = cudaGetDeviceProperties(&prop, dev);
  if (e != cudaSuccess) return from_cuda(e);
  if (prop.major != 10 || prop.minor != 3) return I8C_ERR_NO_DEVICE;
  EncodeTiled encode = get_encode_tiled();
  if (encode == nullptr) return I8C_ERR_CUDA;

  i8c_plan* p = new (std::nothrow) i8c_plan();
  if (p == nullptr) return I8C_ERR_CUDA;
  const i8c_conv_shape& s = *shape;
  p->device = dev;
  const int ctas = o.num_ctas > 0 ? o.num_ctas : prop.multiProcessorCount;
  int64_t split_bytes = 0;
  st = plan_geometry(s, o, P, Q, ctas, false, p, &split_bytes);
  if (st != I8C_OK) {
    delete p;
    return st;
  }
  const int bn = p->block_n;
  const int halo_smem = p->smem_bytes;
  p->timeout_ns = static_cast<uint64_t>(o.wait_timeout_us > 0 ? o.wait_timeout_us : 2000000) * 1000ull;
  p->debug_flags = o.debug_flags;
  p->x_bytes = static_cast<size_t>(s.N) * s.C * s.H * s.W;
  p->f_bytes = static_cast<size_t>(s.K) * s.C * s.R * s.S;
  p->y_bytes = static_cast<size_t>(s.N) * s.K * P * Q;

  e = p->kernel_variant == 6   ? i8c::stack_prepare()
      : p->kernel_variant == 5 ? i8c::tr_prepare_pair()
      : p->kernel_variant == 4 ? i8c::tr_prepare()
      : p->kernel_variant == 3 ? i8c::halo_prepare_pair(bn)
      : p->kernel_variant == 2 ? i8c::halo_prepare_single(bn)
                               : i8c::conv_prepare(bn);
  // the fp16 filter copy: the int8 filter's order, or the stacked-tap
  // kernel's [C/32][R][2][ceil(S/2)][64][32] (one slot more per row and rank
  // pair when S is odd)
  p->f16_bytes = p->kernel_variant == 6
                     ? static_cast<size_t>(s.C / 32) * s.R * 2 * ((s.S + 1) / 2) * 64 * 32 * 2
                     : p->f_bytes * 2;
  if (e == cudaSuccess) e = cudaMalloc(&p->f16, p->f16_bytes);
  if (e == cudaSuccess) e = cudaMalloc(&p->status, sizeof(int));
  if (e == cudaSuccess) e = cudaMemset(p->status, 0, sizeof(int));
  if (e == cudaSuccess && p->kernel_variant == 2 && o.fused_filter == 1) {
    // Single-CTA halo kernel, on request: the filter conversion moves into the
    // kernel (one launch per run) when all of its CTAs fit on the GPU at once.
    // Measured slower than the separate conversion kernel, whose tail the
    // convolution's prologue overlaps (e.g. 37.0 against 35.0 us per run on
    // the 8x256x56x56 layer): the grid barrier delays the first filter load.
    const int fit = i8c::halo_single_max_ctas(bn, p->halo.bgroup, s.S, halo_smem);
    if (fit >= p->num_ctas) {
      e = cudaMalloc(&p->gbar, 2 * sizeof(uint32_t));
      if (e == cudaSuccess) e = cudaMemset(p->gbar, 0, 2 * sizeof(uint32_t));
    }
  }
  p->workspace_bytes = static_cast<int64_t>(p->f16_bytes + sizeof(int));
  if (e == cudaSuccess && split_bytes > 0) {
    const size_t counts = sizeof(int) * static_cast<size_t>(p->split_tiles) * p->cta_group;
    e = cudaMalloc(&p->split_part, static_cast<size_t>(split_bytes));
    if (e == cudaSuccess) e = cudaMalloc(&p->split_count, counts);
    if (e == cudaSuccess) e = cudaMemset(p->split_count, 0, counts);
    p->workspace_bytes += split_bytes + static_cast<int64_t>(counts);
    p->halo.split_part = p->split_part;
    p->halo.split_count = p->split_count;
  }
  if (e == cudaSuccess && (o.debug_flags & I8C_DEBUG_TRACE)) {
    const size_t tb = sizeof(long long) * i8c::kTraceRows * i8c::kTraceSlots;
    e = cudaMalloc(&p->trace, tb);
    if (e == cudaSuccess) e = cudaMemset(p->trace, 0, tb);
  }
  if (e == cudaSuccess && o.host_staging) {
    e = cudaMalloc(&p->stage_x, p->x_bytes);
    if (e == cudaSuccess) e = cudaMalloc(&p->stage_f, p->f_bytes);
    if (e == cudaSuccess) e = cudaMalloc(&p->stage_y, p->y_bytes);
    p->workspace_bytes += static_cast<int64_t>(p->x_bytes + p->f_bytes + p->y_bytes);
  }
  if (e == cudaSuccess && o.host_staging == 2) {
    e = cudaMalloc(&p->stage_x2, p->x_bytes);
    if (e == cudaSuccess) e = cudaMalloc(&p->stage_f2, p->f_bytes);
    if (e == cudaSuccess) e = cudaMalloc(&p->stage_y2, p->y_bytes);
    p->workspace_bytes += static_cast<int64_t>(p->x_bytes + p->f_bytes + p->y_bytes);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p->s_in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p->s_out, cudaStreamNonBlocking);
    for (cudaEvent_t* ev : {&p->ev_begin, &p->ev_in[0], &p->ev_in[1], &p->ev_run[0], &p->ev_run[1], &p->ev_out[0],
                            &p->ev_out[1]})
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
  }
  for (int i = 0; e == cudaSuccess && i < o.timing_events; ++i) {
    cudaEvent_t a = nullptr, b = nullptr;
    e = cudaEventCreate(&a);
    if (e == cudaSuccess) e = cudaEventCreate(&b);
    if (a) p->ev_start.push_back(a);
    if (b) p->ev_end.push_back(b);
  }
  if (e != cudaSuccess) {
    free_plan_memory(p);
    delete p;
    return from_cuda(e);
  }

  // fp16 filter as a 3-D tensor {32 channels, K, C/32*R*S}; one box is the
  // 32-channel rows of the output channels one CTA stages (BN, or BN/2 per
  // CTA of a pair) for a run of K-slices, 64-byte swizzled.
  cuuint64_t dims[3] = {32, static_cast<cuuint64_t>(s.K), static_cast<cuuint64_t>(p->num_slices)};
  cuuint64_t strides[2] = {64, static_cast<cuuint64_t>(s.K) * 64};
  cuuint32_t box[3] = {32, static_cast<cuuint32_t>(bn / p->cta_group),
                       static_cast<cuuint32_t>(p->kernel_variant >= 2 ? p->halo.bgroup : 1)};
  if (p->kernel_variant == 6) {
    // the stacked copy: slots of 64 rows; a box is one filter row's U slots of one rank
    const int U = p->halo.slots;
    dims[1] = 64;
    dims[2] = static_cast<cuuint64_t>(s.C / 32) * s.R * 2 * U;
    strides[1] = 64 * 64;
    box[1] = 64;
    box[2] = static_cast<cuuint32_t>(U);
  }
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult cr = encode(&p->tmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, p->f16, dims, strides, box, estr,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) {
    free_plan_memory(p);
    delete p;
    return I8C_ERR_CUDA;
  }
  *out = p;
  return I8C_OK;
}

namespace {

void fill_layout(const i8c_plan* pl, i8c_layout* L) {
  *L = i8c_layout{};
  L->kernel_variant = pl->kernel_variant;
  L->cta_group = pl->cta_group;
  L->block_n = pl->block_n;
  L->smem_bytes = pl->smem_bytes;
  L->tmem_cols = static_cast<int32_t>(pl->tmem_cols);
  L->chunk_slices = pl->chunk_slices;
  L->num_chunks = pl->num_chunks;
  if (pl->kernel_variant >= 2) {
    const i8c::HaloParams& h = pl->halo;
    L->flat_tiles = h.flat;
    L->tile_px = h.flat ? h.tile_px : pl->kernel_variant == 6 ? h.vq : 0;
    L->halo_rows = h.HR;
    L->halo_cw = h.CW;
    L->positions = h.positions;
    L->plane_bytes = static_cast<int32_t>(h.plane_bytes);
    L->halo_bytes = static_cast<int32_t>(h.halo_bytes);
    L->halo_stages = h.nhs;
    L->off_staging = static_cast<int32_t>(h.off_stg);
    L->staging_slots = h.nstg;
    L->staging_bytes = static_cast<int32_t>(h.stg_bytes);
    L->off_filter = static_cast<int32_t>(h.off_b);
    L->filter_stages = h.nbs;
    L->filter_run = h.bgroup;
    // rows per K-slice of a stage: transposed tiles 128 channels, the stacked
    // kernel a slot of 64 rows, the halo kernel the CTA's share of the tile
    const int rows = pl->kernel_variant == 6 ? 64 : pl->kernel_variant >= 4 ? 128 : pl->block_n / pl->cta_group;
    L->filter_stage_bytes = h.bgroup * rows * 64;
    L->off_out = static_cast<int32_t>(h.off_out);
    L->off_bar = static_cast<int32_t>(h.off_bar);
    L->tma_halo = h.tma_halo;
    L->x8_slots = h.nxs;
    L->off_x8 = static_cast<int32_t>(h.off_x8);
    L->x8_bytes = static_cast<int32_t>(h.x8_bytes);
    L->box_w = h.box_w;
    L->box_h = h.box_h;
    L->bar_bytes = i8c::kHaloBarBytes;
    for (int f = 0; f < 9; ++f) L->phase_off[f] = h.phase_off[f];
    L->subtiles = h.subtiles == 2 ? 2 : 1;
  } else {
    auto gather = [&](auto cfg) {
      using Cfg = decltype(cfg);
      L->gather_stages = Cfg::kStages;
      L->gather_off_a = Cfg::kOffA;
      L->gather_stage_a = Cfg::kAStage;
      L->gather_off_b = Cfg::kOffB;
      L->gather_stage_b = Cfg::kBStage;
      L->gather_off_staging = Cfg::kOffStg;
      L->gather_staging_slots = Cfg::kStg;
      L->gather_staging_bytes = Cfg::kStgBytes;
      L->gather_off_bar = Cfg::kOffBar;
    };
    if (pl->block_n >= 256) gather(i8c::TileCfg<256>{});
    else if (pl->block_n >= 128) gather(i8c::TileCfg<128>{});
    else if (pl->block_n >= 64) gather(i8c::TileCfg<64>{});
    else gather(i8c::TileCfg<32>{});
  }
}

}  // namespace

i8c_status i8c_plan_layout(const i8c_conv_shape* shape, const i8c_options* opts, int32_t num_sms, i8c_layout* out) {
  if (out == nullptr || num_sms < 1) return I8C_ERR_INVALID_ARG;
  int64_t P = 0, Q = 0;
  i8c_status st = check_supported(shape, &P, &Q);
  if (st != I8C_OK) return st;
  i8c_options o{};
  if (opts) o = *opts;
  if (!options_valid(o)) return I8C_ERR_INVALID_ARG;
  i8c_plan pl{};
  int64_t split_bytes = 0;
  st = plan_geometry(*shape, o, P, Q, o.num_ctas > 0 ? o.num_ctas : num_sms, true, &pl, &split_bytes);
  if (st != I8C_OK) return st;
  fill_layout(&pl, out);
  return I8C_OK;
}

i8c_status i8c_plan_get_layout(const i8c_plan* plan, i8c_layout* out) {
  if (plan == nullptr || out == nullptr) return I8C_ERR_INVALID_ARG;
  fill_layout(plan, out);
  return I8C_OK;
}

i8c_status i8c_plan_destroy(i8c_plan* plan) {
  if (plan == nullptr) return I8C_ERR_INVALID_ARG;
  cudaError_t e = cudaDeviceSynchronize();
  free_plan_memory(plan);
  delete plan;
  return from_cuda(e);
}

i8c_status i8c_plan_get_info(const i8c_plan* pl, i8c_plan_info* info) {
  if (pl == nullptr || info == nullptr) return I8C_ERR_INVALID_ARG;
  const i8c_conv_shape& s = pl->shape;
  info->P = pl->P;
  info->Q = pl->Q;
  info->M = pl->M;
  info->gemm_n = s.K;
  info->gemm_k = s.C * s.R * s.S;
  info->block_m = pl->kernel_variant == 4 || pl->kernel_variant == 5 ? pl->cta_group * pl->halo.tile_px
                  : pl->kernel_variant == 6                          ? 2 * pl->halo.vq
                                                                     : 128 * pl->cta_group;
  info->block_n = pl->block_n;
  info->num_tiles = pl->num_tiles;
  info->num_ctas = pl->num_ctas;
  info->num_chunks = pl->num_chunks;
  info->chunk_slices = pl->chunk_slices;
  info->acc_buffers = pl->acc_buffers;
  info->smem_bytes = pl->smem_bytes;
  info->kernels_per_run = pl->gbar != nullptr || (pl->kernel_variant >= 2 && pl->halo.f_smem) ? 1 : 2;
  info->kernel_variant = pl->kernel_variant;
  info->halo_staging = pl->kernel_variant >= 2 ? pl->halo.nstg : 0;
  info->filter_run = pl->kernel_variant >= 2 ? pl->halo.bgroup : 1;
  info->tail_split = pl->kernel_variant >= 2 ? pl->halo.ksplit : 1;
  info->tail_halves = pl->kernel_variant >= 2 ? pl->halo.nsplit : 1;
  info->flat_tiles = pl->kernel_variant >= 2 ? pl->halo.flat : 0;
  info->filter_resident = pl->kernel_variant >= 2 ? pl->halo.resident : 0;
  info->work_units = pl->kernel_variant >= 2 ? pl->halo.num_units : pl->num_tiles;
  info->filter_stages = pl->kernel_variant >= 2 ? pl->halo.nbs
                        : pl->block_n >= 256 ? i8c::TileCfg<256>::kStages
                        : pl->block_n >= 128 ? i8c::TileCfg<128>::kStages
                                             : i8c::TileCfg<64>::kStages;
  info->ops = 2 * pl->M * s.K * static_cast<int64_t>(s.C) * s.R * s.S;
  info->workspace_bytes = pl->workspace_bytes;
  return I8C_OK;
}

i8c_status i8c_plan_trace(const i8c_plan* pl, long long* out, int64_t count) {
  if (pl == nullptr || out == nullptr || count < 0) return I8C_ERR_INVALID_ARG;
  if (pl->trace == nullptr) return I8C_ERR_INVALID_ARG;
  const int64_t n = count < i8c::kTraceRows * i8c::kTraceSlots ? count : i8c::kTraceRows * i8c::kTraceSlots;
  return from_cuda(cudaMemcpy(out, pl->trace, sizeof(long long) * n, cudaMemcpyDeviceToHost));
}

i8c_status i8c_plan_kernel_time(const i8c_plan* pl, double* total_ms, int64_t* launches) {
  if (pl == nullptr || total_ms == nullptr || launches == nullptr) return I8C_ERR_INVALID_ARG;
  const int64_t nev = static_cast<int64_t>(pl->ev_start.size());
  *total_ms = 0.0;
  *launches = 0;
  if (nev == 0 || pl->ev_recorded == 0) return I8C_OK;
  const int64_t count = pl->ev_recorded < nev ? pl->ev_recorded : nev;
  cudaError_t e = cudaEventSynchronize(pl->ev_end[(pl->ev_recorded - 1) % nev]);
  if (e != cudaSuccess) return from_cuda(e);
  double sum = 0.0;
  for (int64_t i = pl->ev_recorded - count; i < pl->ev_recorded; ++i) {
    float ms = 0.0f;
    e = cudaEventElapsedTime(&ms, pl->ev_start[i % nev], pl->ev_end[i % nev]);
    if (e != cudaSuccess) return from_cuda(e);
    sum += ms;
  }
  *total_ms = sum;
  *launches = count;
  pl->ev_recorded = 0;
  return I8C_OK;
}

i8c_status i8c_plan_run(const i8c_plan* plan, const int8_t* x, const int8_t* f, int8_t* y, float alpha,
                        cudaStream_t stream) {
  if (plan == nullptr || x == nullptr || f == nullptr || y == nullptr) return I8C_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(f) || !aligned16(y)) return I8C_ERR_MISALIGNED;
  return run_plan(plan, x, f, y, nullptr, alpha, stream);
}

i8c_status i8c_plan_run_ex(const i8c_plan* plan, const int8_t* x, const int8_t* f, int8_t* y, float alpha,
                           const i8c_epilogue* ep, cudaStream_t stream) {
  if (plan == nullptr || x == nullptr || f == nullptr || y == nullptr) return I8C_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(f) || !aligned16(y)) return I8C_ERR_MISALIGNED;
  if (ep != nullptr && ((ep->alpha != nullptr && !aligned16(ep->alpha)) || (ep->bias != nullptr && !aligned16(ep->bias))))
    return I8C_ERR_MISALIGNED;
  return run_plan(plan, x, f, y, nullptr, alpha, stream, ep);
}

i8c_status i8c_plan_run_acc(const i8c_plan* plan, const int8_t* x, const int8_t* f, int32_t* acc,
                            cudaStream_t stream) {
  if (plan == nullptr || x == nullptr || f == nullptr || acc == nullptr) return I8C_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(f) || !aligned16(acc)) return I8C_ERR_MISALIGNED;
  return run_plan(plan, x, f, nullptr, acc, 1.0f, stream);
}

i8c_status i8c_plan_set_filter(const i8c_plan* plan, const int8_t* f, cudaStream_t stream) {
  if (plan == nullptr || f == nullptr) return I8C_ERR_INVALID_ARG;
  if (!aligned16(f)) return I8C_ERR_MISALIGNED;
  // the kernels that write their resident filter themselves read an int8
  // copy of it at every run; every other kernel reads the converted operand
  const cudaError_t e =
      plan->kernel_variant != 6 && converts_in_kernel(plan) && plan->gbar == nullptr
          ? cudaMemcpyAsync(plan->f16, f, plan->f_bytes, cudaMemcpyDeviceToDevice, stream)
          : convert_filter(plan, f, stream);
  if (e != cudaSuccess) return from_cuda(e);
  plan->prepacked = true;
  plan->filter_fresh = true;
  return I8C_OK;
}

i8c_status i8c_plan_run_prepacked(const i8c_plan* plan, const int8_t* x, int8_t* y, float alpha,
                                  cudaStream_t stream) {
  if (plan == nullptr || x == nullptr || y == nullptr || !plan->prepacked) return I8C_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y)) return I8C_ERR_MISALIGNED;
  return run_plan(plan, x, nullptr, y, nullptr, alpha, stream, nullptr, true);
}

i8c_status i8c_plan_run_prepacked_ex(const i8c_plan* plan, const int8_t* x, int8_t* y, float alpha,
                                     const i8c_epilogue* ep, cudaStream_t stream) {
  if (plan == nullptr || x == nullptr || y == nullptr || !plan->prepacked) return I8C_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y)) return I8C_ERR_MISALIGNED;
  if (ep != nullptr && ((ep->alpha != nullptr && !aligned16(ep->alpha)) || (ep->bias != nullptr && !aligned16(ep->bias))))
    return I8C_ERR_MISALIGNED;
  return run_plan(plan, x, nullptr, y, nullptr, alpha, stream, ep, true);
}

i8c_status i8c_plan_run_host(const i8c_plan* pl, const int8_t* x_host, const int8_t* f_host, int8_t* y_host,
                             float alpha, cudaStream_t stream) {
  if (pl == nullptr || x_host == nullptr || f_host == nullptr || y_host == nullptr) return I8C_ERR_INVALID_ARG;
  if (pl->stage_x == nullptr) return I8C_ERR_INVALID_ARG;
  cudaError_t e = cudaMemcpyAsync(pl->stage_x, x_host, pl->x_bytes, cudaMemcpyHostToDevice, stream);
  if (e == cudaSuccess) e = cudaMemcpyAsync(pl->stage_f, f_host, pl->f_bytes, cudaMemcpyHostToDevice, stream);
  if (e != cudaSuccess) return from_cuda(e);
  i8c_status st = run_plan(pl, pl->stage_x, pl->stage_f, pl->stage_y, nullptr, alpha, stream);
  if (st != I8C_OK) return st;
  return from_cuda(cudaMemcpyAsync(y_host, pl->stage_y, pl->y_bytes, cudaMemcpyDeviceToHost, stream));
}

i8c_status i8c_plan_run_host_pipelined(const i8c_plan* pl, const int8_t* const* x_host, const int8_t* const* f_host,
                                       int8_t* const* y_host, const float* alpha, int32_t steps,
                                       cudaStream_t stream) {
  if (pl == nullptr || x_host == nullptr || f_host == nullptr || y_host == nullptr || alpha == nullptr || steps < 0)
    return I8C_ERR_INVALID_ARG;
  if (pl->stage_x2 == nullptr) return I8C_ERR_INVALID_ARG;
  for (int32_t i = 0; i < steps; ++i)
    if (x_host[i] == nullptr || f_host[i] == nullptr || y_host[i] == nullptr) return I8C_ERR_INVALID_ARG;
  int8_t* const sx[2] = {pl->stage_x, pl->stage_x2};
  int8_t* const sf[2] = {pl->stage_f, pl->stage_f2};
  int8_t* const sy[2] = {pl->stage_y, pl->stage_y2};
  // the copy streams start after the work already on `stream`
  cudaError_t e = cudaEventRecord(pl->ev_begin, stream);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(pl->s_in, pl->ev_begin, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(pl->s_out, pl->ev_begin, 0);
  for (int32_t i = 0; e == cudaSuccess && i < steps; ++i) {
    const int b = i & 1;
    // inputs of step i into set b once run i - 2 has read that set
    if (i >= 2) e = cudaStreamWaitEvent(pl->s_in, pl->ev_run[b], 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(sx[b], x_host[i], pl->x_bytes, cudaMemcpyHostToDevice, pl->s_in);
    if (e == cudaSuccess) e = cudaMemcpyAsync(sf[b], f_host[i], pl->f_bytes, cudaMemcpyHostToDevice, pl->s_in);
    if (e == cudaSuccess) e = cudaEventRecord(pl->ev_in[b], pl->s_in);
    // run i on `stream` once its inputs are in and step i - 2's output has left set b
    if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, pl->ev_in[b], 0);
    if (e == cudaSuccess && i >= 2) e = cudaStreamWaitEvent(stream, pl->ev_out[b], 0);
    if (e != cudaSuccess) break;
    const i8c_status st = run_plan(pl, sx[b], sf[b], sy[b], nullptr, alpha[i], stream);
    if (st != I8C_OK) return st;
    e = cudaEventRecord(pl->ev_run[b], stream);
    // output of step i back to the host
    if (e == cudaSuccess) e = cudaStreamWaitEvent(pl->s_out, pl->ev_run[b], 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(y_host[i], sy[b], pl->y_bytes, cudaMemcpyDeviceToHost, pl->s_out);
    if (e == cudaSuccess) e = cudaEventRecord(pl->ev_out[b], pl->s_out);
  }
  // `stream` reaches the end of the call once the last output copy is done
  if (e == cudaSuccess) e = cudaEventRecord(pl->ev_begin, pl->s_out);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, pl->ev_begin, 0);
  return from_cuda(e);
}

i8c_status i8c_plan_status(const i8c_plan* pl, cudaStream_t stream) {
  if (pl == nullptr) return I8C_ERR_INVALID_ARG;
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return from_cuda(e);
  int h = 0;
  e = cudaMemcpy(&h, pl->status, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return from_cuda(e);
  if (h != 0) {
    e = cudaMemset(pl->status, 0, sizeof(int));
    // a launch that gave up may have left split-tile arrivals behind
    if (e == cudaSuccess && pl->split_count != nullptr)
      e = cudaMemset(pl->split_count, 0, sizeof(int) * static_cast<size_t>(pl->split_tiles) * pl->cta_group);
    // and a grid barrier with missing arrivals
    if (e == cudaSuccess && pl->gbar != nullptr) e = cudaMemset(pl->gbar, 0, 2 * sizeof(uint32_t));
    if (e != cudaSuccess) return from_cuda(e);
  }
  return h == 0 ? I8C_OK : static_cast<i8c_status>(h);
}

i8c_status i8c_conv2d_fprop(const int8_t* x, const int8_t* f, int8_t* y, const i8c_conv_shape* shape, float alpha,
                            cudaStream_t stream) {
  if (x == nullptr || f == nullptr || y == nullptr) return I8C_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(f) || !aligned16(y)) return I8C_ERR_MISALIGNED;
  i8c_plan* p = nullptr;
  i8c_status st = cached_plan(shape, stream, &p);
  if (st != I8C_OK) return st;
  return run_plan(p, x, f, y, nullptr, alpha, stream);
}

i8c_status i8c_conv2d_fprop_ex(const int8_t* x, const int8_t* f, int8_t* y, const i8c_conv_shape* shape,
                               float alpha, const i8c_epilogue* ep, cudaStream_t stream) {
  if (x == nullptr || f == nullptr || y == nullptr) return I8C_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(f) || !aligned16(y)) return I8C_ERR_MISALIGNED;
  if (ep != nullptr && ((ep->alpha != nullptr && !aligned16(ep->alpha)) || (ep->bias != nullptr && !aligned16(ep->bias))))
    return I8C_ERR_MISALIGNED;
  i8c_plan* p = nullptr;
  i8c_status st = cached_plan(shape, stream, &p);
  if (st != I8C_OK) return st;
  return run_plan(p, x, f, y, nullptr, alpha, stream, ep);
}

i8c_status i8c_conv2d_fprop_acc(const int8_t* x, const int8_t* f, int32_t* acc, const i8c_conv_shape* shape,
                                cudaStream_t stream) {
  if (x == nullptr || f == nullptr || acc == nullptr) return I8C_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(f) || !aligned16(acc)) return I8C_ERR_MISALIGNED;
  i8c_plan* p = nullptr;
  i8c_status st = cached_plan(shape, stream, &p);
  if (st != I8C_OK) return st;
  return run_plan(p, x, f, nullptr, acc, 1.0f, stream);
}

i8c_status i8c_last_device_status(cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return from_cuda(e);
  e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return from_cuda(e);
  i8c_status first = I8C_OK;
  {
    std::lock_guard<std::mutex> lock(g_cache_mu);
    const int64_t sk = static_cast<int64_t>(reinterpret_cast<uintptr_t>(stream));
    for (auto& kv : g_cache) {
      if (kv.first[0] != dev || kv.first[1] != sk) continue;
      const i8c_status st = i8c_plan_status(kv.second.plan, stream);
      if (st != I8C_OK && first == I8C_OK) first = st;
    }
  }
  const i8c_status na = static_cast<i8c_status>(i8c::noalloc_take_status(dev));
  return first != I8C_OK ? first : na;
}

i8c_status i8c_debug_set_oneshot(int32_t debug_flags, int32_t wait_timeout_us) {
  if (debug_flags < 0 || wait_timeout_us < 0) return I8C_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_cache_mu);
  for (auto& kv : g_cache) i8c_plan_destroy(kv.second.plan);
  g_cache.clear();
  g_oneshot_debug_flags = debug_flags;
  g_oneshot_timeout_us = wait_timeout_us;
  i8c::noalloc_set_debug(debug_flags, wait_timeout_us);
  return I8C_OK;
}

int64_t i8c_oneshot_cached_plans(void) {
  std::lock_guard<std::mutex> lock(g_cache_mu);
  return static_cast<int64_t>(g_cache.size());
}

i8c_status i8c_pack_nchw_to_ncxhwx32(const int8_t* src, int8_t* dst, int32_t N, int32_t C, int32_t H, int32_t W,
                                     cudaStream_t stream) {
  if (src == nullptr || dst == nullptr || N < 1 || C < 1 || H < 1 || W < 1) return I8C_ERR_INVALID_ARG;
  if (C % 32 != 0) return I8C_ERR_UNSUPPORTED;
  return from_cuda(i8c::launch_pack_act(src, dst, N, C, H, W, true, stream));
}

i8c_status i8c_unpack_ncxhwx32_to_nchw(const int8_t* src, int8_t* dst, int32_t N, int32_t C, int32_t H, int32_t W,
                                       cudaStream_t stream) {
  if (src == nullptr || dst == nullptr || N < 1 || C < 1 || H < 1 || W < 1) return I8C_ERR_INVALID_ARG;
  if (C % 32 != 0) return I8C_ERR_UNSUPPORTED;
  return from_cuda(i8c::launch_pack_act(src, dst, N, C, H, W, false, stream));
}

i8c_status i8c_pack_kcrs_to_cxrskx32(const int8_t* src, int8_t* dst, int32_t K, int32_t C, int32_t R, int32_t S,
                                     cudaStream_t stream) {
  if (src == nullptr || dst == nullptr || K < 1 || C < 1 || R < 1 || S < 1) return I8C_ERR_INVALID_ARG;
  if (C % 32 != 0) return I8C_ERR_UNSUPPORTED;
  return from_cuda(i8c::launch_pack_filter(src, dst, K, C, R, S, true, stream));
}

i8c_status i8c_unpack_cxrskx32_to_kcrs(const int8_t* src, int8_t* dst, int32_t K, int32_t C, int32_t R, int32_t S,
                                       cudaStream_t stream) {
  if (src == nullptr || dst == nullptr || K < 1 || C < 1 || R < 1 || S < 1) return I8C_ERR_INVALID_ARG;
  if (C % 32 != 0) return I8C_ERR_UNSUPPORTED;
  return from_cuda(i8c::launch_pack_filter(src, dst, K, C, R, S, false, stream));
}

}  // extern "C"
