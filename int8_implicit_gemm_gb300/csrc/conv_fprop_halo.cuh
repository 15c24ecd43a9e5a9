// INT8 NCxHWx<32> Conv2d fprop on the sm_103a tensor cores, halo variant.
//
// Same GEMM view and exact fp16/fp32-chunk arithmetic as conv_fprop_tc.cuh,
// but the 128 GEMM rows of a tile are a 16 x 8 patch of output pixels of one
// image (16 output rows, 8 consecutive output columns).  For one 32-channel
// block cb the producers load the input region every tap of the patch needs
// -- the halo, (15*sh + (R-1)*dh + 1) rows x (7*sw + (S-1)*dw + 1) columns --
// once, convert it to fp16 once, and store it as four 8-channel planes in the
// canonical no-swizzle K-major layout with one 16-byte entry per pixel.  The
// A operand of filter tap (r, s) is then a shifted view of that halo: eight
// consecutive output columns are eight consecutive 16-byte entries (a core
// matrix), consecutive output rows are sh halo rows apart (the descriptor's
// stride), and the tap offset moves the start address by r*dh rows and
// s*dw columns.  Each input vector is converted once per patch instead of
// once per tap.  Column strides > 1 are handled by storing the halo columns
// phase by phase (all columns c with c % sw == 0 first, then 1, ...), so the
// eight columns of a core matrix stay adjacent.
//
// Warp roles (512 threads): warp 0 MMA issuer and TMEM owner, warp 4 filter
// TMA, warps 1-3 and 5-7 halo producers, warps 8-15 epilogue (two per TMEM
// lane quarter, each draining half of the tile's columns).  All waits are
// bounded.
#pragma once

#include "conv_fprop_tc.cuh"

namespace i8c {

struct HaloParams {
  ConvParams c;
  // Tile geometry.  2-D patches: 16 x 8 output pixels, TPH x TQW per image.
  // Flat tiles (stride 1 only): 128 consecutive pixels of the output laid
  // out row-major with the zero-padded input's row width CW; tpi per image
  // (the CW - Q pixels at the end of each row are computed and discarded),
  // and the halo is the contiguous run of `positions` padded input pixels
  // that the 128 pixels' taps read.
  int flat;
  int TPH, TQW;             // 2-D: patches per image along P (16 rows each) and Q (8 columns each)
  int tpi;                  // flat: tiles per image, ceil(P * CW / tile_px)
  int tile_px;              // flat: output pixels per tile (128; the transposed-tile kernel: 16..256)
  int num_patches;          // N * TPH * TQW, or N * tpi
  int HR, CW;               // halo rows, halo positions per row (flat: CW = padded input width)
  int positions;            // halo positions: HR * CW, or (flat) 128 + (R-1)*dh*CW + (S-1)*dw
  uint32_t plane_bytes;     // one 8-channel plane: HR*CW*16 (rounded up to 128)
  uint32_t halo_bytes;      // one halo stage: 4 planes
  uint32_t stg_bytes;       // one int8 staging slot: HR*CW*32 (rounded up to 128)
  int nstg;                 // int8 staging slots: 2 or 3, or 0 (producers load into registers)
  int nbs;                  // filter pipeline stages (<= kMaxBStages)
  int resident;             // 1: the nbs stages are one unit's whole filter, loaded once and kept
  int nhs;                  // fp16 halo stages: 2 or 3
  int bgroup;               // K-slices per filter stage (one TMA box, one wait, one release)
  uint32_t off_stg, off_b, off_bar;
  uint32_t off_out;         // transposed-tile kernel: the epilogue's output staging rows
  int phase_off[9];         // first position of column phase f (f < sw); phase_off[sw] = CW
  // Work units: tiles [0, full_units) whole; the remaining tiles (the last,
  // partial wave) each split into ksplit units over ranges of channel blocks,
  // whose int32 partial sums meet in split_part and are combined by the unit
  // that finishes last (split_count: arrivals per tile and CTA rank).
  // Or (nsplit = 2, single CTAs) each remaining tile splits into its two
  // halves of output channels: two units with disjoint outputs, MMAs of N =
  // BN/2, no partial sums.
  int num_units, full_units, ksplit, nsplit;
  int* split_count;         // [tail tiles][cg], zero between launches
  int32_t* split_part;      // [tail tiles][ksplit][cg][BN/4][128][4]
  // In-kernel filter conversion (single CTAs, cooperative launch): the
  // epilogue warps of every CTA convert a share of the int8 filter into f16
  // before their first drain; a grid barrier (gbar: arrivals, generation)
  // tells the filter TMA warps that the whole copy is written.
  const int8_t* f_int8;     // null: the conversion kernel ran before this one
  uint16_t* f16;
  int64_t f_vecs;           // 16-element vectors of the filter
  uint32_t* gbar;           // {arrivals, generation}, arrivals zero between launches
  // Stacked-tap kernel (64 output channels): tiles of 128 consecutive output
  // columns of one row, vq of them valid, tq per output row; the halo is one
  // segment of seg_len input columns per filter row; slots = MMAs (tap pairs
  // and an odd last tap) per filter row and 16-channel half.
  int seg_len, vq, tq, slots;
  // Halo loads by TMA (tma_halo = 1): for every channel block, one box of
  // the input -- the tile's halo region in natural order (2-D patches:
  // box_h rows x box_w columns), or the whole zero-padded input rows the
  // flat run spans (flat tiles: box_w = W + 2*pad_w) -- lands in one of nxs
  // int8 slots of x8_bytes at off_x8 (x8_box bytes each), and the producer
  // threads convert it to the fp16 halo.  The kernels take the activations'
  // tensor map (a 4-D tensor {32 channels, W, H, N*C/32} of bytes, encoded
  // for every run) as a parameter of its own.
  int tma_halo, nxs, box_w, box_h;
  uint32_t off_x8, x8_bytes, x8_box;
  // Resident filter written by the kernel itself (f_smem = 1): all threads
  // convert the int8 CxRSKx<32> filter f_src straight into the filter stages
  // before the warp roles split; there is no fp16 copy in global memory and
  // no filter TMA, so a run is one launch.
  int f_smem;
  const int8_t* f_src;
  // 1: the filter operand (the fp16 copy, or f_src) was not written by the
  // kernel launched just before this one (a prepacked run after the first),
  // so it is read without waiting for that kernel
  int filter_ready;
  // 2-D patches of 16 x (8 * subtiles) output pixels: subtiles = 2 puts two
  // 16x8 sub-tiles side by side on one halo (16x16 patches); every tap then
  // issues two M = 128 MMAs per K half, the second on the halo 8 positions
  // on, into an accumulator pair (BN columns each) per buffer.  0 or 1: one.
  int subtiles;
};


constexpr int kMaxBStages = 16;
// Warp roles: 0 MMA issuer, kTmaWarp filter TMA, the other warps below 8 halo
// producers, 8-15 epilogue.  Warps w, w+4, w+8, w+12 share one scheduler;
// the mostly sleeping TMA warp sits next to the MMA warp, whose issue latency
// the tensor core's short queue exposes, instead of a busy producer warp.
constexpr int kTmaWarp = 4;
constexpr int kProducers = 192;   // halo producer threads: warps 2-7
constexpr int kEpilogue = 256;    // epilogue threads: warps 8-15, two per TMEM lane quarter
constexpr int kHaloThreads = 512;
// Register budgets per warpgroup after setmaxnreg: the two epilogue warpgroups
// hold the running sums; 128 * (2 * kWorkerRegs + 2 * kEpilogueRegs) must not
// exceed the 512 * 128 registers the block is launched with.
constexpr uint32_t kWorkerRegs = 72;
constexpr uint32_t kEpilogueRegs = 184;
static_assert(128 * (2 * kWorkerRegs + 2 * kEpilogueRegs) <= 512 * 128, "register split");
constexpr int kHaloBarBytes = 512;

struct PatchTile {
  int n, p0, q0, nt;
  bool valid;  // false for the missing second patch of a CTA pair's last tile
  int m0;      // flat tiles: first pixel in the padded row-major output (p0 = q0 = 0)
};

// Tile schedule of one CTA: tiles first, first + step, ...; a tile is
// (group of cg patches, N-tile) and this CTA computes patch `rank` of the
// group (cg = 2 for CTA pairs, whose two CTAs walk the same tiles).  fwd:
// a pair's rank 1 arrives on its own halo barriers, whose completions one
// lane forwards to rank 0 (the halo kernel's producers).
struct TileSched {
  int first, step, rank, cg, fwd;
};

// Derived from the block index alone, so the compiler can recompute it
// instead of keeping it in registers: in a 1-D grid of clusters of two, CTA
// 2c + r is rank r of cluster c.
template <int CG>
__device__ __forceinline__ TileSched tile_sched() {
  if constexpr (CG == 2)
    return {static_cast<int>(blockIdx.x) >> 1, static_cast<int>(gridDim.x) >> 1, static_cast<int>(blockIdx.x) & 1,
            2};
  return {static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x), 0, 1};
}

__device__ __forceinline__ PatchTile decode_patch(int tile, const HaloParams& hp, const TileSched& ts) {
  const int nt = tile % hp.c.num_n_tiles;
  const int patch = (tile / hp.c.num_n_tiles) * ts.cg + ts.rank;
  if (hp.flat) return {patch / hp.tpi, 0, 0, nt, patch < hp.num_patches, (patch % hp.tpi) * hp.tile_px};
  const int qt = patch % hp.TQW;
  const int rest = patch / hp.TQW;
  const int pt = rest % hp.TPH;
  return {rest / hp.TPH, pt * 16, qt * (hp.subtiles == 2 ? 16 : 8), nt, patch < hp.num_patches, 0};
}

// Arrive on a barrier of the MMA-issuing CTA, called by all 32 lanes of a
// warp (`mine`: whether this lane's arrival counts): each lane arrives on
// this CTA's own barrier, or for rank 1 of a pair one lane arrives for the
// whole warp on the barrier at the same offset in rank 0, after a warp
// barrier that orders the other lanes' writes before its cluster-scope
// release (one remote transaction per warp instead of 32).  (One local
// arrive per warp as well, after the same warp barrier, measured slower:
// 326.7 against 314.6 us on the 64-channel 5x9 layer.)
__device__ __forceinline__ void arrive_on_leader(uint64_t* bar, const TileSched& ts, bool mine = true) {
  if (ts.rank == 0 || ts.fwd) {
    if (mine) ptx::mbar_arrive(bar);
  } else {
    __syncwarp();  // orders every lane's prior shared-memory writes before lane 0's release
    const uint32_t n = __popc(__ballot_sync(0xffffffffu, mine));
    if ((threadIdx.x & 31) == 0 && n != 0) ptx::mbar_arrive_remote(ptx::mapa(ptx::smem_addr(bar), 0), n);
  }
}

// Producer thread t of a group of whole warps stores the 16-byte half
// halo_lane_half(t) of halo position halo_lane_pos(t), then of the positions
// (group threads / 2) apart from it: each quarter-warp (the eight lanes whose
// 16-byte stores share one shared-memory wavefront) writes eight consecutive
// positions of one 8-channel plane, 128 contiguous bytes without a bank
// conflict, and each warp still reads 16 whole 32-byte input vectors.
__device__ __forceinline__ int halo_lane_half(int t) { return (t >> 3) & 1; }
__device__ __forceinline__ int halo_lane_pos(int t) { return ((t >> 5) << 4) + (((t >> 4) & 1) << 3) + (t & 7); }

// First halo position of thread pt and the walk between its positions.
struct HaloWalk {
  int e_first, b_first, pos_first, b_step, pos_step;
};
constexpr int kHaloStep = kProducers / 2;

__device__ __forceinline__ HaloWalk halo_walk(const HaloParams& hp, int pt) {
  HaloWalk w;
  w.e_first = halo_lane_pos(pt);
  w.b_first = w.e_first / hp.CW;
  w.pos_first = w.e_first - w.b_first * hp.CW;
  w.b_step = kHaloStep / hp.CW;
  w.pos_step = kHaloStep - w.b_step * hp.CW;
  return w;
}

// Flat tiles start m0 pixels into the padded image: move a walk's (row,
// column) there (m0 = 0 for 2-D patches).
__device__ __forceinline__ void halo_walk_origin(const HaloParams& hp, int m0, int& b, int& pos) {
  if (m0 == 0) return;
  const int mq = m0 / hp.CW;
  pos += m0 - mq * hp.CW;
  b += mq;
  if (pos >= hp.CW) {
    pos -= hp.CW;
    ++b;
  }
}

// Index in its row of the halo position that holds input column c (relative
// to the halo's first column): positions are ordered by column phase (column
// mod stride_w), phase f from phase_off[f].
__device__ __forceinline__ int halo_phase_index(const HaloParams& hp, int c) {
  const int sw = hp.c.stride_w;
  if (sw == 1) return c;
  if (sw == 2) return (c >> 1) + ((c & 1) ? hp.phase_off[1] : 0);
  const int f = c % sw;
  return hp.phase_off[f] + c / sw;
}

// A work unit: channel blocks [cb0, cb1) of one tile; part < 0 for a whole
// tile, else its index among the ksplit units of a split tile.
struct WorkUnit {
  int tile, cb0, cb1, part;
  int nh;  // half of the tile's output channels (0 or 1), or -1 for all of them
};

__device__ __forceinline__ WorkUnit decode_unit(int i, const HaloParams& hp) {
  const int CB = hp.c.CB;
  if (i < hp.full_units) return {i, 0, CB, -1, -1};
  const int j = i - hp.full_units;
  if (hp.nsplit == 2) return {hp.full_units + j / 2, 0, CB, -1, j % 2};
  const int part = j % hp.ksplit;
  return {hp.full_units + j / hp.ksplit, part * CB / hp.ksplit, (part + 1) * CB / hp.ksplit, part, -1};
}

// This CTA's channel blocks in order: unit by unit (first, first + step, ...),
// each unit's blocks cb0 .. cb1 - 1.
struct StageIter {
  int unit, cb, tile, cb_end;
  __device__ __forceinline__ void load(const HaloParams& hp) {
    const WorkUnit wu = decode_unit(unit, hp);
    tile = wu.tile;
    cb = wu.cb0;
    cb_end = wu.cb1;
  }
  __device__ __forceinline__ StageIter(const HaloParams& hp, const TileSched& ts) : unit(ts.first), cb(0) {
    if (unit < hp.num_units) load(hp);
  }
  __device__ __forceinline__ bool valid(const HaloParams& hp) const { return unit < hp.num_units; }
  __device__ __forceinline__ void next(const HaloParams& hp, const TileSched& ts) {
    if (++cb == cb_end) {
      unit += ts.step;
      if (unit < hp.num_units) load(hp);
    }
  }
};

__device__ __forceinline__ void halo_store_f16(const HaloParams& hp, uint8_t* halo, int e, int h, const uint4& v) {
  uint4 c0, c1;
  i8x4_to_f16x4(v.x, c0.x, c0.y);
  i8x4_to_f16x4(v.y, c0.z, c0.w);
  i8x4_to_f16x4(v.z, c1.x, c1.y);
  i8x4_to_f16x4(v.w, c1.z, c1.w);
  *reinterpret_cast<uint4*>(halo + (2 * h) * hp.plane_bytes + e * 16) = c0;
  *reinterpret_cast<uint4*>(halo + (2 * h + 1) * hp.plane_bytes + e * 16) = c1;
}

// Producer through the int8 staging ring (hp.nstg slots of 32 bytes per
// position).  Returns false when a wait timed out.
__device__ __forceinline__ bool halo_produce_staged(const HaloParams& hp, const TileSched& ts, uint8_t* smem,
                                                   uint64_t* h_full, uint64_t* h_empty, volatile int* abort_flag,
                                                   int pt) {
  const ConvParams& p = hp.c;
  const int h = halo_lane_half(pt);
  const int positions = hp.positions;
  const HaloWalk w = halo_walk(hp, pt);
  const int HW32 = p.H * p.W * 32;
  const uint32_t stg_base = ptx::smem_addr(smem + hp.off_stg);
  StageIter lit(hp, ts);  // the stage being loaded, nstg - 1 ahead

  auto issue_load = [&](uint32_t slot) {
    if (lit.valid(hp)) {
      const PatchTile t = decode_patch(lit.tile, hp, ts);
      const int hb0 = t.p0 * p.stride_h - p.pad_h;
      const int wb0 = t.q0 * p.stride_w - p.pad_w;
      const int8_t* img = p.x + static_cast<int64_t>(t.n) * p.img_stride + lit.cb * HW32;
      const uint32_t dst0 = stg_base + slot * hp.stg_bytes;
      int b = w.b_first, pos = w.pos_first;
      halo_walk_origin(hp, t.m0, b, pos);
      for (int e = w.e_first; e < positions; e += kHaloStep) {  // natural order: pos is the input column
        const int hh = hb0 + b, ww = wb0 + pos;
        const bool in = t.valid && hh >= 0 && hh < p.H && ww >= 0 && ww < p.W;
        const int8_t* src = in ? img + (hh * p.W + ww) * 32 + h * 16 : p.x;
        ptx::cp_async_16_ca(dst0 + e * 32 + h * 16, src, in ? 16u : 0u);
        b += w.b_step;
        pos += w.pos_step;
        if (pos >= hp.CW) {
          pos -= hp.CW;
          ++b;
        }
      }
      lit.next(hp, ts);
    }
    ptx::cp_async_commit();
  };

  const int nstg = hp.nstg;
  for (int i = 0; i < nstg - 1; ++i) issue_load(static_cast<uint32_t>(i));
  bool ok = true;
  uint32_t s = 0, hs = 0, hph = 0;  // stage count; halo stage and its phase parity
#if defined(I8C_PIPELINE_TRACE)
  const bool ptrace = p.trace != nullptr && blockIdx.x < 2 && pt == 0;
#endif
  for (StageIter it(hp, ts); it.valid(hp); it.next(hp, ts), ++s) {
    issue_load((s + nstg - 1) % nstg);
    if (nstg == 3) ptx::cp_async_wait<2>();
    else ptx::cp_async_wait<1>();
    // warp-uniform outcome: the arrive below is a warp-wide operation
    if (!__all_sync(0xffffffffu, ptx::mbar_wait(&h_empty[hs], hph ^ 1u, p.timeout_ns, abort_flag))) {
      ok = false;
      break;
    }
#if defined(I8C_PIPELINE_TRACE)
    if (ptrace && s < static_cast<uint32_t>(kTraceSlots))
      p.trace[(16 + 2 * blockIdx.x) * kTraceSlots + s] = static_cast<long long>(ptx::globaltimer_ns());
#endif
    const uint8_t* stg = smem + hp.off_stg + (s % nstg) * hp.stg_bytes;
    uint8_t* halo = smem + hs * hp.halo_bytes;
    // the ring holds the pixels in natural order; the halo by column phase
    int ps = w.pos_first;
    if (hp.flat) ps = 0;  // stride 1: the phase order is the natural order
    for (int e = w.e_first; e < positions; e += kHaloStep) {
      halo_store_f16(hp, halo, e - ps + halo_phase_index(hp, ps), h,
                     *reinterpret_cast<const uint4*>(stg + e * 32 + h * 16));
      ps += w.pos_step;
      ps -= ps >= hp.CW ? hp.CW : 0;
    }
    ptx::fence_proxy_async_smem();
    arrive_on_leader(&h_full[hs], ts, !((p.debug_flags & 1) && s == 0 && pt == 0));
#if defined(I8C_PIPELINE_TRACE)
    if (ptrace && s < static_cast<uint32_t>(kTraceSlots))
      p.trace[(17 + 2 * blockIdx.x) * kTraceSlots + s] = static_cast<long long>(ptx::globaltimer_ns());
#endif
    hs = hs + 1 == static_cast<uint32_t>(hp.nhs) ? 0u : hs + 1;
    hph ^= hs == 0 ? 1u : 0u;
  }
  ptx::cp_async_wait_all();
  return ok;
}

// Producer that loads straight into registers, kBatch positions at a time
// (zeros outside the image).  Returns false when a wait timed out.
// kBatch loads per thread and batch: the batch the thread keeps in flight
// while it waits for its halo stage is the whole halo when it fits (6 loads
// for the 561 positions of a stride-2 16x8 patch, 8 for the 768 of the
// dilated 5x9 layer; 10 would not fit the producers' registers); the smaller
// batch where 6 suffice keeps the loop short.  kUnit: the kernel runs
// stride-1 layers only, whose column-phase order is the natural order.
template <int kBatch, bool kUnit = false>
__device__ __forceinline__ bool halo_produce_direct(const HaloParams& hp, const TileSched& ts, uint8_t* smem,
                                                   uint64_t* h_full, uint64_t* h_empty, volatile int* abort_flag,
                                                   int pt) {
  const ConvParams& p = hp.c;
  const int h = halo_lane_half(pt);
  const int positions = hp.positions;
  const HaloWalk w = halo_walk(hp, pt);
  const int HW32 = p.H * p.W * 32;
  uint32_t hs = 0, hph = 0;  // halo stage and its phase parity
  bool skip = (p.debug_flags & 1) && pt == 0;  // test hook: this thread skips its first arrival
#if defined(I8C_PIPELINE_TRACE)
  const bool ptrace = p.trace != nullptr && blockIdx.x < 2 && pt == 0;
  int tseq = 0;
#endif
  for (StageIter it(hp, ts); it.valid(hp); it.next(hp, ts)) {
    const PatchTile t = decode_patch(it.tile, hp, ts);
    const int hb0 = t.p0 * p.stride_h - p.pad_h;
    const int wb0 = t.q0 * p.stride_w - p.pad_w;
    const int8_t* img = p.x + static_cast<int64_t>(t.n) * p.img_stride + it.cb * HW32;
    uint8_t* halo = smem + hs * hp.halo_bytes;
    int e = w.e_first, b = w.b_first, pos = w.pos_first;
    halo_walk_origin(hp, t.m0, b, pos);
    bool stage_free = false;
    // the tile's next channel block (the same pixels one channel-block plane
    // on) is prefetched into L2 from these loads, one lane per 32-byte pixel
    const bool pf = h == 0 && it.cb + 1 < it.cb_end;
#if defined(I8C_PIPELINE_TRACE)
    if (ptrace && tseq < kTraceSlots)
      p.trace[(30 + blockIdx.x) * kTraceSlots + tseq] = static_cast<long long>(ptx::globaltimer_ns());
#endif
    do {
      // The walk visits the halo's input pixels in natural order (pos: the
      // input column within the halo, e: row * CW + pos), so that a warp's
      // loads are contiguous and no column needs a phase lookup; each pixel
      // is stored at its column-phase position in the row.
      uint4 v[kBatch];
      const int e0 = e, pos0 = pos;  // the walk's start: v[k] is k steps on
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        v[k] = make_uint4(0, 0, 0, 0);
        if (e < positions) {
          const int hh = hb0 + b, ww = wb0 + pos;
          const bool in = t.valid && hh >= 0 && hh < p.H && ww >= 0 && ww < p.W;
          const int8_t* src = img + (hh * p.W + ww) * 32 + h * 16;
          v[k] = ptx::ldg16_or_zero(src, in);
          if (pf && in) ptx::prefetch_l2(src + HW32);
          e += kHaloStep;
          b += w.b_step;
          pos += w.pos_step;
          if (pos >= hp.CW) {
            pos -= hp.CW;
            ++b;
          }
        }
      }
      if (!stage_free) {
#if defined(I8C_PIPELINE_TRACE)
        if (ptrace && tseq < kTraceSlots)
          p.trace[(28 + blockIdx.x) * kTraceSlots + tseq] = static_cast<long long>(ptx::globaltimer_ns());
#endif
        // every lane runs the first batch, so the warp is converged here; the
        // outcome is made warp-uniform because the arrive below is warp-wide
        if (!__all_sync(0xffffffffu, ptx::mbar_wait(&h_empty[hs], hph ^ 1u, p.timeout_ns, abort_flag)))
          return false;
        stage_free = true;
#if defined(I8C_PIPELINE_TRACE)
        if (ptrace && tseq < kTraceSlots)
          p.trace[(16 + 2 * blockIdx.x) * kTraceSlots + tseq] = static_cast<long long>(ptx::globaltimer_ns());
#endif
      }
      int ps = pos0;
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int ek = e0 + k * kHaloStep;
        if constexpr (kUnit) {
          if (ek < positions) halo_store_f16(hp, halo, ek, h, v[k]);
        } else {
          if (ek < positions) halo_store_f16(hp, halo, ek - ps + halo_phase_index(hp, ps), h, v[k]);
          ps += w.pos_step;
          ps -= ps >= hp.CW ? hp.CW : 0;
        }
      }
    } while (e < positions);
#if defined(I8C_PIPELINE_TRACE)
    if (ptrace && tseq < kTraceSlots)
      p.trace[(26 + blockIdx.x) * kTraceSlots + tseq] = static_cast<long long>(ptx::globaltimer_ns());
#endif
    ptx::fence_proxy_async_smem();
    arrive_on_leader(&h_full[hs], ts, !skip);
    skip = false;
#if defined(I8C_PIPELINE_TRACE)
    if (ptrace && tseq < kTraceSlots)
      p.trace[(17 + 2 * blockIdx.x) * kTraceSlots + tseq] = static_cast<long long>(ptx::globaltimer_ns());
    ++tseq;
#endif
    hs = hs + 1 == static_cast<uint32_t>(hp.nhs) ? 0u : hs + 1;
    hph ^= hs == 0 ? 1u : 0u;
  }
  return true;
}

// Producer for halos of at most (kProducers / ng / 2) * kB positions (one
// batch of 16-byte loads per thread and channel block), in ng groups of
// kProducers / ng threads (whole warps) that take channel blocks in turn:
// group g the blocks i with i % ng == g.  A group issues a channel block's
// loads as soon as it has stored its previous one, ng channel blocks
// earlier, so each load round trip (a DRAM miss for the first touch of an
// input row) has the MMAs of ng channel blocks to complete in, with one
// batch of registers per thread (kB loads: the kernel's register split for
// the producer warps decides it).  Three groups when the halo fits and there
// are three halo stages (one each), else two.  Returns false when a wait
// timed out.
template <int kB>
__device__ __forceinline__ int halo_groups(const HaloParams& hp) {
  if (hp.nstg != 0 || hp.tma_halo) return 0;
  if (hp.nhs >= 3 && hp.positions <= (kProducers / 6) * kB) return 3;
  if (hp.positions <= (kProducers / 4) * kB) return 2;
  return 0;
}
// Producer arrivals that complete a halo stage (per CTA).
template <int kB>
__device__ __forceinline__ uint32_t halo_arrivals(const HaloParams& hp) {
  const int ng = halo_groups<kB>(hp);
  return ng > 0 ? kProducers / ng : kProducers;
}

template <int kB, bool kUnit = false>
__device__ __forceinline__ bool halo_produce_split(const HaloParams& hp, const TileSched& ts, uint8_t* smem,
                                                  uint64_t* h_full, uint64_t* h_empty, volatile int* abort_flag,
                                                  int pt, int ng) {
  const ConvParams& p = hp.c;
  const int gsize = kProducers / ng;  // threads per group: 96 or 64 (whole warps)
  const uint32_t grp = static_cast<uint32_t>(pt / gsize);
  const int lt = pt - static_cast<int>(grp) * gsize;
  const int step = gsize / 2;  // positions between a thread's loads, two threads per position
  const int h = halo_lane_half(lt);
  const int e_first = halo_lane_pos(lt);
  const int b_first = e_first / hp.CW, pos_first = e_first - b_first * hp.CW;
  const int b_step = step / hp.CW, pos_step = step - b_step * hp.CW;
  const int positions = hp.positions;
  const int HW32 = p.H * p.W * 32;
  const uint32_t nhs = static_cast<uint32_t>(hp.nhs);
  bool skip = (p.debug_flags & 1) && pt == 0;  // test hook: this thread skips its first arrival
  uint32_t i = 0, gi = 0;  // channel blocks of this CTA so far (all groups'); i % ng
  for (StageIter it(hp, ts); it.valid(hp); it.next(hp, ts), ++i, gi = gi + 1 == static_cast<uint32_t>(ng) ? 0u : gi + 1) {
    if (gi != grp) continue;
    const PatchTile t = decode_patch(it.tile, hp, ts);
    const int hb0 = t.p0 * p.stride_h - p.pad_h;
    const int wb0 = t.q0 * p.stride_w - p.pad_w;
    const int8_t* img = p.x + static_cast<int64_t>(t.n) * p.img_stride + it.cb * HW32;
    int e = e_first, b = b_first, pos = pos_first;
    halo_walk_origin(hp, t.m0, b, pos);
    uint4 v[kB];
#pragma unroll
    for (int k = 0; k < kB; ++k) {
      v[k] = make_uint4(0, 0, 0, 0);
      if (e < positions) {  // natural order: pos is the input column
        const int hh = hb0 + b, ww = wb0 + pos;
        v[k] = ptx::ldg16_or_zero(img + (hh * p.W + ww) * 32 + h * 16,
                                  t.valid && hh >= 0 && hh < p.H && ww >= 0 && ww < p.W);
        e += step;
        b += b_step;
        pos += pos_step;
        if (pos >= hp.CW) {
          pos -= hp.CW;
          ++b;
        }
      }
    }
    // channel block i uses halo stage i % nhs for the (i / nhs)-th time
    const uint32_t hs = i % nhs;
    const uint32_t hph = (i / nhs) & 1u;
    // warp-uniform outcome: the arrive below is a warp-wide operation
    if (!__all_sync(0xffffffffu, ptx::mbar_wait(&h_empty[hs], hph ^ 1u, p.timeout_ns, abort_flag))) return false;
    uint8_t* halo = smem + hs * hp.halo_bytes;
    int ps = hp.flat ? 0 : pos_first;  // stride 1 (flat tiles): the phase order is the natural order
#pragma unroll
    for (int k = 0; k < kB; ++k) {
      const int ek = e_first + k * step;
      if constexpr (kUnit) {
        if (ek < positions) halo_store_f16(hp, halo, ek, h, v[k]);
      } else {
        if (ek < positions) halo_store_f16(hp, halo, ek - ps + halo_phase_index(hp, ps), h, v[k]);
        ps += pos_step;
        ps -= ps >= hp.CW ? hp.CW : 0;
      }
    }
    ptx::fence_proxy_async_smem();
    arrive_on_leader(&h_full[hs], ts, !skip);
    skip = false;
  }
  return true;
}

// Which register producer a halo takes: groups taking channel blocks in turn
// when a channel block is one batch of kB loads per thread, else all
// producers on every channel block.
constexpr int kHaloSplitBatch = 4;  // the halo kernel's producers: the most that fits 72 registers

template <int kB, bool kUnit = false>
__device__ __forceinline__ bool halo_produce_registers(const HaloParams& hp, const TileSched& ts, uint8_t* smem,
                                                      uint64_t* h_full, uint64_t* h_empty, volatile int* abort_flag,
                                                      int pt) {
  const int ng = halo_groups<kB>(hp);
  if (ng > 0) return halo_produce_split<kB, kUnit>(hp, ts, smem, h_full, h_empty, abort_flag, pt, ng);
  return hp.positions > 6 * kHaloStep
             ? halo_produce_direct<8, kUnit>(hp, ts, smem, h_full, h_empty, abort_flag, pt)
             : halo_produce_direct<6, kUnit>(hp, ts, smem, h_full, h_empty, abort_flag, pt);
}

// Producer fed by TMA: thread 0 issues, nxs channel blocks ahead, one box
// per channel block into an int8 slot (x_full[slot] counts its bytes); every
// producer thread converts its positions of the slot into the fp16 halo
// stage, arrives on h_full as the register producers do and on
// x_done[slot]; once all have (warp 1 waits for that), thread 0 reuses the
// slot for the next box.  No registers hold loads in flight and the box's
// zero fill takes the place of the bounds checks.  Returns false when a wait
// timed out; boxes still in flight then land before the function returns.
__device__ __forceinline__ bool halo_produce_tma(const HaloParams& hp, const TileSched& ts, uint8_t* smem,
                                                 uint64_t* h_full, uint64_t* h_empty, uint64_t* x_full,
                                                 uint64_t* x_done, const CUtensorMap* tmap_x,
                                                 volatile int* abort_flag, int pt) {
  const ConvParams& p = hp.c;
  const int h = halo_lane_half(pt);
  const int positions = hp.positions;
  const HaloWalk w = halo_walk(hp, pt);
  const uint32_t nxs = static_cast<uint32_t>(hp.nxs);
  // Warp 1 (producer threads 0-31) tracks the next channel block to load --
  // every one of its lanes, so that its warp-wide waits below stay uniform --
  // and its lane 0 issues the boxes.
  StageIter lit(hp, ts);
  uint32_t issued = 0;
  auto issue = [&](uint32_t slot) {  // all lanes of warp 1: the box of channel block `lit` into `slot`
    if (pt == 0) {
      const PatchTile t = decode_patch(lit.tile, hp, ts);
      int c1, c2;
      if (hp.flat) {
        c1 = -p.pad_w;
        c2 = t.m0 / hp.CW - p.pad_h;
      } else {
        c1 = t.q0 * p.stride_w - p.pad_w;
        c2 = t.p0 * p.stride_h - p.pad_h;
      }
      if (!t.valid) c2 = p.H + 256;  // a pair's missing patch: a box wholly outside the image, all zeros
      ptx::mbar_arrive_expect_tx(&x_full[slot], hp.x8_box);
      ptx::tma_load_4d(smem + hp.off_x8 + slot * hp.x8_bytes, tmap_x, &x_full[slot], 0, c1, c2,
                       t.n * p.CB + lit.cb);
    }
    lit.next(hp, ts);
    ++issued;
  };
  if (pt < 32)
    for (uint32_t j = 0; j < nxs && lit.valid(hp); ++j) issue(j);
  bool skip = (p.debug_flags & 1) && pt == 0;  // test hook: this thread skips its first arrival
  uint32_t hs = 0, hph = 0, i = 0;
  bool ok = true;
  for (StageIter it(hp, ts); it.valid(hp); it.next(hp, ts), ++i) {
    const uint32_t slot = i % nxs, xph = (i / nxs) & 1u;
    // warp-uniform outcomes: the arrives below are warp-wide
    if (!__all_sync(0xffffffffu, ptx::mbar_wait(&x_full[slot], xph, p.timeout_ns, abort_flag)) ||
        !__all_sync(0xffffffffu, ptx::mbar_wait(&h_empty[hs], hph ^ 1u, p.timeout_ns, abort_flag))) {
      ok = false;
      break;
    }
    const PatchTile t = decode_patch(it.tile, hp, ts);
    const uint8_t* x8 = smem + hp.off_x8 + slot * hp.x8_bytes;
    uint8_t* halo = smem + hs * hp.halo_bytes;
    // the box in natural order: flat tiles (stride 1) store position e
    // from f0 + e (the run starts f0 positions into the box's first padded
    // row); 2-D patches walk the box's pixels e = row * CW + column and store
    // each at its column-phase position in the row
    const int f0 = hp.flat ? t.m0 - (t.m0 / hp.CW) * hp.CW : 0;
    int pos = w.pos_first;
    for (int e = w.e_first; e < positions; e += kHaloStep) {
      const int src = hp.flat ? f0 + e : e;
      const int dst = hp.flat ? e : e - pos + halo_phase_index(hp, pos);
      halo_store_f16(hp, halo, dst, h, *reinterpret_cast<const uint4*>(x8 + src * 32 + h * 16));
      pos += w.pos_step;
      pos -= pos >= hp.CW ? hp.CW : 0;
    }
    ptx::fence_proxy_async_smem();
    arrive_on_leader(&h_full[hs], ts, !skip);
    skip = false;
    ptx::mbar_arrive(&x_done[slot]);
    hs = hs + 1 == static_cast<uint32_t>(hp.nhs) ? 0u : hs + 1;
    hph ^= hs == 0 ? 1u : 0u;
    if (pt < 32 && lit.valid(hp)) {  // warp 1: the slot is free once every producer has read it
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(&x_done[slot], xph, p.timeout_ns, abort_flag))) {
        ok = false;
        break;
      }
      issue(slot);
      __syncwarp();
    }
  }
  // boxes issued but not consumed (after a timeout) land before the CTA moves on
  if (pt == 0)
    for (uint32_t k = i; k < issued; ++k)
      if (!ptx::mbar_wait(&x_full[k % nxs], (k / nxs) & 1u, p.timeout_ns, nullptr)) break;
  return ok;
}

// GT > 0 fixes the run length (K-slices per filter stage) at compile time so
// that the per-run tap loop is unrolled; GT == 0 reads it from the parameters.
// CG == 2: CTA pairs (clusters of two) issue M = 256 MMAs whose A rows come
// from the two CTAs' patches and whose B columns are split between them, so
// each CTA stages half of every filter tile; rank 0 issues the MMAs, both
// The resident filter straight from the int8 CxRSKx<32> filter into shared
// memory, in the layout the filter TMA would give it: stage st holds K-slices
// st*G .. st*G + G - 1 of the first unit, each BN/CG rows (output channels
// n0 ..) of 32 fp16 channels, 64 bytes per row in the 64-byte swizzle (the
// 16-byte chunk c of row j at chunk c ^ ((j >> 1) & 3) of an 8-row, 512-byte
// atom).  Rows past K and slices past the filter are zeros, as the TMA's
// out-of-bounds fill would make them.  Run by all the CTA's threads before
// the warp roles split, kBatch 16-byte loads in flight per thread; the
// caller's CTA (and cluster) barrier then orders the stores, made visible to
// the tensor core's proxy here, before the first MMA.  (Measured: the same
// work done by the non-producer warps after the split, overlapping the first
// halo loads, made the whole kernel slower.)
template <int BN, int CG>
__device__ __forceinline__ void resident_filter_to_smem(const HaloParams& hp, uint8_t* smem, int G) {
  constexpr int kBatch = 8;
  constexpr int BNH = BN / CG;
  const ConvParams& p = hp.c;
  const TileSched ts = tile_sched<CG>();
  if (ts.first >= hp.num_units) return;  // no unit, no MMA reads these stages
  const WorkUnit wu = decode_unit(ts.first, hp);
  const int n0 = (wu.tile % p.num_n_tiles) * BN + ts.rank * BNH;
  const int kk0 = wu.cb0 * p.R * p.S;
  const int kk_end = p.CB * p.R * p.S;
  const int per_stage = G * BNH * 2;
  const int total = hp.nbs * per_stage;
  if (!hp.filter_ready) ptx::griddep_wait();  // the filter may come from the kernel before this one
  for (int b0 = 0; b0 < total; b0 += kBatch * kHaloThreads) {
    uint4 v[kBatch];
#pragma unroll
    for (int q = 0; q < kBatch; ++q) {
      const int i = b0 + q * kHaloThreads + static_cast<int>(threadIdx.x);
      const int st = i / per_stage, r = i - st * per_stage;
      const int j = (r >> 1) % BNH, t = (r >> 1) / BNH;
      const int kk = kk0 + st * G + t, n = n0 + j;
      const bool live = i < total && kk < kk_end && n < p.K;
      v[q] = ptx::ldg16_or_zero(
          hp.f_src + ((static_cast<int64_t>(live ? kk : 0) * p.K + (live ? n : 0)) * 32 + (r & 1) * 16), live);
    }
#pragma unroll
    for (int q = 0; q < kBatch; ++q) {
      const int i = b0 + q * kHaloThreads + static_cast<int>(threadIdx.x);
      if (i < total) {
        const int st = i / per_stage, r = i - st * per_stage;
        const int j = (r >> 1) % BNH, t = (r >> 1) / BNH, half = r & 1;
        uint8_t* row = smem + hp.off_b + (static_cast<uint32_t>(st * G + t) * BNH + j) * 64;
        const int sw = (j >> 1) & 3;
        uint4 c0, c1;
        i8x4_to_f16x4(v[q].x, c0.x, c0.y);
        i8x4_to_f16x4(v[q].y, c0.z, c0.w);
        i8x4_to_f16x4(v[q].z, c1.x, c1.y);
        i8x4_to_f16x4(v[q].w, c1.z, c1.w);
        *reinterpret_cast<uint4*>(row + (((2 * half) ^ sw) << 4)) = c0;
        *reinterpret_cast<uint4*>(row + (((2 * half + 1) ^ sw) << 4)) = c1;
      }
    }
  }
  ptx::fence_proxy_async_smem();
}

// CTAs produce their own halo and drain their own 128 accumulator rows.
template <int BN, int GT, int CG, int SUB = 1>
__global__ void __launch_bounds__(kHaloThreads, 1)
    conv_fprop_halo_kernel(const __grid_constant__ CUtensorMap tmap_f, const __grid_constant__ CUtensorMap tmap_x,
                           const HaloParams hp) {
  static_assert(CG == 1 || CG == 2, "CTA group");
  // SUB = 2: 16x16 patches (hp.subtiles == 2), issued through the whole-row
  // run block below, with two BN-column accumulators per buffer
  static_assert(SUB == 1 || (SUB == 2 && GT > 0 && BN <= 128), "16x16 patches");
  static_assert(CG == 1 || BN >= 64, "a CTA pair splits B into halves of at least 32 rows");
  const ConvParams& p = hp.c;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + hp.off_bar);
  uint64_t* b_full = bars;
  uint64_t* b_empty = bars + kMaxBStages;
  uint64_t* h_full = bars + 2 * kMaxBStages;
  uint64_t* h_empty = h_full + 3;  // up to three halo stages
  uint64_t* acc_full = h_full + 6;
  uint64_t* acc_empty = h_full + 8;
  uint64_t* drain = h_full + 10;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(h_full + 11);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(h_full + 11) + 1;
  uint64_t* epi_sync = h_full + 12;                                    // the epilogue warps' own barrier
  volatile int* split_last = reinterpret_cast<volatile int*>(h_full + 13);  // this CTA combines a split tile
  uint64_t* fconv_done = h_full + 14;  // this CTA's share of the filter is converted and announced
  volatile uint32_t* fconv_gen = reinterpret_cast<volatile uint32_t*>(h_full + 15);  // grid barrier generation seen
  uint64_t* x_full = h_full + 16;  // TMA-fed halo: int8 slot loaded (up to three slots)
  uint64_t* x_done = h_full + 19;  // TMA-fed halo: int8 slot converted
  uint64_t* h_fwd = h_full + 22;   // a pair's rank 1: its own producers' halo arrivals (up to three stages)

  const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x) >> 5, 0);
  const int lane = threadIdx.x & 31;
  const int nbs = hp.nbs;
  constexpr int BNH = BN / CG;  // filter rows (output channels) this CTA stages per K-slice
  // A dependent launch after this one (the next run) may start as soon as
  // SMs free up: every read of memory an earlier kernel may write (the
  // activations, the filter or its converted copy) and every write of the
  // fp16 copy waits for the earlier grid (griddep_wait); the outputs are
  // written only after those reads.
  if (threadIdx.x == 0) ptx::griddep_launch_dependents();
#if defined(I8C_PIPELINE_TRACE)
  // per-CTA span (global timer) and SM, for the pipeline analysis build only
  if (p.trace != nullptr && threadIdx.x == 0 && blockIdx.x < kTraceSlots) {
    p.trace[8 * kTraceSlots + blockIdx.x] = static_cast<long long>(ptx::globaltimer_ns());
    p.trace[10 * kTraceSlots + blockIdx.x] = static_cast<long long>(ptx::smid());
  }
#endif

  if (threadIdx.x == 0) {
    for (int i = 0; i < nbs; ++i) {
      ptx::mbar_init(&b_full[i], 1);
      ptx::mbar_init(&b_empty[i], 1);
    }
    for (int i = 0; i < hp.nhs; ++i) {
      ptx::mbar_init(&h_full[i], halo_arrivals<kHaloSplitBatch>(hp) * CG);  // a pair's rank 0 counts both CTAs'
      ptx::mbar_init(&h_empty[i], 1);
      if (CG == 2) ptx::mbar_init(&h_fwd[i], halo_arrivals<kHaloSplitBatch>(hp));
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&acc_full[i], 1);
      ptx::mbar_init(&acc_empty[i], kEpilogue * CG);
    }
    ptx::mbar_init(drain, 1);
    ptx::mbar_init(epi_sync, kEpilogue);
    ptx::mbar_init(fconv_done, 1);
    for (int i = 0; i < 3; ++i) {
      ptx::mbar_init(&x_full[i], 1);
      ptx::mbar_init(&x_done[i], kProducers);
    }
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kTmaWarp && lane == 0) ptx::prefetch_tensormap(&tmap_f);
  if (warp == 0) {
    ptx::tmem_alloc_cg<CG>(tmem_slot, p.tmem_cols);
    ptx::tmem_relinquish_cg<CG>();
  }
  if (hp.f_smem) resident_filter_to_smem<BN, CG>(hp, smem, GT > 0 ? GT : hp.bgroup);
  ptx::tc_fence_before();
  __syncthreads();
  if (CG == 2) ptx::cluster_sync();  // the peer's barriers are initialised before any remote arrive
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // a filter written above (both CTAs of a pair, ordered by the barriers just
  // passed) is complete: its stages are announced once, as the TMA would
  if (hp.f_smem && threadIdx.x == 0)
    for (int i = 0; i < nbs; ++i) ptx::mbar_arrive(&b_full[i]);

  if (warp == 0) {
    // ------------------------------------------------------------ MMA issuer
    ptx::setmaxnreg_dec<kWorkerRegs>();
    const TileSched ts = tile_sched<CG>();  // per role: kept live only where used
    if (CG == 1 || ts.rank == 0) {
      // The whole warp runs the loop in uniform control flow so that every
      // descriptor is computed from loop counters and kernel parameters in
      // uniform registers; one elected lane issues each MMA and commit.
      constexpr uint32_t idesc = ptx::idesc_f16_f32(128 * CG, BN);
      constexpr bool kCW = CG == 2;  // barriers with arrivals from the peer CTA: cluster-scope acquire
      constexpr uint16_t kPair = 3;  // commits of a pair signal the barrier in both CTAs
      auto commit_all = [&](uint64_t* bar) {
        if constexpr (CG == 2) ptx::mma_commit_pair(bar, kPair);
        else ptx::mma_commit(bar);
      };
      // 8-row groups of A: sh halo rows apart (2-D patches), 8 positions apart (flat)
      const uint32_t sbo = hp.flat ? 128u : static_cast<uint32_t>(p.stride_h * hp.CW * 16);
      const uint32_t lbo = hp.plane_bytes;
      const uint64_t a_desc0 = ptx::smem_desc_noswizzle_kmajor(0, lbo, sbo);
      const uint64_t b_desc0 = ptx::smem_desc_sw64_kmajor(0);
      constexpr bool wide = SUB == 2;  // 16x16 patches
      // start-address fields (16-byte units)
      const uint32_t h_lo = ptx::smem_addr(smem) >> 4;
      const uint32_t b_lo = ptx::smem_addr(smem + hp.off_b) >> 4;
      const uint32_t halo_lo = hp.halo_bytes >> 4;
      const uint32_t chunk2_lo = (2 * lbo) >> 4;
      const int G = GT > 0 ? GT : hp.bgroup;
      const uint32_t slice_lo = static_cast<uint32_t>(BNH * 64) >> 4;
      const uint32_t stage_lo = static_cast<uint32_t>(G) * slice_lo;
      // tap (r, s) -> halo position r*dh*CW + phase_off(f) + idx with
      // s*dw = idx*sw + f; phase_off(f) = f*(CW/sw) + min(f, CW%sw)
      const int row_step = p.dil_h * hp.CW;
      const int dw_div = p.dil_w / p.stride_w, dw_mod = p.dil_w % p.stride_w;
      const int cw_q = hp.CW / p.stride_w, cw_r = hp.CW % p.stride_w;
      // Runs: a run is one filter stage of G K-slices, G taps of one channel
      // block -- part of a filter row (G divides S) or whole rows (S divides
      // G, G divides R*S) -- so a run never spans two channel blocks.  Its
      // slices are unrolled into MMA pairs whose tap addresses advance with
      // selects.  Waits, releases and accumulator switches happen only at run
      // boundaries (chunk lengths are multiples of G); a barrier wait costs a
      // few hundred cycles even when its phase has completed, so fewer, longer
      // runs keep the tensor core's short instruction queue fed.
      const int runs_per_cb = (p.R * p.S) / G;
      // GT > 0 (the host picks it only when S divides GT): a run is GT / S
      // whole filter rows, and the halo offsets of its taps relative to its
      // first row are the same for every run -- computed once, so a K-slice
      // costs one add on its way to the descriptor.
      int tapoff[GT > 0 ? GT : 1];
      if constexpr (GT > 0) {
#pragma unroll
        for (int t = 0; t < GT; ++t) {
          const int r = t / p.S, sd = (t - r * p.S) * p.dil_w;
          const int f = sd % p.stride_w;
          tapoff[t] = r * row_step + f * cw_q + min(f, cw_r) + sd / p.stride_w;
        }
      }
      const int run_rowstep = GT > 0 ? (G / p.S) * row_step : 0;
      uint32_t u = 0, hst = 0, hph = 0, st = 0, bph = 0, g = 0;  // hst, hph: halo stage and its parity
      // resident filter: the stages are loaded once, during the first
      // first_pass K-slices, and never released
      const bool resident = hp.resident != 0;
      const uint32_t first_pass = static_cast<uint32_t>(nbs * G);
      bool ok = true;
#if defined(I8C_PIPELINE_TRACE)
      const bool tracing = p.trace != nullptr && blockIdx.x == 0;
      long long stall_acc = 0, stall_b = 0, stall_h = 0;
      long long nr_acc = 0, nr_b = 0, nr_h = 0;  // waits that found the phase still open
      int cbseq = 0;
#endif
      auto wwait = [&](uint64_t* bar, uint32_t parity) -> bool {
        return __all_sync(0xffffffffu, ptx::mbar_wait<kCW>(bar, parity, p.timeout_ns, abort_flag));
      };
      trace_mark(p, 0, 0, 0);  // whole warp: no lane-dependent code around the issue loop
      for (int unit = ts.first; ok && unit < hp.num_units; unit += ts.step) {
        const WorkUnit wu = decode_unit(unit, hp);
        const int unit_runs = (wu.cb1 - wu.cb0) * runs_per_cb;
        // a half-width unit: N = BN/2 MMAs on its half of the filter rows and
        // of the accumulator columns
        const bool half_n = CG == 1 && wu.nh >= 0;
        const uint32_t idesc_u = half_n ? ptx::idesc_f16_f32(128, BN / 2) : idesc;
        const uint32_t nh_cols = half_n ? static_cast<uint32_t>(wu.nh) * (BN / 2) : 0u;
        const uint32_t nh_lo = nh_cols * (64 >> 4);  // those filter rows, 64 bytes each, in 16-byte units
        int kk = 0, next_chunk = 0;  // slices of this unit issued; where the next chunk starts
        uint32_t buf = 0, d_tmem = tmem_base + nh_cols;
        uint32_t acc_flag = 0;  // 0 for the first MMA of a chunk, then 1
        // tap state: column count tc within the filter row, row trow within
        // the channel block, the halo offset of the row, column phase and index
        // (GT > 0: only the run within the channel block and its first row)
        int tc = 0, trow = 0, rowpos = 0, fph = 0, idx = 0, rcb = 0;
        for (int run = 0; run < unit_runs; ++run) {
          if (GT > 0 ? rcb == 0 : (tc == 0 && trow == 0)) {  // first run of a channel block: its halo
#if defined(I8C_PIPELINE_TRACE)
            const long long th = tracing ? clock64() : 0;
            nr_h += ptx::mbar_test_wait<kCW>(&h_full[hst], hph) ? 0 : 1;
#endif
            if (!wwait(&h_full[hst], hph)) {
              ok = false;
              break;
            }
#if defined(I8C_PIPELINE_TRACE)
            if (tracing) stall_h += clock64() - th;
            if (tracing && cbseq < kTraceSlots)
              p.trace[20 * kTraceSlots + cbseq] = static_cast<long long>(ptx::globaltimer_ns());
#endif
          }
          if (kk == next_chunk) {
            // a new exact-fp32 chunk: hand the previous accumulator to the
            // epilogue and take the next buffer
            if (kk != 0) {
              if (ptx::elect_one()) commit_all(&acc_full[buf]);
              __syncwarp();
#if defined(I8C_PIPELINE_TRACE)
              trace_mark(p, 0, 2, u);
#endif
              ++u;
            }
            buf = u & 1u;
            const uint32_t aph = (u >> 1) & 1u;
#if defined(I8C_PIPELINE_TRACE)
            const long long ta = tracing ? clock64() : 0;
            nr_acc += ptx::mbar_test_wait<kCW>(&acc_empty[buf], aph ^ 1u) ? 0 : 1;
#endif
            if (!wwait(&acc_empty[buf], aph ^ 1u)) {
              ok = false;
              break;
            }
#if defined(I8C_PIPELINE_TRACE)
            if (tracing) stall_acc += clock64() - ta;
            trace_mark(p, 0, 3, u);
#endif
            d_tmem = tmem_base + buf * BN * static_cast<uint32_t>(SUB) + nh_cols;
            next_chunk = kk + p.chunk_slices;
            acc_flag = 0;
          }
#if defined(I8C_PIPELINE_TRACE)
          const long long tb = tracing ? clock64() : 0;
          if (!resident || g < first_pass) nr_b += ptx::mbar_test_wait<kCW>(&b_full[st], bph) ? 0 : 1;
#endif
          // a resident filter is waited for only on its first pass
          if ((!resident || g < first_pass) && !wwait(&b_full[st], bph)) {
            ok = false;
            break;
          }
#if defined(I8C_PIPELINE_TRACE)
          if (tracing) stall_b += clock64() - tb;
          trace_mark(p, 0, 1, g / G);  // filter stage acquired
#endif
          ptx::tc_fence_after();
          const uint32_t h_stage = h_lo + hst * halo_lo;
          uint32_t b_cur = b_lo + st * stage_lo;
          // Narrow tiles (short MMAs): the stage's descriptors are computed by
          // the whole warp first and one elected lane issues all its MMAs and
          // the release in one block (measured 17% faster at BN = 64; at
          // BN = 256 the per-slice form is 2% faster).
          constexpr bool kOneBlock = GT > 0 && BN <= 128;
          if constexpr (kOneBlock) {
            uint64_t adv0[kOneBlock ? GT : 1], adv1[kOneBlock ? GT : 1], bdv[kOneBlock ? GT : 1];
#pragma unroll
            for (int t = 0; t < GT; ++t) {
              const uint32_t a_c = h_stage + static_cast<uint32_t>(rowpos + tapoff[t]);
              adv0[t] = a_desc0 | static_cast<uint64_t>(a_c & 0x3FFFu);
              adv1[t] = a_desc0 | static_cast<uint64_t>((a_c + chunk2_lo) & 0x3FFFu);
              bdv[t] = b_desc0 | static_cast<uint64_t>((b_cur + nh_lo + t * slice_lo) & 0x3FFFu);
            }
            if (ptx::elect_one()) {
#pragma unroll
              for (int t = 0; t < GT; ++t) {
                if constexpr (CG == 2) {
                  ptx::mma_f16_ss_pair(d_tmem, adv0[t], bdv[t], idesc, t == 0 ? acc_flag : 1u);
                  ptx::mma_f16_ss_pair(d_tmem, adv1[t], bdv[t] + 2, idesc, 1u);
                } else {
                  ptx::mma_f16_ss(d_tmem, adv0[t], bdv[t], idesc_u, t == 0 ? acc_flag : 1u);
                  ptx::mma_f16_ss(d_tmem, adv1[t], bdv[t] + 2, idesc_u, 1u);
                }
              }
              if constexpr (wide) {
                // the second 16x8 sub-tile: its 8-column groups start 8 halo
                // positions on (128 bytes, 8 in the 16-byte address field)
#pragma unroll
                for (int t = 0; t < GT; ++t) {
                  if constexpr (CG == 2) {
                    ptx::mma_f16_ss_pair(d_tmem + BN, adv0[t] + 8, bdv[t], idesc, t == 0 ? acc_flag : 1u);
                    ptx::mma_f16_ss_pair(d_tmem + BN, adv1[t] + 8, bdv[t] + 2, idesc, 1u);
                  } else {
                    ptx::mma_f16_ss(d_tmem + BN, adv0[t] + 8, bdv[t], idesc_u, t == 0 ? acc_flag : 1u);
                    ptx::mma_f16_ss(d_tmem + BN, adv1[t] + 8, bdv[t] + 2, idesc_u, 1u);
                  }
                }
              }
              if (!resident) commit_all(&b_empty[st]);
            }
            __syncwarp();
            acc_flag = 1;
          }
#pragma unroll
          for (int t = 0; t < (kOneBlock ? 0 : G); ++t) {
            const uint32_t a_cur =
                GT > 0 ? h_stage + static_cast<uint32_t>(rowpos + tapoff[GT > 0 ? t : 0])
                       : h_stage + static_cast<uint32_t>(rowpos + fph * cw_q + min(fph, cw_r) + idx);
            const uint64_t ad0 = a_desc0 | static_cast<uint64_t>(a_cur & 0x3FFFu);
            const uint64_t ad1 = a_desc0 | static_cast<uint64_t>((a_cur + chunk2_lo) & 0x3FFFu);
            const uint64_t bd = b_desc0 | static_cast<uint64_t>((b_cur + nh_lo) & 0x3FFFu);
            if (ptx::elect_one()) {
              if constexpr (CG == 2) {
                ptx::mma_f16_ss_pair(d_tmem, ad0, bd, idesc, acc_flag);
                ptx::mma_f16_ss_pair(d_tmem, ad1, bd + 2, idesc, 1u);
              } else {
                ptx::mma_f16_ss(d_tmem, ad0, bd, idesc_u, acc_flag);
                ptx::mma_f16_ss(d_tmem, ad1, bd + 2, idesc_u, 1u);
              }
            }
            __syncwarp();
            acc_flag = 1;
            b_cur += slice_lo;
            if constexpr (GT > 0) continue;
            // next tap: column s + 1 of the row (s*dw = idx*sw + fph), or the
            // first column of the next row, or of the first row after the
            // channel block's last tap
            fph += dw_mod;
            const int carry = fph >= p.stride_w ? 1 : 0;
            fph -= carry * p.stride_w;
            idx += dw_div + carry;
            ++tc;
            const bool row_end = tc == p.S;
            tc = row_end ? 0 : tc;
            fph = row_end ? 0 : fph;
            idx = row_end ? 0 : idx;
            rowpos += row_end ? row_step : 0;
            trow += row_end ? 1 : 0;
            const bool cb_end = trow == p.R;
            trow = cb_end ? 0 : trow;
            rowpos = cb_end ? 0 : rowpos;
          }
          if constexpr (!kOneBlock) {
            if (!resident && ptx::elect_one()) commit_all(&b_empty[st]);
            __syncwarp();
          }
#if defined(I8C_PIPELINE_TRACE)
          trace_mark(p, 1, 2, g / G);  // filter stage released (commit issued)
#endif
          st = st + 1 == static_cast<uint32_t>(nbs) ? 0u : st + 1;
          bph ^= st == 0 ? 1u : 0u;
          kk += G;
          g += G;
          bool cb_done = tc == 0 && trow == 0;
          if constexpr (GT > 0) {
            rowpos += run_rowstep;
            cb_done = ++rcb == runs_per_cb;
            rcb = cb_done ? 0 : rcb;
            rowpos = cb_done ? 0 : rowpos;
          }
          if (cb_done) {  // channel block done: release its halo
            if (ptx::elect_one()) commit_all(&h_empty[hst]);
            __syncwarp();
#if defined(I8C_PIPELINE_TRACE)
            if (tracing && cbseq < kTraceSlots)
              p.trace[21 * kTraceSlots + cbseq] = static_cast<long long>(ptx::globaltimer_ns());
            ++cbseq;
#endif
            hst = hst + 1 == static_cast<uint32_t>(hp.nhs) ? 0u : hst + 1;
            hph ^= hst == 0 ? 1u : 0u;
          }
        }
        if (!ok) break;
        if (ptx::elect_one()) commit_all(&acc_full[buf]);
        __syncwarp();
        ++u;
      }
      trace_mark(p, 0, 0, 1);
      if (p.trace != nullptr && blockIdx.x == 0) {
        p.trace[4 * kTraceSlots] = g;
#if defined(I8C_PIPELINE_TRACE)
        p.trace[4 * kTraceSlots + 1] = stall_acc;
        p.trace[4 * kTraceSlots + 2] = stall_b;
        p.trace[4 * kTraceSlots + 3] = stall_h;
        p.trace[4 * kTraceSlots + 4] = nr_acc;
        p.trace[4 * kTraceSlots + 5] = nr_b;
        p.trace[4 * kTraceSlots + 6] = nr_h;
#endif
      }
      if (!ok && lane == 0) raise_timeout(p, abort_flag);
      // every MMA issued by this warp has completed before TMEM is freed
      // (a pair's rank 1 learns it through the final cluster barrier)
      if (ptx::elect_one()) {
        if constexpr (CG == 2) ptx::mma_commit_pair(drain, 1);
        else ptx::mma_commit(drain);
      }
      __syncwarp();
      if (!ptx::mbar_wait(drain, 0, p.timeout_ns, nullptr) && lane == 0) raise_timeout(p, abort_flag);
    } else if constexpr (CG == 2) {
      // A pair's rank 1: forward each completed fill of its own halo stages
      // as one arrival (all of its producers' count) on rank 0's barrier.
      // The producers' stores are ordered before it by their release on the
      // local barrier and this lane's acquire of it; rank 0's MMAs read them
      // after acquiring its barrier.  It never runs two fills ahead: a stage
      // is refilled only after the MMAs have consumed the forwarded fill.
      const uint32_t n = halo_arrivals<kHaloSplitBatch>(hp);
      uint32_t hs = 0, hph = 0;
      bool fine = true;
      for (StageIter it(hp, ts); it.valid(hp); it.next(hp, ts)) {
        fine = __all_sync(0xffffffffu, ptx::mbar_wait(&h_fwd[hs], hph, p.timeout_ns, abort_flag));
        if (!fine) break;
        if (lane == 0) ptx::mbar_arrive_remote(ptx::mapa(ptx::smem_addr(&h_full[hs]), 0), n);
        __syncwarp();
        hs = hs + 1 == static_cast<uint32_t>(hp.nhs) ? 0u : hs + 1;
        hph ^= hs == 0 ? 1u : 0u;
      }
      if (!fine && lane == 0) raise_timeout(p, abort_flag);
    }
  } else if (warp == kTmaWarp) {
    // ------------------------------------------------------------ filter TMA producer
    ptx::setmaxnreg_dec<kWorkerRegs>();
    if (hp.f_int8 != nullptr) {
      // the filter is converted inside this launch: wait until every CTA's
      // share is written (grid barrier), then let TMA read it
      bool fine = __all_sync(0xffffffffu, ptx::mbar_wait(fconv_done, 0, p.timeout_ns, abort_flag));
      if (fine) {
        const uint32_t seen = *fconv_gen;
        const uint64_t t0 = ptx::globaltimer_ns();
        while (ptx::ld_acquire_gpu(hp.gbar + 1) == seen) {
          if (ptx::globaltimer_ns() - t0 > p.timeout_ns || *abort_flag) {
            fine = false;
            break;
          }
          __nanosleep(64);
        }
        fine = __all_sync(0xffffffffu, fine);
      }
      ptx::fence_proxy_async_global();
      if (!fine && lane == 0) raise_timeout(p, abort_flag);
    } else if (!hp.filter_ready) {
      // the fp16 filter is written by the conversion kernel launched just
      // before this one, which this kernel may overlap (dependent launch)
      ptx::griddep_wait();
    }
    const TileSched ts = tile_sched<CG>();
    const int G = GT > 0 ? GT : hp.bgroup;
    const uint32_t stage_bytes = static_cast<uint32_t>(G * BNH * 64);
    uint32_t g = 0, st = 0, bph = 0;
    bool ok = true;
    const int RS = p.R * p.S;
    // (nothing to load when the epilogue warps write the filter)
    for (int unit = ts.first; ok && !hp.f_smem && unit < hp.num_units; unit += ts.step) {
      if (hp.resident && unit != ts.first) break;  // every unit reuses the first unit's stages
      const WorkUnit wu = decode_unit(unit, hp);
      const int n0 = (wu.tile % p.num_n_tiles) * BN + ts.rank * BNH;
      for (int kk = wu.cb0 * RS; kk < wu.cb1 * RS; kk += G, ++g) {
        if (!__all_sync(0xffffffffu, ptx::mbar_wait(&b_empty[st], bph ^ 1u, p.timeout_ns, abort_flag))) {
          ok = false;
          break;
        }
#if defined(I8C_PIPELINE_TRACE)
        trace_mark(p, 1, 3, g);  // slot free
#endif
        // G consecutive K-slices; slices past the end of the filter read as
        // zeros.  A pair's two halves both complete on rank 0's barrier.
        if (ptx::elect_one()) {
          uint8_t* dst = smem + hp.off_b + st * stage_bytes;
          if constexpr (CG == 1) {
            ptx::mbar_arrive_expect_tx(&b_full[st], stage_bytes);
            ptx::tma_load_3d(dst, &tmap_f, &b_full[st], 0, n0, kk);
          } else if (ts.rank == 0) {
            ptx::mbar_arrive_expect_tx(&b_full[st], 2 * stage_bytes);
            ptx::tma_load_3d_pair(dst, &tmap_f, ptx::smem_addr(&b_full[st]), 0, n0, kk);
          } else {
            ptx::tma_load_3d_pair(dst, &tmap_f, ptx::mapa(ptx::smem_addr(&b_full[st]), 0), 0, n0, kk);
          }
        }
        __syncwarp();
#if defined(I8C_PIPELINE_TRACE)
        trace_mark(p, 1, 1, g);  // load issued
#endif
        if (++st == static_cast<uint32_t>(nbs)) {
          st = 0;
          bph ^= 1u;
        }
      }
    }
    if (!ok && lane == 0) raise_timeout(p, abort_flag);
    // wait for the loads still in flight (at most one per stage); rank 0 of a
    // pair waits for both CTAs' halves, which rank 1 cannot observe
    const uint32_t first = g > static_cast<uint32_t>(nbs) ? g - nbs : 0u;
    for (uint32_t i = (CG == 2 && ts.rank != 0) ? g : first; i < g; ++i) {
      if (!ptx::mbar_wait<CG == 2>(&b_full[i % nbs], (i / nbs) & 1u, p.timeout_ns, nullptr)) {
        if (lane == 0) raise_timeout(p, abort_flag);
        break;
      }
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ halo producers
    // Thread pt owns the 16-byte half halo_lane_half(pt) of halo positions
    // e = halo_lane_pos(pt) + k*(kProducers/2), k = 0, 1, ...  Two ways to bring a channel
    // block in, chosen by the plan: through an int8 staging ring that
    // cp.async fills nstg-1 channel blocks ahead (deep prefetch, costs
    // shared memory), or straight into registers in batches whose first one
    // is in flight while the thread waits for the halo stage (no staging
    // memory, which leaves room for longer filter stages).  Either way the
    // bytes are converted to fp16 and stored into the free halo stage.
    ptx::setmaxnreg_dec<kWorkerRegs>();
    ptx::griddep_wait();  // the activations may come from the kernel before this one
    const int pt = (warp < kTmaWarp ? warp - 1 : warp - 2) * 32 + lane;
    TileSched ts = tile_sched<CG>();
    // a pair's rank 1 arrives on its own barriers (warp 0 forwards them):
    // its producer warps do not wait for a cluster-scope release
    uint64_t* hf = h_full;
    if (CG == 2 && ts.rank == 1) {
      ts.fwd = 1;
      hf = h_fwd;
    }
    const bool ok = hp.tma_halo ? halo_produce_tma(hp, ts, smem, hf, h_empty, x_full, x_done, &tmap_x,
                                                   abort_flag, pt)
                    : hp.nstg > 0 ? halo_produce_staged(hp, ts, smem, hf, h_empty, abort_flag, pt)
                                  : halo_produce_registers<kHaloSplitBatch>(hp, ts, smem, hf, h_empty,
                                                                             abort_flag, pt);
    if (!ok) raise_timeout(p, abort_flag);
  } else if (warp >= 8) {
    // ------------------------------------------------------------ epilogue
    // The int32 running sums of a tile live in these warps' registers (the two
    // epilogue warpgroups raise their register budget), so tensor memory only
    // holds two fp32 chunk accumulators and a drain is one read of the
    // accumulator that overlaps the MMAs of the next chunk.
    ptx::setmaxnreg_inc<kEpilogueRegs>();
    if (hp.f_int8 != nullptr) {
      ptx::griddep_wait();  // the kernel before this one may still read the fp16 copy
      // this CTA's share of the int8 -> f16 filter copy (same layout), then
      // one arrival per CTA on the grid barrier; the generation it saw goes to
      // the TMA warp
      const int64_t per = (hp.f_vecs + gridDim.x - 1) / gridDim.x;
      const int64_t v0 = per * blockIdx.x;
      const int64_t v1 = v0 + per < hp.f_vecs ? v0 + per : hp.f_vecs;
      const uint4* src = reinterpret_cast<const uint4*>(hp.f_int8);
      uint4* dst = reinterpret_cast<uint4*>(hp.f16);
      for (int64_t i = v0 + (threadIdx.x - 8 * 32); i < v1; i += kEpilogue) {
        const uint4 v = __ldg(src + i);
        uint4 c0, c1;
        i8x4_to_f16x4(v.x, c0.x, c0.y);
        i8x4_to_f16x4(v.y, c0.z, c0.w);
        i8x4_to_f16x4(v.z, c1.x, c1.y);
        i8x4_to_f16x4(v.w, c1.z, c1.w);
        dst[2 * i] = c0;
        dst[2 * i + 1] = c1;
      }
      ptx::fence_proxy_async_global();
      __threadfence();
      ptx::mbar_arrive(epi_sync);
      const bool all_done = ptx::mbar_wait(epi_sync, 0, p.timeout_ns, abort_flag);
      if (threadIdx.x == 8 * 32 && all_done) {
        const uint32_t gen = *reinterpret_cast<volatile uint32_t*>(hp.gbar + 1);
        __threadfence();
        if (atomicAdd(hp.gbar, 1u) == gridDim.x - 1) {
          // last arrival: reset the count for the next launch, open the barrier
          atomicExch(hp.gbar, 0u);
          __threadfence();
          atomicAdd(hp.gbar + 1, 1u);
        }
        *fconv_gen = gen;
        ptx::mbar_arrive(fconv_done);
      }
      if (!__all_sync(0xffffffffu, all_done) && lane == 0) raise_timeout(p, abort_flag);
    }
    const int qd = warp & 3;
    const int row = 32 * qd + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(32 * qd) << 16;
    // columns of this warp: half `eh` of the tile (all of it when BN == 32, for warps 8-11)
    const int eh = (warp - 8) >> 2;
    constexpr int kColsPerWarp = BN >= 64 ? BN / 2 : BN;
    const int col0 = BN >= 64 ? eh * kColsPerWarp : 0;
    const bool col_owner = BN >= 64 || eh == 0;
    // 16x16 patches: this thread's pixel in each 16x8 sub-tile
    constexpr int kSub = SUB;
    constexpr int sub = SUB;
    uint32_t run[kSub * kColsPerWarp];  // running int32 sums of this thread's pixel(s) over its columns
    uint32_t u = 0, esync = hp.f_int8 != nullptr ? 1u : 0u;  // epi_sync phases used so far
    bool ok = true;
    const int RS = p.R * p.S;
    // all epilogue threads meet (bounded wait: a warp that gave up cannot hang the others)
    auto epi_barrier = [&]() -> bool {
      ptx::mbar_arrive(epi_sync);
      const bool met = ptx::mbar_wait(epi_sync, esync & 1u, p.timeout_ns, abort_flag);
      ++esync;
      return __all_sync(0xffffffffu, met);
    };
    for (int unit = tile_sched<CG>().first; ok && unit < hp.num_units; unit += tile_sched<CG>().step) {
      const WorkUnit wu = decode_unit(unit, hp);
      const int nch = ((wu.cb1 - wu.cb0) * RS + p.chunk_slices - 1) / p.chunk_slices;
      // a half-width unit's columns belong to one column half of the warps
      const bool mine = col_owner && (wu.nh < 0 || wu.nh == eh);
      for (int c = 0; c < nch; ++c, ++u) {
        const uint32_t buf = u & 1u;
#if defined(I8C_PIPELINE_TRACE)
        if (warp == 8 && lane == 0) trace_mark(p, 3, 0, u);
#endif
        const bool got = ptx::mbar_wait(&acc_full[buf], (u >> 1) & 1u, p.timeout_ns, abort_flag);
#if defined(I8C_PIPELINE_TRACE)
        if (warp == 8 && lane == 0) trace_mark(p, 3, 1, u);
#endif
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t t_acc = tmem_base + lane_addr + buf * BN * static_cast<uint32_t>(sub) + col0;
        const bool first = c == 0;
        if (mine) {
#pragma unroll
          for (int sb = 0; sb < kSub; ++sb) {
            if (sb >= sub) break;
#pragma unroll
            for (int g = 0; g < kColsPerWarp / 32; ++g) {
              uint32_t v[32];
              ptx::tmem_ld_32x32b_x32(t_acc + sb * BN + g * 32, v);
              ptx::tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                const uint32_t a = static_cast<uint32_t>(__float2int_rn(__uint_as_float(v[i])));
                const int j = sb * kColsPerWarp + g * 32 + i;
                run[j] = first ? a : run[j] + a;
              }
            }
          }
        }
        // the accumulator buffer is free once read (a pair's rank 0 waits for both CTAs)
        ptx::tc_fence_before();
        arrive_on_leader(&acc_empty[buf], tile_sched<CG>());
#if defined(I8C_PIPELINE_TRACE)
        if (warp == 8 && lane == 0) trace_mark(p, 3, 2, u);
#endif
        if (c + 1 < nch) continue;
        if (wu.part >= 0) {
          // A split tile: publish this unit's partial sums; the unit that
          // arrives last adds the others' and stores the tile.
          const int tail = wu.tile - hp.full_units;
          const int rank = tile_sched<CG>().rank;
          constexpr size_t kBlock = static_cast<size_t>(128) * BN;  // int32 per (tile, part, rank)
          int32_t* const blocks = hp.split_part + static_cast<size_t>(tail) * hp.ksplit * CG * kBlock;
          if (col_owner) {
            int4* mine = reinterpret_cast<int4*>(blocks + (static_cast<size_t>(wu.part) * CG + rank) * kBlock);
#pragma unroll
            for (int q = 0; q < kColsPerWarp / 4; ++q)
              __stcg(mine + (col0 / 4 + q) * 128 + row,
                     make_int4(static_cast<int>(run[4 * q]), static_cast<int>(run[4 * q + 1]),
                               static_cast<int>(run[4 * q + 2]), static_cast<int>(run[4 * q + 3])));
          }
          __threadfence();
          if (!epi_barrier()) {
            ok = false;
            break;
          }
          if (threadIdx.x == 8 * 32) {
            int* cnt = hp.split_count + tail * CG + rank;
            const int before = atomicAdd(cnt, 1);
            const bool last = before == hp.ksplit - 1;
            if (last) *cnt = 0;  // every part has arrived: ready for the next launch
            __threadfence();
            *split_last = last ? 1 : 0;
          }
          if (!epi_barrier()) {
            ok = false;
            break;
          }
          if (*split_last == 0) continue;
          __threadfence();
          if (col_owner) {
            for (int part = 0; part < hp.ksplit; ++part) {
              if (part == wu.part) continue;
              const int4* other =
                  reinterpret_cast<const int4*>(blocks + (static_cast<size_t>(part) * CG + rank) * kBlock);
#pragma unroll
              for (int q = 0; q < kColsPerWarp / 4; ++q) {
                const int4 v = __ldcg(other + (col0 / 4 + q) * 128 + row);
                run[4 * q] += static_cast<uint32_t>(v.x);
                run[4 * q + 1] += static_cast<uint32_t>(v.y);
                run[4 * q + 2] += static_cast<uint32_t>(v.z);
                run[4 * q + 3] += static_cast<uint32_t>(v.w);
              }
            }
          }
        }
        if (!mine) continue;
        const PatchTile t = decode_patch(wu.tile, hp, tile_sched<CG>());
        const int pp = hp.flat ? (t.m0 + row) / hp.CW : t.p0 + (row >> 3);
        const int qq0 = hp.flat ? (t.m0 + row) - pp * hp.CW : t.q0 + (row & 7);
#pragma unroll
        for (int sb = 0; sb < kSub; ++sb) {
          if (sb >= sub) break;
          const int qq = qq0 + 8 * sb;  // the sub-tile's column (2-D patches only)
          if (!(t.valid && pp < p.P && qq < p.Q)) continue;
#pragma unroll
          for (int g = 0; g < kColsPerWarp / 32; ++g) {
            const int k0 = t.nt * BN + col0 + g * 32;
            const int j0 = sb * kColsPerWarp + g * 32;
            if (k0 < p.K) {
              const int64_t off = ((static_cast<int64_t>(t.n) * p.KB + (k0 >> 5)) * p.P + pp) * p.Q + qq;
              if (p.out_mode == 0) {
                uint32_t o[8];
                requant32(p, k0, [&](int i) { return static_cast<int>(run[j0 + i]); }, o);
                uint4* dst = reinterpret_cast<uint4*>(p.y + off * 32);
                dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
                dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
              } else {
                uint4* dst = reinterpret_cast<uint4*>(p.acc + off * 32);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                  dst[i] = make_uint4(run[j0 + 4 * i], run[j0 + 4 * i + 1], run[j0 + 4 * i + 2], run[j0 + 4 * i + 3]);
              }
            }
          }
        }
      }
    }
    if (!ok) raise_timeout(p, abort_flag);
  }

  ptx::tc_fence_before();
  __syncthreads();
  // A pair's CTAs leave together: no remote arrive, multicast commit or MMA
  // operand read targets a CTA that has exited, and both free their tensor
  // memory together.
  if (CG == 2) ptx::cluster_sync();
#if defined(I8C_PIPELINE_TRACE)
  if (p.trace != nullptr && threadIdx.x == 0 && blockIdx.x < kTraceSlots)
    p.trace[9 * kTraceSlots + blockIdx.x] = static_cast<long long>(ptx::globaltimer_ns());
#endif
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_cg<CG>(tmem_base, p.tmem_cols);
  }
}

}  // namespace i8c
