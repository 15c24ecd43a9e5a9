// INT8 NCxHWx<32> Conv2d fprop on the sm_103a tensor cores, transposed tiles.
//
// The same implicit GEMM as the other kernels (rows N*P*Q output pixels,
// columns K output channels, reduction C*R*S), computed as its transpose:
// the MMA's M = 128 rows are 128 output channels, drawn from the fp16 filter
// by TMA, and its N columns are tile_px output pixels (a multiple of 16, up
// to 256), drawn from a halo of the input.  Stride-1 layers only: the pixels
// of a tile are tile_px consecutive positions of the output laid out
// row-major with the zero-padded input's row width CW (the CW - Q positions
// past the end of each output row are computed and discarded), so the B
// operand of filter tap (r, s) is the contiguous run of halo positions that
// starts r*dh*CW + s*dw positions in -- eight consecutive pixels are one
// 128-byte core matrix of the no-swizzle K-major layout.
//
// Why the transpose: the filter (the large operand per K-slice) now fills
// only the 128-row side, so a filter stage of a whole 3x3 channel block
// (9 K-slices, 72 KB) fits twice beside the halo and the MMA warp waits once
// per channel block instead of once per filter row; and the tile's pixel
// count is free, so the plan can pick the width whose tile count fills the
// SMs' waves best.
//
// CTA pairs (CG = 2, clusters of two): M = 256 MMAs whose rows are 128
// output channels from each CTA's own filter stage and whose N pixel columns
// are split in halves, each CTA building the halo of its half -- half the
// halo production per tensor-core cycle of a single CTA.  Rank 0 issues; both
// drain their own 128 channels over all N columns.
//
// Warp roles (512 threads) as in the halo kernel: warp 0 MMA issuer and TMEM
// owner, warp 4 filter TMA, warps 1-3 and 5-7 halo producers, warps 8-15
// epilogue.  TMEM lane i of the accumulator is output channel 128*kt + i, so
// a warp's 32 lanes are one 32-channel block of the output and a column (one
// pixel) is one 32-byte NCxHWx<32> vector: the epilogue writes it with one
// coalesced warp store, no transpose.  All waits are bounded.
#pragma once

#include "conv_fprop_halo.cuh"

namespace i8c {

constexpr int kTrRows = 128;   // output channels per tile: the MMA's M
constexpr int kTrMaxPx = 256;  // output pixels per tile: the MMA's N, at most

// Register split by the widest MMA N an instantiation serves: MAXPX = 192
// leaves an epilogue thread 96 running sums, so its warps need fewer
// registers and the producer warps get enough for batches of eight loads;
// MAXPX = 256 keeps the halo kernel's split and batches of four.
template <int MAXPX>
struct TrRegs {
  static constexpr uint32_t kWorker = MAXPX <= 192 ? 104 : kWorkerRegs;
  static constexpr uint32_t kEpi = MAXPX <= 192 ? 152 : kEpilogueRegs;
  static constexpr int kBatch = MAXPX <= 192 ? 8 : kHaloSplitBatch;
  static_assert(128 * (2 * kWorker + 2 * kEpi) <= 512 * 128, "register split");
};

// GT > 0: filter stages of GT K-slices that are whole filter rows (S divides
// GT), their taps' halo offsets precomputed and all their MMAs issued by one
// elected lane in one block; GT == 0: any stage length, taps advanced slice
// by slice.  MAXPX: the widest MMA N (CG * tile_px) the instantiation
// serves.  CG: CTAs per MMA tile (1, or 2 for pairs).
template <int GT, int MAXPX, int CG>
__global__ void __launch_bounds__(kHaloThreads, 1)
    conv_fprop_tr_kernel(const __grid_constant__ CUtensorMap tmap_f, const __grid_constant__ CUtensorMap tmap_x,
                         const HaloParams hp) {
  static_assert(CG == 1 || CG == 2, "CTA group");
  using Regs = TrRegs<MAXPX>;
  constexpr int kMaxGroupsPerWarp = MAXPX / 16;  // 8-column groups of one epilogue warp
  const ConvParams& p = hp.c;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + hp.off_bar);
  uint64_t* b_full = bars;
  uint64_t* b_empty = bars + kMaxBStages;
  uint64_t* h_full = bars + 2 * kMaxBStages;
  uint64_t* h_empty = h_full + 3;
  uint64_t* acc_full = h_full + 6;
  uint64_t* acc_empty = h_full + 8;
  uint64_t* drain = h_full + 10;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(h_full + 11);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(h_full + 11) + 1;
  uint64_t* x_full = h_full + 16;  // TMA-fed halo: int8 slot loaded (up to three slots)
  uint64_t* x_done = h_full + 19;  // TMA-fed halo: int8 slot converted

  const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x) >> 5, 0);
  const int lane = threadIdx.x & 31;
  // the next run may launch as soon as SMs free up; every read of memory an
  // earlier kernel may write waits for it (griddep_wait in the producers and
  // the filter TMA warp), and the outputs are written only after those reads
  if (threadIdx.x == 0) ptx::griddep_launch_dependents();
  const int nbs = hp.nbs;
  const int NP = CG * hp.tile_px;  // the MMA's N: pixels per tile over the CTA group
  const int RS = p.R * p.S;
  const int G = GT > 0 ? GT : hp.bgroup;  // K-slices (taps of one channel block) per filter stage
#if defined(I8C_PIPELINE_TRACE)
  // per-CTA span (global timer), for the pipeline analysis build only
  if (p.trace != nullptr && threadIdx.x == 0 && blockIdx.x < kTraceSlots)
    p.trace[8 * kTraceSlots + blockIdx.x] = static_cast<long long>(ptx::globaltimer_ns());
#endif

  if (threadIdx.x == 0) {
    for (int i = 0; i < nbs; ++i) {
      ptx::mbar_init(&b_full[i], 1);
      ptx::mbar_init(&b_empty[i], 1);
    }
    for (int i = 0; i < hp.nhs; ++i) {
      ptx::mbar_init(&h_full[i], halo_arrivals<Regs::kBatch>(hp) * CG);  // rank 0 counts both CTAs'
      ptx::mbar_init(&h_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&acc_full[i], 1);
      ptx::mbar_init(&acc_empty[i], kEpilogue * CG);
    }
    ptx::mbar_init(drain, 1);
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
  ptx::tc_fence_before();
  __syncthreads();
  if (CG == 2) ptx::cluster_sync();  // the peer's barriers are initialised before any remote arrive
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ MMA issuer
    ptx::setmaxnreg_dec<Regs::kWorker>();
    const TileSched ts = tile_sched<CG>();
    if (CG == 1 || ts.rank == 0) {
    // The whole warp runs the loop in uniform control flow; one elected lane
    // issues each MMA and commit (measured no slower than lane 0 alone).
    const uint32_t idesc = ptx::idesc_f16_f32(kTrRows * CG, NP);
    const uint64_t f_desc0 = ptx::smem_desc_sw64_kmajor(0);
    // the halo as B: 8-pixel groups 128 bytes apart, 8-channel planes plane_bytes apart
    const uint64_t h_desc0 = ptx::smem_desc_noswizzle_kmajor(0, hp.plane_bytes, 128);
    const uint32_t h_lo = ptx::smem_addr(smem) >> 4;  // start-address fields, 16-byte units
    const uint32_t f_lo = ptx::smem_addr(smem + hp.off_b) >> 4;
    const uint32_t halo_lo = hp.halo_bytes >> 4;
    const uint32_t chunk2_lo = (2 * hp.plane_bytes) >> 4;  // channels 16-31: planes 2 and 3
    constexpr uint32_t slice_lo = (kTrRows * 64) >> 4;     // one K-slice of the filter stage
    const uint32_t stage_lo = static_cast<uint32_t>(G) * slice_lo;
    const int row_step = p.dil_h * hp.CW;  // halo positions between filter rows
    const int stages_per_cb = RS / G;
    const uint32_t buf_cols = p.tmem_cols / 2;  // accumulator 1 starts at a power-of-two column
    // GT > 0: halo offsets of a stage's taps relative to its first filter row
    int tapoff[GT > 0 ? GT : 1];
    if constexpr (GT > 0) {
#pragma unroll
      for (int t = 0; t < GT; ++t) {
        const int r = t / p.S;
        tapoff[t] = r * row_step + (t - r * p.S) * p.dil_w;
      }
    }
    const int stage_rowstep = GT > 0 ? (GT / p.S) * row_step : 0;
    uint32_t u = 0, hst = 0, hph = 0, st = 0, bph = 0;
    bool ok = true;
    // barriers with arrivals from the peer CTA: cluster-scope acquire
    auto wwait = [&](uint64_t* bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, ptx::mbar_wait<CG == 2>(bar, parity, p.timeout_ns, abort_flag));
    };
    // one elected lane's tcgen05 issue (MMAs or a commit)
    auto issue = [&](auto&& f) {
      if (ptx::elect_one()) f();
      __syncwarp();
    };
    // a pair's MMAs and commits: both CTAs' accumulators and barriers
    auto mma = [&](uint32_t d, uint64_t a, uint64_t b, uint32_t accumulate) {
      if constexpr (CG == 2) ptx::mma_f16_ss_pair(d, a, b, idesc, accumulate);
      else ptx::mma_f16_ss(d, a, b, idesc, accumulate);
    };
    auto commit = [&](uint64_t* bar) {
      if constexpr (CG == 2) ptx::mma_commit_pair(bar, 3);
      else ptx::mma_commit(bar);
    };
#if defined(I8C_PIPELINE_TRACE)
    // CTA 0: cycles spent in each kind of wait and in the MMA issue blocks
    const bool tracing = p.trace != nullptr && blockIdx.x == 0;
    long long stall_acc = 0, stall_b = 0, stall_h = 0, t_issue = 0, t_first = 0, t_post = 0, t_end = 0;
    long long stall_h_first = 0;  // halo waits during the CTA's first tile
    uint32_t slices = 0;
    if (tracing) t_first = clock64();
    if (p.trace != nullptr && lane == 0 && blockIdx.x < kTraceSlots)
      p.trace[24 * kTraceSlots + blockIdx.x] = static_cast<long long>(ptx::globaltimer_ns());
#endif
    for (int unit = ts.first; ok && unit < hp.num_units; unit += ts.step) {
      const int unit_stages = p.CB * stages_per_cb;
      int kk = 0, next_chunk = 0;  // K-slices issued; where the next exact-fp32 chunk starts
      uint32_t buf = 0, d_tmem = tmem_base;
      uint32_t acc_flag = 0;  // 0 for the first MMA of a chunk
      // tap state within the channel block: filter column, halo offset (positions)
      int sc = 0, tcol = 0, toff = 0;
      for (int stg = 0; stg < unit_stages; ++stg) {
#if defined(I8C_PIPELINE_TRACE)
        const long long th = tracing ? clock64() : 0;
        if (tracing && t_end != 0) t_post += th - t_end;
#endif
        if (sc == 0 && !wwait(&h_full[hst], hph)) {  // first stage of a channel block: its halo
          ok = false;
          break;
        }
#if defined(I8C_PIPELINE_TRACE)
        if (tracing) stall_h += clock64() - th;
        if (tracing && unit == ts.first) stall_h_first += clock64() - th;
#endif
        if (kk == next_chunk) {
          if (kk != 0) {
            issue([&] { commit(&acc_full[buf]); });
#if defined(I8C_PIPELINE_TRACE)
            if (tracing && lane == 0) trace_mark(p, 0, 2, u);
#endif
            ++u;
          }
          buf = u & 1u;
#if defined(I8C_PIPELINE_TRACE)
          const long long ta = tracing ? clock64() : 0;
#endif
          if (!wwait(&acc_empty[buf], ((u >> 1) & 1u) ^ 1u)) {
            ok = false;
            break;
          }
#if defined(I8C_PIPELINE_TRACE)
          if (tracing) stall_acc += clock64() - ta;
          if (tracing && lane == 0) trace_mark(p, 0, 3, u);
#endif
          d_tmem = tmem_base + buf * buf_cols;
          next_chunk = kk + p.chunk_slices;
          acc_flag = 0;
        }
#if defined(I8C_PIPELINE_TRACE)
        const long long tb = tracing ? clock64() : 0;
#endif
        if (!wwait(&b_full[st], bph)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
#if defined(I8C_PIPELINE_TRACE)
        const long long ti = tracing ? clock64() : 0;
        if (tracing) stall_b += ti - tb;
#endif
        const uint32_t h_stage = h_lo + hst * halo_lo;
        uint32_t f_cur = f_lo + st * stage_lo;
        if constexpr (GT > 0) {
          // descriptors of the stage's first tap; the others differ only in
          // their start-address fields (no carry: shared addresses stay below
          // 2^18 bytes)
          const uint64_t hd_base = h_desc0 | static_cast<uint64_t>((h_stage + static_cast<uint32_t>(toff)) & 0x3FFFu);
          const uint64_t fd_base = f_desc0 | static_cast<uint64_t>(f_cur & 0x3FFFu);
          // the stage's MMAs, the filter stage's release and, when the stage
          // ends a channel block, the halo's release in one elected block
          const bool cb_last = sc + 1 == stages_per_cb;
          issue([&] {
#pragma unroll
            for (int t = 0; t < GT; ++t) {
              const uint64_t hd = hd_base + static_cast<uint64_t>(tapoff[t]);
              const uint64_t fd = fd_base + static_cast<uint64_t>(t * slice_lo);
              mma(d_tmem, fd, hd, t == 0 ? acc_flag : 1u);
              mma(d_tmem, fd + 2, hd + chunk2_lo, 1u);
            }
            commit(&b_empty[st]);
            if (cb_last) commit(&h_empty[hst]);
          });
          acc_flag = 1;
          toff += stage_rowstep;
        }
        for (int t = 0; t < (GT > 0 ? 0 : G); ++t) {
          const uint32_t b_cur = h_stage + static_cast<uint32_t>(toff);
          const uint64_t fd = f_desc0 | static_cast<uint64_t>(f_cur & 0x3FFFu);
          const uint64_t hd0 = h_desc0 | static_cast<uint64_t>(b_cur & 0x3FFFu);
          const uint64_t hd1 = h_desc0 | static_cast<uint64_t>((b_cur + chunk2_lo) & 0x3FFFu);
          issue([&] {
            mma(d_tmem, fd, hd0, acc_flag);
            mma(d_tmem, fd + 2, hd1, 1u);  // filter channels 16-31: 32 bytes on
          });
          acc_flag = 1;
          f_cur += slice_lo;
          // next tap: the next filter column, or the first of the next row
          ++tcol;
          toff += p.dil_w;
          const bool row_end = tcol == p.S;
          tcol = row_end ? 0 : tcol;
          toff += row_end ? row_step - p.S * p.dil_w : 0;
        }
        if constexpr (GT == 0) issue([&] { commit(&b_empty[st]); });
#if defined(I8C_PIPELINE_TRACE)
        if (tracing) t_end = clock64();
        if (tracing) t_issue += t_end - ti;
        slices += G;
#endif
        st = st + 1 == static_cast<uint32_t>(nbs) ? 0u : st + 1;
        bph ^= st == 0 ? 1u : 0u;
        kk += G;
        if (++sc == stages_per_cb) {  // channel block done: release its halo
          sc = 0;
          tcol = 0;
          toff = 0;
          if constexpr (GT == 0) issue([&] { commit(&h_empty[hst]); });  // GT > 0: released above
          hst = hst + 1 == static_cast<uint32_t>(hp.nhs) ? 0u : hst + 1;
          hph ^= hst == 0 ? 1u : 0u;
        }
      }
      if (!ok) break;
      issue([&] { commit(&acc_full[buf]); });
#if defined(I8C_PIPELINE_TRACE)
      if (tracing && lane == 0) trace_mark(p, 0, 2, u);
#endif
      ++u;
    }
#if defined(I8C_PIPELINE_TRACE)
    if (p.trace != nullptr && lane == 0 && blockIdx.x < kTraceSlots)
      p.trace[25 * kTraceSlots + blockIdx.x] = static_cast<long long>(ptx::globaltimer_ns());
    if (tracing && lane == 0) {
      p.trace[0] = t_first;
      p.trace[1] = clock64();
      p.trace[4 * kTraceSlots] = slices;
      p.trace[4 * kTraceSlots + 1] = stall_acc;
      p.trace[4 * kTraceSlots + 2] = stall_b;
      p.trace[4 * kTraceSlots + 3] = stall_h;
      p.trace[4 * kTraceSlots + 7] = t_issue;
      p.trace[4 * kTraceSlots + 8] = t_post;
      p.trace[4 * kTraceSlots + 9] = stall_h_first;
    }
#endif
    if (!ok && lane == 0) raise_timeout(p, abort_flag);
    // every MMA issued by this warp has completed before TMEM is freed (a
    // pair's rank 1 learns it through the final cluster barrier)
    issue([&] {
      if constexpr (CG == 2) ptx::mma_commit_pair(drain, 1);
      else ptx::mma_commit(drain);
    });
    if (!ptx::mbar_wait(drain, 0, p.timeout_ns, nullptr) && lane == 0) raise_timeout(p, abort_flag);
    }  // rank 0
  } else if (warp == kTmaWarp) {
    // ------------------------------------------------------------ filter TMA producer
    ptx::setmaxnreg_dec<Regs::kWorker>();
    // the fp16 filter is written by the conversion kernel launched just
    // before this one, which this kernel may overlap (dependent launch)
    if (!hp.filter_ready) ptx::griddep_wait();
    const TileSched ts = tile_sched<CG>();
    const uint32_t stage_bytes = static_cast<uint32_t>(G * kTrRows * 64);
    uint32_t g = 0, st = 0, bph = 0;
    bool ok = true;
    for (int unit = ts.first; ok && unit < hp.num_units; unit += ts.step) {
      // first output channel of this CTA's 128 rows of the tile
      const int k0 = (unit % p.num_n_tiles) * (kTrRows * CG) + ts.rank * kTrRows;
      for (int kk = 0; kk < p.CB * RS; kk += G, ++g) {
        if (!__all_sync(0xffffffffu, ptx::mbar_wait(&b_empty[st], bph ^ 1u, p.timeout_ns, abort_flag))) {
          ok = false;
          break;
        }
        // G consecutive K-slices of 128 output channels; channels past K read as
        // zeros.  A pair's two stages both complete on rank 0's barrier.
        if (ptx::elect_one()) {
          uint8_t* dst = smem + hp.off_b + st * stage_bytes;
          if constexpr (CG == 1) {
            ptx::mbar_arrive_expect_tx(&b_full[st], stage_bytes);
            ptx::tma_load_3d(dst, &tmap_f, &b_full[st], 0, k0, kk);
          } else if (ts.rank == 0) {
            ptx::mbar_arrive_expect_tx(&b_full[st], 2 * stage_bytes);
            ptx::tma_load_3d_pair(dst, &tmap_f, ptx::smem_addr(&b_full[st]), 0, k0, kk);
          } else {
            ptx::tma_load_3d_pair(dst, &tmap_f, ptx::mapa(ptx::smem_addr(&b_full[st]), 0), 0, k0, kk);
          }
        }
        __syncwarp();
        if (++st == static_cast<uint32_t>(nbs)) {
          st = 0;
          bph ^= 1u;
        }
      }
    }
    if (!ok && lane == 0) raise_timeout(p, abort_flag);
    // wait for the loads still in flight (at most one per stage); rank 0 of a
    // pair waits for both CTAs' stages, which rank 1 cannot observe
    const uint32_t first = g > static_cast<uint32_t>(nbs) ? g - nbs : 0u;
    for (uint32_t i = (CG == 2 && ts.rank != 0) ? g : first; i < g; ++i) {
      if (!ptx::mbar_wait<CG == 2>(&b_full[i % nbs], (i / nbs) & 1u, p.timeout_ns, nullptr)) {
        if (lane == 0) raise_timeout(p, abort_flag);
        break;
      }
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ halo producers
    // The contiguous run of padded input positions the tile's taps read, per
    // 32-channel block, loaded into registers (or through the int8 staging
    // ring), converted to fp16 and stored as four 8-channel planes: the same
    // producers as the halo kernel's flat tiles, with tile_px pixels per tile.
    ptx::setmaxnreg_dec<Regs::kWorker>();
    ptx::griddep_wait();  // the activations may come from the kernel before this one
    const int pt = (warp < kTmaWarp ? warp - 1 : warp - 2) * 32 + lane;
    const TileSched ts = tile_sched<CG>();
    const bool ok = hp.tma_halo ? halo_produce_tma(hp, ts, smem, h_full, h_empty, x_full, x_done, &tmap_x,
                                                   abort_flag, pt)
                    : hp.nstg > 0 ? halo_produce_staged(hp, ts, smem, h_full, h_empty, abort_flag, pt)
                                  : halo_produce_registers<Regs::kBatch, true>(hp, ts, smem, h_full, h_empty,
                                                                               abort_flag, pt);
    if (!ok) raise_timeout(p, abort_flag);
  } else {
    // ------------------------------------------------------------ epilogue
    // Warp 8 + 4*eh + qd reads TMEM lanes 32*qd .. 32*qd + 31 (output
    // channel block 4*(CG*kt + rank) + qd of the tile) and column half eh;
    // its lane l keeps the int32 running sums of channel 32*qd + l over that
    // half's pixels in registers.  In a pair the column halves are the two
    // CTAs' pixel halves, i.e. two flat tiles of tile_px pixels.
    ptx::setmaxnreg_inc<Regs::kEpi>();
    const int qd = warp & 3;
    const uint32_t lane_addr = static_cast<uint32_t>(32 * qd) << 16;
    const int eh = (warp - 8) >> 2;
    const int gh = NP / 16;  // 8-column groups per warp half
    const int c0 = eh * gh * 8;  // first column of this warp
    const int nch = (p.CB * RS + p.chunk_slices - 1) / p.chunk_slices;
    uint32_t run[kMaxGroupsPerWarp * 8];
    uint32_t u = 0;
    bool ok = true;
    for (int unit = tile_sched<CG>().first; ok && unit < hp.num_units; unit += tile_sched<CG>().step) {
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
        const uint32_t t_acc = tmem_base + lane_addr + buf * (p.tmem_cols / 2) + static_cast<uint32_t>(c0);
        const bool first = c == 0;
#pragma unroll
        for (int q = 0; q < kMaxGroupsPerWarp / 4; ++q) {
          if (4 * q >= gh) break;
          uint32_t v[4][8];
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (4 * q + j < gh) ptx::tmem_ld_32x32b_x8(t_acc + (4 * q + j) * 8, v[j]);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if (4 * q + j >= gh) continue;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              // exact: every chunk sum is an integer below 2^24 in magnitude
              const uint32_t a = static_cast<uint32_t>(__float2int_rn(__uint_as_float(v[j][i])));
              const int r = (4 * q + j) * 8 + i;
              run[r] = first ? a : run[r] + a;
            }
          }
        }
        // the accumulator buffer is free once read (a pair's rank 0 waits for both CTAs)
        ptx::tc_fence_before();
        arrive_on_leader(&acc_empty[buf], tile_sched<CG>());
#if defined(I8C_PIPELINE_TRACE)
        if (warp == 8 && lane == 0) trace_mark(p, 3, 2, u);
        if (warp == 15 && lane == 0) trace_mark(p, 3, 3, u);
#endif
      }
      if (!ok) break;
      // Store: column j is the pixel at flat position m0 + j of the padded
      // row-major output, and this warp holds its 32 channels of output
      // block cbk -- one contiguous 32-byte NCxHWx<32> vector per pixel.
      const TileSched ts = tile_sched<CG>();
      // the flat tile of these columns: in a pair, column half eh is the
      // pixel half (tile) of CTA eh; a single CTA's halves split one tile
      const PatchTile t = decode_patch(unit, hp, TileSched{ts.first, ts.step, CG == 2 ? eh : 0, CG});
      const int coff = CG == 2 ? 0 : c0;  // this warp's first column within its flat tile
      const int cbk = t.nt * (4 * CG) + ts.rank * 4 + qd;
      if (!t.valid || cbk >= p.KB) continue;
      const int64_t plane = (static_cast<int64_t>(t.n) * p.KB + cbk) * p.P;
      const int ncols = gh * 8;
      if (p.out_mode == 0) {
        // The requantised bytes go to this warp's staging rows (32 bytes per
        // pixel; the 32 lanes of one column fill one row), and a short rolled
        // loop copies the rows out with 16-byte stores.  Kept compact: the
        // per-column code runs once per tile, and fully unrolled stores with
        // their address arithmetic would not stay in the instruction cache.
        uint8_t* wbuf = smem + hp.off_out + (warp - 8) * (NP * 16);
        // this lane's output channel: its scale and bias (or the scalar alpha and 0)
        const int kch = cbk * 32 + lane;
        const float scale = p.alpha_k != nullptr ? __ldg(p.alpha_k + kch) : p.alpha;
        const float bias = p.bias_k != nullptr ? __ldg(p.bias_k + kch) : 0.0f;
        const int lo = p.relu ? 0 : INT_MIN;
#pragma unroll
        for (int g = 0; g < kMaxGroupsPerWarp; ++g) {
          if (g >= gh) break;
#pragma unroll
          for (int i = 0; i < 8; ++i)
            wbuf[(g * 8 + i) * 32 + lane] =
                static_cast<uint8_t>(sat_s8(requant_ch(static_cast<int>(run[g * 8 + i]), scale, bias, lo)));
        }
        __syncwarp();
        for (int e = lane; e < 2 * ncols; e += 32) {
          const int col = e >> 1;
          const int m = t.m0 + coff + col;
          const int pp = m / hp.CW;
          const int qq = m - pp * hp.CW;
          if (pp < p.P && qq < p.Q) {
            const uint4 v = *reinterpret_cast<const uint4*>(wbuf + col * 32 + (e & 1) * 16);
            *reinterpret_cast<uint4*>(p.y + ((plane + pp) * p.Q + qq) * 32 + (e & 1) * 16) = v;
          }
        }
        __syncwarp();  // the rows are rewritten for the next tile
      } else {
        // int32 accumulators (parity checks): one coalesced 128-byte warp
        // store per pixel
        const int m = t.m0 + coff;
        int pp = m / hp.CW;
        int qq = m - pp * hp.CW;
#pragma unroll
        for (int g = 0; g < kMaxGroupsPerWarp; ++g) {
          if (g >= gh) break;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if (pp < p.P && qq < p.Q) p.acc[((plane + pp) * p.Q + qq) * 32 + lane] = static_cast<int32_t>(run[g * 8 + i]);
            if (++qq == hp.CW) {
              qq = 0;
              ++pp;
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
