// INT8 NCxHWx<32> Conv2d fprop on the sm_103a tensor cores for layers with
// 64 output channels: two filter taps per MMA.
//
// With K = 64 output channels the halo kernel's MMAs are N = 64 wide, and an
// N = 64 MMA is bound by its operand reads rather than by its arithmetic: the
// tensor core reads the 128-pixel A tile (4 KB per 16 channels) from shared
// memory for only 64 columns of work.  This kernel gives every A read 128
// columns instead, by stacking the filters of two taps of the same filter row
// side by side on the MMA's N: columns 0-63 are tap s, columns 64-127 tap
// s + 1, both multiplied by the A view of tap s.  Column block 0 is then tap
// s's contribution to output pixel m; column block 1 is tap (s + 1)'s
// contribution to output pixel m - dw (its input lies dw positions further
// along the row), so the epilogue adds column block 1 shifted by dw rows
// (TMEM lanes) onto column block 0.  An odd last tap of a row takes an
// N = 64 MMA into column block 0 alone.
//
// Tiles are 128 consecutive output columns of one output row; since the
// shifted block needs dw lanes beyond a tile's last valid pixel, a tile
// yields vq = 128 - dw valid outputs and tiles start vq columns apart.  The
// halo of a tile and 32-channel block is one segment of L = 128 + (S-1)*dw
// consecutive input columns per filter row (R segments), so the A view of tap
// (r, s) starts r*L + s*dw positions in.
//
// CTA pairs (clusters of two): M = 256 MMAs whose rows are the two CTAs'
// tiles (each CTA its own tile and halo); B's 128 columns are split between
// the CTAs: rank 0 holds the even taps' 64 filter rows, rank 1 the odd taps'
// (for an odd last tap, rank 0 its channels 0-31 and rank 1 its channels
// 32-63, for the N = 64 MMA).  The plan writes the fp16 filter in that
// order ([32-channel block][filter row][rank][slot][64 rows][32 channels]),
// one filter stage per filter row and rank, kept resident when all stages
// fit.
//
// Exactness: a column accumulates at most ceil(S/2) taps x 32 channels per
// filter row, so chunks of at most 32 / ceil(S/2) filter rows keep every
// fp32 partial sum below 2^24 in magnitude (every product is at most 2^14).
//
// Warp roles (512 threads) as in the halo kernel: warp 0 MMA issuer (rank 0)
// and TMEM owner, warp 4 filter TMA, warps 1-3 and 5-7 halo producers, warps
// 8-15 epilogue (warp 8 + 4*eh + qd: TMEM lane quarter qd, output channels
// 32*eh .. 32*eh + 31).  All waits are bounded.
#pragma once

#include "conv_fprop_halo.cuh"

namespace i8c {

constexpr int kStackMaxSlots = 8;    // tap pairs per filter row: S <= 16
constexpr int kStackMaxShift = 8;    // dw: the shift of column block 1, in TMEM lanes
constexpr int kStackSlotBytes = 64 * 64;  // one tap's 64 fp16 filter rows of 32 channels

struct RowTile {
  int n, p, q0;
  bool valid;
};

// Tile t of the row tiling: image n, output row p, first column q0.
__device__ __forceinline__ RowTile decode_row_tile(int t, const HaloParams& hp) {
  if (t >= hp.num_patches) return {0, 0, 0, false};
  const int per_img = hp.c.P * hp.tq;
  const int n = t / per_img;
  const int rem = t - n * per_img;
  const int pp = rem / hp.tq;
  return {n, pp, (rem - pp * hp.tq) * hp.vq, true};
}

// Halo producer: segment r of a tile is input row p + r*dh - pad_h, columns
// q0 - pad_w .. q0 - pad_w + L - 1 (zeros outside the image); thread pt owns
// the 16-byte half halo_lane_half(pt) of positions halo_lane_pos(pt) + k*96.  Loads go straight
// into registers, kB at a time; the first batch is in flight while the thread
// waits for the halo stage to be free.  Returns false when a wait timed out.
template <int kB>
__device__ __forceinline__ bool stack_produce(const HaloParams& hp, const TileSched& ts, uint8_t* smem,
                                              uint64_t* h_full, uint64_t* h_empty, volatile int* abort_flag, int pt) {
  const ConvParams& p = hp.c;
  const int h = halo_lane_half(pt);
  const int positions = hp.positions;
  const int L = hp.seg_len;
  const int HW32 = p.H * p.W * 32;
  uint32_t hs = 0, hph = 0;
  bool skip = (p.debug_flags & 1) && pt == 0;  // test hook: this thread skips its first arrival
  uint32_t tix = 0;                             // trace index: channel blocks so far
  for (int unit = ts.first; unit < hp.num_units; unit += ts.step) {
    const RowTile t = decode_row_tile(2 * unit + ts.rank, hp);
    for (int cb = 0; cb < p.CB; ++cb) {
      const int8_t* img = p.x + static_cast<int64_t>(t.n) * p.img_stride + cb * HW32;
      uint8_t* halo = smem + hs * hp.halo_bytes;
      int e = halo_lane_pos(pt), r = 0, o = e;  // position, its segment and offset (96 < L)
      bool stage_free = false;
      do {
        uint4 v[kB];
        const int e0 = e;
#pragma unroll
        for (int k = 0; k < kB; ++k) {
          v[k] = make_uint4(0, 0, 0, 0);
          if (e < positions) {
            const int hh = t.p + r * p.dil_h - p.pad_h, ww = t.q0 + o - p.pad_w;
            v[k] = ptx::ldg16_or_zero(img + (hh * p.W + ww) * 32 + h * 16,
                                      t.valid && hh >= 0 && hh < p.H && ww >= 0 && ww < p.W);
            e += kProducers / 2;
            o += kProducers / 2;
            if (o >= L) {
              o -= L;
              ++r;
            }
          }
        }
        if (!stage_free) {
          if (pt == 0) trace_mark(p, 2, 0, tix);
          // the warp is converged here (every lane runs the first batch); the
          // arrive below is warp-wide, so the outcome is made warp-uniform
          if (!__all_sync(0xffffffffu, ptx::mbar_wait(&h_empty[hs], hph ^ 1u, p.timeout_ns, abort_flag)))
            return false;
          stage_free = true;
          if (pt == 0) trace_mark(p, 2, 1, tix);
        }
#pragma unroll
        for (int k = 0; k < kB; ++k)
          if (e0 + k * (kProducers / 2) < positions) halo_store_f16(hp, halo, e0 + k * (kProducers / 2), h, v[k]);
      } while (e < positions);
      ptx::fence_proxy_async_smem();
      arrive_on_leader(&h_full[hs], ts, !skip);
      if (pt == 0) trace_mark(p, 2, 2, tix);
      ++tix;
      skip = false;
      hs = hs + 1 == static_cast<uint32_t>(hp.nhs) ? 0u : hs + 1;
      hph ^= hs == 0 ? 1u : 0u;
    }
  }
  return true;
}

// SLOTS = ceil(S/2): the MMAs per filter row and 16-channel half, fixed at
// compile time so that a row's descriptors are computed by the whole warp in
// uniform registers before one elected lane issues them back to back.
template <int SLOTS>
__global__ void __launch_bounds__(kHaloThreads, 1)
    conv_fprop_stack_kernel(const __grid_constant__ CUtensorMap tmap_f, const __grid_constant__ CUtensorMap tmap_x,
                            const HaloParams hp) {
  static_assert(SLOTS >= 1 && SLOTS <= kStackMaxSlots, "tap pairs per filter row");
  constexpr int CG = 2;
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
  uint64_t* epi_sync = h_full + 12;  // the epilogue warps' own barrier

  const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x) >> 5, 0);
  const int lane = threadIdx.x & 31;
  // the next run may launch as soon as SMs free up; every read of memory an
  // earlier kernel may write waits for it (griddep_wait in the producers and
  // the filter TMA warp), and the outputs are written only after those reads
  if (threadIdx.x == 0) ptx::griddep_launch_dependents();
  const int nbs = hp.nbs;
  constexpr int U = SLOTS;              // MMAs per filter row and 16-channel half
  const bool odd = (p.S & 1) != 0;      // the last slot is a single tap (N = 64)
  const int row_stages = p.CB * p.R;    // filter stages (rows) per tile
  const int chunk_rows = p.chunk_slices;  // filter rows per exact fp32 chunk

  if (threadIdx.x == 0) {
    for (int i = 0; i < nbs; ++i) {
      ptx::mbar_init(&b_full[i], 1);
      ptx::mbar_init(&b_empty[i], 1);
    }
    for (int i = 0; i < hp.nhs; ++i) {
      ptx::mbar_init(&h_full[i], kProducers * CG);  // rank 0 counts both CTAs' producers
      ptx::mbar_init(&h_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&acc_full[i], 1);
      ptx::mbar_init(&acc_empty[i], kEpilogue * CG);
    }
    ptx::mbar_init(drain, 1);
    ptx::mbar_init(epi_sync, kEpilogue);
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
  ptx::cluster_sync();  // the peer's barriers are initialised before any remote arrive
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ MMA issuer
    ptx::setmaxnreg_dec<kWorkerRegs>();
    const TileSched ts = tile_sched<CG>();
    if (ts.rank == 0) {
      const uint32_t idesc_pair = ptx::idesc_f16_f32(256, 128);  // two taps x 64 channels
      const uint32_t idesc_single = ptx::idesc_f16_f32(256, 64);
      // A: the halo view, 8-pixel groups 128 bytes apart, 8-channel planes plane_bytes apart
      const uint64_t a_desc0 = ptx::smem_desc_noswizzle_kmajor(0, hp.plane_bytes, 128);
      const uint64_t b_desc0 = ptx::smem_desc_sw64_kmajor(0);
      // start-address fields, in 16-byte units (one halo position is 16 bytes)
      const uint32_t h_lo = ptx::smem_addr(smem) >> 4;
      const uint32_t b_lo = ptx::smem_addr(smem + hp.off_b) >> 4;
      const uint32_t halo_lo = hp.halo_bytes >> 4;
      const uint32_t half_lo = (2 * hp.plane_bytes) >> 4;          // channels 16-31: planes 2 and 3
      const uint32_t seg_lo = static_cast<uint32_t>(hp.seg_len);   // one filter row's segment
      const uint32_t pair_lo = static_cast<uint32_t>(2 * p.dil_w); // the next tap pair's view
      constexpr uint32_t slot_lo = kStackSlotBytes >> 4;
      const uint32_t stage_lo = static_cast<uint32_t>(U) * slot_lo;
      const bool resident = hp.resident != 0;
      uint32_t u = 0, hst = 0, hph = 0, st = 0, bph = 0, g = 0;
      bool ok = true;
      auto wwait = [&](uint64_t* bar, uint32_t parity) -> bool {
        return __all_sync(0xffffffffu, ptx::mbar_wait<true>(bar, parity, p.timeout_ns, abort_flag));
      };
      uint32_t tix = 0;  // tiles of this CTA so far (trace index)
      for (int unit = ts.first; ok && unit < hp.num_units; unit += ts.step, ++tix) {
        uint32_t buf = 0, d_tmem = tmem_base, acc_flag = 0;
        int sidx = 0;  // filter row stage of this tile
        for (int cb = 0; ok && cb < p.CB; ++cb) {
          if (cb == 0) trace_mark(p, 0, 0, tix);
          if (!wwait(&h_full[hst], hph)) {
            ok = false;
            break;
          }
          if (cb == 0) trace_mark(p, 0, 1, tix);
          for (int r = 0; r < p.R; ++r, ++sidx) {
            if (sidx % chunk_rows == 0) {
              // a new exact-fp32 chunk: hand the previous accumulator over, take the next buffer
              if (sidx != 0) {
                if (ptx::elect_one()) ptx::mma_commit_pair(&acc_full[buf], 3);
                __syncwarp();
                ++u;
              }
              buf = u & 1u;
              if (!wwait(&acc_empty[buf], ((u >> 1) & 1u) ^ 1u)) {
                ok = false;
                break;
              }
              d_tmem = tmem_base + buf * 128;
              acc_flag = 0;
              if (sidx == 0) trace_mark(p, 0, 2, tix);
            }
            // a resident filter is waited for only on its first pass
            if ((!resident || g < static_cast<uint32_t>(nbs)) && !wwait(&b_full[st], bph)) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            const uint32_t a_row = h_lo + hst * halo_lo + static_cast<uint32_t>(r) * seg_lo;
            const uint32_t b_row = b_lo + st * stage_lo;
            // the row's descriptors, by the whole warp (no carry out of the
            // start-address fields: shared addresses stay below 2^18 bytes)
            uint64_t adv[2][U], bdv[2][U];
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
              for (int s2 = 0; s2 < U; ++s2) {
                adv[hf][s2] = a_desc0 | static_cast<uint64_t>((a_row + s2 * pair_lo + hf * half_lo) & 0x3FFFu);
                bdv[hf][s2] = b_desc0 | static_cast<uint64_t>((b_row + s2 * slot_lo + hf * 2) & 0x3FFFu);
              }
            }
            if (ptx::elect_one()) {
#pragma unroll
              for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
                for (int s2 = 0; s2 < U; ++s2)
                  ptx::mma_f16_ss_pair(d_tmem, adv[hf][s2], bdv[hf][s2],
                                       odd && s2 == U - 1 ? idesc_single : idesc_pair,
                                       hf == 0 && s2 == 0 ? acc_flag : 1u);
              }
              if (!resident) ptx::mma_commit_pair(&b_empty[st], 3);
            }
            __syncwarp();
            acc_flag = 1;
            st = st + 1 == static_cast<uint32_t>(nbs) ? 0u : st + 1;
            bph ^= st == 0 ? 1u : 0u;
            ++g;
          }
          if (!ok) break;
          // channel block done: release its halo (both CTAs' stages)
          if (ptx::elect_one()) ptx::mma_commit_pair(&h_empty[hst], 3);
          __syncwarp();
          hst = hst + 1 == static_cast<uint32_t>(hp.nhs) ? 0u : hst + 1;
          hph ^= hst == 0 ? 1u : 0u;
        }
        if (!ok) break;
        if (ptx::elect_one()) ptx::mma_commit_pair(&acc_full[buf], 3);
        __syncwarp();
        trace_mark(p, 0, 3, tix);
        ++u;
      }
      if (!ok && lane == 0) raise_timeout(p, abort_flag);
      // every MMA issued has completed before TMEM is freed (rank 1 learns it
      // through the final cluster barrier)
      if (ptx::elect_one()) ptx::mma_commit_pair(drain, 1);
      __syncwarp();
      if (!ptx::mbar_wait(drain, 0, p.timeout_ns, nullptr) && lane == 0) raise_timeout(p, abort_flag);
    }
  } else if (warp == kTmaWarp) {
    // ------------------------------------------------------------ filter TMA producer
    ptx::setmaxnreg_dec<kWorkerRegs>();
    // the fp16 filter is written by the conversion kernel launched just
    // before this one, which this kernel may overlap (dependent launch)
    if (!hp.filter_ready) ptx::griddep_wait();
    const TileSched ts = tile_sched<CG>();
    const uint32_t stage_bytes = static_cast<uint32_t>(U * kStackSlotBytes);
    uint32_t g = 0, st = 0, bph = 0;
    bool ok = true;
    for (int unit = ts.first; ok && unit < hp.num_units; unit += ts.step) {
      if (hp.resident && unit != ts.first) break;  // every unit reuses the first unit's stages
      for (int sidx = 0; sidx < row_stages; ++sidx, ++g) {
        if (!__all_sync(0xffffffffu, ptx::mbar_wait(&b_empty[st], bph ^ 1u, p.timeout_ns, abort_flag))) {
          ok = false;
          break;
        }
        // this rank's U slots of filter row sidx (channel block sidx / R);
        // both CTAs' loads complete on rank 0's barrier
        if (ptx::elect_one()) {
          uint8_t* dst = smem + hp.off_b + st * stage_bytes;
          const int slot0 = (sidx * 2 + ts.rank) * U;
          if (ts.rank == 0) {
            ptx::mbar_arrive_expect_tx(&b_full[st], 2 * stage_bytes);
            ptx::tma_load_3d_pair(dst, &tmap_f, ptx::smem_addr(&b_full[st]), 0, 0, slot0);
          } else {
            ptx::tma_load_3d_pair(dst, &tmap_f, ptx::mapa(ptx::smem_addr(&b_full[st]), 0), 0, 0, slot0);
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
    // wait for the loads still in flight (at most one per stage); rank 0 waits
    // for both CTAs' halves, which rank 1 cannot observe
    const uint32_t first = g > static_cast<uint32_t>(nbs) ? g - nbs : 0u;
    for (uint32_t i = ts.rank != 0 ? g : first; i < g; ++i) {
      if (!ptx::mbar_wait<true>(&b_full[i % nbs], (i / nbs) & 1u, p.timeout_ns, nullptr)) {
        if (lane == 0) raise_timeout(p, abort_flag);
        break;
      }
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ halo producers
    ptx::setmaxnreg_dec<kWorkerRegs>();
    ptx::griddep_wait();  // the activations may come from the kernel before this one
    const int pt = (warp < kTmaWarp ? warp - 1 : warp - 2) * 32 + lane;
    if (!stack_produce<kHaloSplitBatch + 2>(hp, tile_sched<CG>(), smem, h_full, h_empty, abort_flag, pt))
      raise_timeout(p, abort_flag);
  } else {
    // ------------------------------------------------------------ epilogue
    // Warp 8 + 4*eh + qd holds, for the 32 pixels of TMEM lane quarter qd and
    // output channels 32*eh .. 32*eh + 31, the int32 running sums of column
    // block 0 (run0: taps whose view is the pixel's own) and of column block 1
    // (run1: the second tap of each pair, whose contribution belongs dw
    // pixels earlier).
    ptx::setmaxnreg_inc<kEpilogueRegs>();
    const int qd = warp & 3;
    const int eh = (warp - 8) >> 2;
    const uint32_t lane_addr = static_cast<uint32_t>(32 * qd) << 16;
    const int dw = p.dil_w;
    const int nch = (row_stages + chunk_rows - 1) / chunk_rows;
    uint32_t run0[32], run1[32];
    uint32_t u = 0, esync = 0, tl = 0;
    bool ok = true;
    auto epi_barrier = [&]() -> bool {
      ptx::mbar_arrive(epi_sync);
      const bool met = ptx::mbar_wait(epi_sync, esync & 1u, p.timeout_ns, abort_flag);
      ++esync;
      return __all_sync(0xffffffffu, met);
    };
    const TileSched ts = tile_sched<CG>();
    for (int unit = ts.first; ok && unit < hp.num_units; unit += ts.step, ++tl) {
      const bool tr = warp == 8 && lane == 0;
      for (int c = 0; c < nch; ++c, ++u) {
        const uint32_t buf = u & 1u;
        if (!__all_sync(0xffffffffu, ptx::mbar_wait(&acc_full[buf], (u >> 1) & 1u, p.timeout_ns, abort_flag))) {
          ok = false;
          break;
        }
        if (tr && c == 0) trace_mark(p, 3, 0, tl);
        ptx::tc_fence_after();
        const uint32_t t_acc = tmem_base + lane_addr + buf * 128 + 32 * eh;
        uint32_t v[32];
        ptx::tmem_ld_32x32b_x32(t_acc, v);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          // exact: every chunk sum is an integer below 2^24 in magnitude
          const uint32_t a = static_cast<uint32_t>(__float2int_rn(__uint_as_float(v[i])));
          run0[i] = c == 0 ? a : run0[i] + a;
        }
        ptx::tmem_ld_32x32b_x32(t_acc + 64, v);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const uint32_t a = static_cast<uint32_t>(__float2int_rn(__uint_as_float(v[i])));
          run1[i] = c == 0 ? a : run1[i] + a;
        }
        // the accumulator buffer is free once read (rank 0 waits for both CTAs)
        ptx::tc_fence_before();
        arrive_on_leader(&acc_empty[buf], ts);
        if (tr && c == nch - 1) trace_mark(p, 3, 1, tl);
      }
      if (!ok) break;
      // Shift column block 1 down by dw pixels: lanes below 32 - dw take it
      // from lane + dw of this warp, the last dw lanes from the first dw lanes
      // of the next lane quarter's warp (same channels) through shared memory
      // (two buffers, alternating tile by tile; one barrier per tile suffices
      // because a warp can only reuse a buffer after every warp has passed
      // the next tile's barrier).  The last quarter's last dw pixels are past
      // the tile's valid outputs.
      uint32_t* xb = reinterpret_cast<uint32_t*>(smem + hp.off_out) + (tl & 1u) * (8 * kStackMaxShift * 32);
      if (lane < dw) {
        uint4* row = reinterpret_cast<uint4*>(xb + ((warp - 8) * kStackMaxShift + lane) * 32);
#pragma unroll
        for (int i = 0; i < 8; ++i) row[i] = make_uint4(run1[4 * i], run1[4 * i + 1], run1[4 * i + 2], run1[4 * i + 3]);
      }
      if (!epi_barrier()) {
        ok = false;
        break;
      }
      if (tr) trace_mark(p, 3, 2, tl);
#pragma unroll
      for (int i = 0; i < 32; ++i) run1[i] = __shfl_down_sync(0xffffffffu, run1[i], dw);
      const int src_lane = lane - (32 - dw);  // >= 0: from the next quarter's warp (same eh)
      if (src_lane >= 0) {
        if (qd < 3) {
          const uint4* row = reinterpret_cast<const uint4*>(xb + ((warp - 8 + 1) * kStackMaxShift + src_lane) * 32);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint4 w = row[i];
            run1[4 * i] = w.x;
            run1[4 * i + 1] = w.y;
            run1[4 * i + 2] = w.z;
            run1[4 * i + 3] = w.w;
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) run1[i] = 0u;  // past the tile's valid outputs
        }
      }
      const RowTile t = decode_row_tile(2 * unit + ts.rank, hp);
      const int m = 32 * qd + lane;  // pixel of this lane: output column q0 + m
      if (t.valid && m < hp.vq && t.q0 + m < p.Q) {
        const int64_t off = ((static_cast<int64_t>(t.n) * p.KB + eh) * p.P + t.p) * p.Q + t.q0 + m;
        if (p.out_mode == 0) {
          uint32_t o[8];
          requant32(p, 32 * eh, [&](int i) { return static_cast<int>(run0[i] + run1[i]); }, o);
          uint4* dst = reinterpret_cast<uint4*>(p.y + off * 32);
          dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
          dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
        } else {
          uint4* dst = reinterpret_cast<uint4*>(p.acc + off * 32);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[i] = make_uint4(run0[4 * i] + run1[4 * i], run0[4 * i + 1] + run1[4 * i + 1],
                                run0[4 * i + 2] + run1[4 * i + 2], run0[4 * i + 3] + run1[4 * i + 3]);
        }
      }
      if (tr) trace_mark(p, 3, 3, tl);
    }
    if (!ok) raise_timeout(p, abort_flag);
  }

  ptx::tc_fence_before();
  __syncthreads();
  // the pair's CTAs leave together: no remote arrive, multicast commit or
  // MMA operand read targets a CTA that has exited
  ptx::cluster_sync();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_cg<CG>(tmem_base, p.tmem_cols);
  }
}

}  // namespace i8c
