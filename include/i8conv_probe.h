/*
 * i8conv engine probes -- microbenchmarks of the tensor-core engine the
 * convolution kernels are built on, for choosing tile shapes and for the
 * roofline denominator.  Not part of the convolution path.  The pages have no
 * counterpart; they name only the Ampere 16x8x32 integer MMA of the CUTLASS
 * configuration in the "int8 fprop2d kernel with NCxHWx interleaved layout"
 * issue, which sm_103a's tcgen05 tensor cores do not offer.
 */
#ifndef I8CONV_PROBE_H_
#define I8CONV_PROBE_H_

#include "i8conv.h"

#ifdef __cplusplus
extern "C" {
#endif

/* One CTA per SM (num_ctas CTAs); in each, one thread issues `iters`
 * tcgen05.mma.cta_group::1.kind::f16 instructions (M = 128, N = n in
 * {32, 64, 128, 176, 224, 256}, K = 16, fp32 accumulate) back to back on zero operands
 * resident in shared memory.  a_swizzled selects A's layout: 1 = 64-byte
 * swizzle; 0 = no swizzle with contiguous 8-row core matrices; 2 = no swizzle
 * with 8-row groups 160 bytes apart (a 10-position halo row); 3 = as 2 but
 * starting 16 bytes into the buffer (a filter tap shifted by one column).
 * B is 64-byte swizzled, except in loop_mode 0 with a_swizzled 4 or 5 (the
 * transposed-tile kernel's operands): A 64-byte swizzled, B without swizzle
 * in 8-channel planes of n*16 bytes with 8-row groups 128 bytes apart,
 * starting at the buffer (4) or 48 bytes into it (5, a shifted filter tap
 * whose core matrices straddle 128-byte lines).  loop_mode 0 issues bare MMAs; 1-3 issue them
 * in the convolution's per-K-slice pattern (pairs of MMAs with the A start
 * from a shared-memory table; 2 adds a completed-barrier check every 4
 * slices, 3 also a commit every 4 slices).  Modes 4-18 issue from a whole
 * warp in uniform control flow with one elected lane: 4 (A start from loop
 * counters), 5 (from a table), 6-7 (with epilogue warps waiting, sleeping or
 * polling), 8-9 (the convolution's run loop: runs of three K-slices, a
 * completed-barrier wait before and a commit after each run), 10 (four
 * warps storing to shared memory alongside), 11-14 (six MMAs, then 0, 200,
 * 400 or 800 idle cycles: queue depth), 15-18 (mode 8 without its commit,
 * without its wait, with one elected block per run, with one elected block
 * and neither wait nor commit), 19-20 (mode 8's loop on a four-stage ring of
 * full/empty barriers re-armed each run by a producer warp that sleeps (19)
 * or spins (20) in its waits).  iters must be a multiple of 6.
 *   cycles: DEVICE buffer of 3*num_ctas int64, per CTA: SM cycles to issue,
 *           SM cycles until all MMAs completed, 1 if the completion wait
 *           succeeded (bounded at 2 s)
 *   elapsed_ms: host float, kernel duration from CUDA events on `stream`.
 * Synchronises `stream`. */
i8c_status i8c_probe_mma_f16(int32_t n, int32_t a_swizzled, int32_t loop_mode, int32_t num_ctas, int32_t iters,
                             long long* cycles, float* elapsed_ms, cudaStream_t stream);

/* The warp-level integer MMA the Ampere configurations use
 * (mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32: 16 x 8 x 32 int8
 * multiply-adds per warp instruction, 8192 int8 ops): num_ctas CTAs of
 * warps_per_cta warps (1-16), each warp issuing iters x 8 MMAs on register
 * operands into 8 independent accumulators.
 *   cycles: DEVICE buffer of 3*num_ctas int64, per CTA: SM cycles of the loop
 *           (twice), 1;  sink: DEVICE int (written only if the accumulators
 *           come out at an impossible value: keeps them live)
 *   elapsed_ms: host float, kernel duration from CUDA events on `stream`.
 * Synchronises `stream`. */
i8c_status i8c_probe_imma_s8(int32_t num_ctas, int32_t warps_per_cta, int32_t iters, long long* cycles, int* sink,
                             float* elapsed_ms, cudaStream_t stream);

/* tcgen05.mma.cta_group::1.kind::f8f6f4 with e4m3 A and B and fp32
 * accumulation (M = 128, N = n in {64, 128, 256}, K = 32: the engine an
 * exact e4m3 nibble split of int8 operands would use), issued back to back
 * by one thread per CTA on zero operands in shared memory; cycles and
 * elapsed_ms as for i8c_probe_mma_f16.  Synchronises `stream`. */
i8c_status i8c_probe_mma_f8(int32_t n, int32_t num_ctas, int32_t iters, long long* cycles, float* elapsed_ms,
                            cudaStream_t stream);

/* L2 -> shared memory read rate of the SMs (the bound on how fast a CTA can
 * stream filter stages and halos): num_ctas CTAs of 512 threads, one per SM,
 * each moving `iters` chunks of chunk_bytes (a multiple of 16, at most 49152)
 * from the DEVICE buffer src (16-byte aligned, region_bytes long, a multiple
 * of chunk_bytes; small enough to stay in L2 once read, or not, as the
 * measurement wants) into four shared-memory buffers.  Step i of CTA c reads
 * chunk (c + i * num_ctas) mod (region_bytes / chunk_bytes).  mode 0: one
 * thread keeps four untiled bulk copies (cp.async.bulk, the TMA) in flight;
 * mode 1: every thread loads 16-byte vectors, four in flight, and stores
 * them to shared memory (chunk_bytes a multiple of 32768); mode 2: clusters
 * of two CTAs (num_ctas even, chunk_bytes a multiple of 32), each copying
 * half of every chunk into both CTAs' buffer with one multicast bulk copy
 * (this GPU's memory only), four chunks in flight, a buffer refilled once
 * both CTAs hold its previous chunk; step i of cluster c reads chunk
 * (c + i * num_ctas / 2) mod (region_bytes / chunk_bytes), and the bytes
 * counted per CTA are the bytes it received; mode 3: every thread copies
 * its 16-byte pieces of each chunk with cp.async (global -> shared, no
 * registers), one commit group per chunk, three groups in flight.
 *   cycles: DEVICE buffer of 3*num_ctas int64, per CTA: SM cycles of the
 *           loop, bytes moved, 1 if every bounded wait succeeded
 *   elapsed_ms as for i8c_probe_mma_f16.  Synchronises `stream`. */
i8c_status i8c_probe_l2_ingress(const void* src, int64_t region_bytes, int32_t chunk_bytes, int32_t mode,
                                int32_t num_ctas, int32_t iters, long long* cycles, float* elapsed_ms,
                                cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* I8CONV_PROBE_H_ */
