/*
 * i8conv -- INT8 Conv2d forward propagation (fprop) on one GB300 (sm_103a).
 *
 * The operation is the one configured in the CUTLASS issue "How to optimize
 * cutlass int8 fprop2d kernel with NCxHWx interleaved layout" (section "CUTLASS
 * Kernel Configuration"): DefaultConv2dFprop with int8 activations in
 * NCxHWx<32>, int8 filters in CxRSKx<32>, int8 outputs in NCxHWx<32>, an int32
 * accumulator and the LinearCombinationClamp epilogue with alpha-only scaling:
 *
 *     acc[n][k][p][q] = sum_{c,r,s} x[n][c][p*stride_h - pad_h + r*dil_h]
 *                                         [q*stride_w - pad_w + s*dil_w] * f[k][c][r][s]
 *     y[n][k][p][q]   = clamp(rint(alpha * (float)acc), -128, 127)
 *
 * with zero padding, P = floor((H + 2*pad_h - dil_h*(R-1) - 1)/stride_h) + 1
 * and Q likewise (the output-size formula of the POPCORNBENCH l1_p80 trace,
 * first analysis paragraph).  (float)acc rounds to nearest even, the product
 * is one fp32 multiply, rint rounds half to even.  Results are bit-exact.
 *
 * Memory layouts (all int8, all dense, no padding between elements):
 *   NCxHWx<32>: element (n, c, h, w) at (((n*C/32 + c/32)*H + h)*W + w)*32 + c%32
 *   CxRSKx<32>: element (k, c, r, s) at ((((c/32)*R + r)*S + s)*K + k)*32 + c%32
 *   NCHW / KCRS: the plain row-major orders (used only by the pack helpers).
 * The CxRSKx<32> formula is our reading of the layout's name by analogy with
 * NCxHWx<32>; the pack/unpack helpers below define it.
 *
 * Conventions for every entry point:
 *   - Tensor pointers are DEVICE pointers owned by the caller, 16-byte aligned
 *     (the configuration's 16/16 alignment), and inputs never alias outputs.
 *   - Work is enqueued on `stream` (0 = legacy default stream) and returns
 *     immediately; results are valid once the stream reaches that point.
 *   - No entry point throws; each returns an i8c_status.  Argument errors are
 *     detected on the host before anything is enqueued.  Errors raised while a
 *     kernel runs (a bounded wait that ran out) are recorded in a device
 *     status word: read per plan by i8c_plan_status(), and for the checked
 *     one-shot calls by i8c_last_device_status().
 *   - There is no CPU fallback: without a usable CUDA device the calls fail
 *     with I8C_ERR_CUDA / I8C_ERR_NO_DEVICE.
 */
#ifndef I8CONV_H_
#define I8CONV_H_

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  I8C_OK = 0,
  I8C_ERR_INVALID_ARG = 1,   /* null pointer, non-positive size, bad option   */
  I8C_ERR_UNSUPPORTED = 2,   /* C or K not a multiple of 32, empty output     */
  I8C_ERR_MISALIGNED = 3,    /* a tensor pointer is not 16-byte aligned       */
  I8C_ERR_OVERFLOW_RISK = 4, /* C*R*S*128*128 could exceed int32, or a size
                                overflows 32-bit indexing                      */
  I8C_ERR_CUDA = 5,          /* a CUDA runtime/driver call failed             */
  I8C_ERR_TIMEOUT = 6,       /* a kernel's bounded wait ran out (device side) */
  I8C_ERR_NO_DEVICE = 7      /* no CUDA device, or not an sm_103 device       */
} i8c_status;

/* Convolution geometry.  Padding, stride and dilation are per axis (h, w);
 * the same padding is applied on both sides of an axis, as in nn.Conv2d. */
typedef struct {
  int32_t N, C, H, W; /* batch, input channels, input height and width   */
  int32_t K, R, S;    /* output channels, filter height and width         */
  int32_t pad_h, pad_w, stride_h, stride_w, dil_h, dil_w;
} i8c_conv_shape;

/* Plan options.  Zero-initialise for defaults. */
typedef struct {
  int32_t block_n;           /* output channels per tile: 0 = auto, else 32, 64, 128 or 256   */
  int32_t num_ctas;          /* persistent CTAs: 0 = one per SM                                */
  int32_t max_chunk_slices;  /* K-slices (32 channels each) per exact fp32 chunk: 0 = 32      */
  int32_t wait_timeout_us;   /* device-side bounded waits: 0 = 2,000,000 us                     */
  int32_t host_staging;      /* 1 = allocate device staging buffers for i8c_plan_run_host,
                                2 = two staging sets and copy streams, for
                                i8c_plan_run_host_pipelined as well                        */
  int32_t debug_flags;       /* test hooks, see I8C_DEBUG_*; 0 in production                  */
  int32_t timing_events;     /* > 0: bracket each convolution kernel with CUDA events (keeps
                                the last timing_events launches) for i8c_plan_kernel_time;
                                for benchmarks, not for use under graph capture               */
  int32_t kernel_variant;    /* 0 = auto, 1 = per-tap gather kernel, 2 = halo kernel (16x8
                                output patches; I8C_ERR_UNSUPPORTED if its halo does not fit),
                                3 = halo kernel on CTA pairs (clusters of two SMs sharing one
                                M = 256 MMA per K-step; block_n 64, 128 or 256), 4 = transposed
                                tiles (128 output channels x tile_px output pixels per tile, the
                                MMA's M on the channels; stride 1 only, else
                                I8C_ERR_UNSUPPORTED), 5 = transposed tiles on CTA pairs (256
                                output channels, 128 per CTA, x tile_px pixels, each CTA
                                building the halo of half of them; stride 1 only), 6 = stacked
                                taps (64 output channels only, stride 1, 2 <= S <= 16,
                                dil_w <= 8: two filter taps of a row per N = 128 MMA on CTA
                                pairs; row tiles of 128 - dil_w output columns)               */
  int32_t halo_loads;        /* halo and transposed-tile kernels, how activations reach
                                shared memory: 0 = auto, 1 = int8 staging ring filled by
                                cp.async ahead of use, 2 = straight into registers (no
                                staging memory), 3 = one TMA box per tile and channel block
                                into int8 slots, converted to fp16 in shared memory;
                                I8C_ERR_UNSUPPORTED if the forced form does not fit        */
  int32_t tail_split;        /* halo kernel, the tiles of a partial last wave: 0 = auto (split
                                along the channel blocks when the estimated saving clearly
                                exceeds the partial-sum traffic), 1 = never split, 2 = split
                                along the channel blocks (int32 partial sums combined by the
                                unit that finishes last; needs plan workspace) whenever the
                                last wave is partial, 3 = halve them along the output channels
                                (N = BN/2 MMAs, disjoint outputs) when the halves fit in the
                                wave and the tile is 128 or 256 wide                         */
  int32_t tile_shape;        /* halo kernel, the output pixels of a tile: 0 = auto, 1 = a 16x8
                                patch, 2 = 128 consecutive pixels of the output laid out with
                                the zero-padded input's row width (stride 1 only; the pixels
                                past Q in each row are computed and discarded), 3 = a 16x16
                                patch: two 16x8 sub-tiles on one halo, two MMAs per tap and K
                                half (block_n <= 128, whole filter rows per filter stage,
                                register or staged halo loads, no split tail; else
                                I8C_ERR_UNSUPPORTED).  Auto takes 16x16 patches at block_n
                                <= 64 where they keep the filter resident (one output-
                                channel tile whose every stage fits) and the planner's cost
                                model prefers them                                          */
  int32_t fused_filter;      /* where the int8 filter becomes the fp16 MMA operand:
                                0 = auto (2 where the halo kernel keeps the whole filter
                                resident in shared memory, else 3);
                                1 = halo kernel on single CTAs: inside the convolution kernel,
                                each CTA converting a share into a global fp16 copy behind a
                                grid barrier (one launch per run; all CTAs resident;
                                measured slower);
                                2 = halo kernel (single CTAs or pairs) with a resident filter:
                                every CTA converts the rows and K-slices it keeps straight
                                into its shared-memory filter stages before its warps split
                                into roles (one launch per run, no fp16 copy);
                                I8C_ERR_UNSUPPORTED where the filter is not resident;
                                3 = a separate conversion kernel launched first, writing the
                                fp16 copy the filter TMA reads (the convolution's prologue
                                overlaps its tail)                                           */
  int32_t tile_px;           /* transposed tiles: output pixels per tile (the MMA's N; on
                                pairs split between the two CTAs), 0 = auto (the width whose
                                tile count fills the SMs' waves best), else a multiple of 16
                                from 16 to 256                                                */
  int32_t filter_run;        /* transposed tiles: K-slices (taps of one channel block) per
                                filter stage, 0 = auto (the longest that leaves two stages),
                                else a divisor of R*S; I8C_ERR_UNSUPPORTED if it does not fit */
} i8c_options;

/* debug_flags: make the activation producers skip their first arrival, so
 * the MMA warp's bounded wait runs out and the kernel reports
 * I8C_ERR_TIMEOUT without faulting or hanging.  Used by the failure tests. */
#define I8C_DEBUG_SKIP_FIRST_ARRIVE 1
/* debug_flags: record clock64 timestamps of the pipeline waits of CTA 0 in a
 * plan-owned buffer, read back with i8c_plan_trace (pipeline analysis). */
#define I8C_DEBUG_TRACE 2

typedef struct i8c_plan i8c_plan;


/* Per-output-channel epilogue of i8c_plan_run_ex / i8c_conv2d_fprop_ex (the
 * row-wise scaling of the weight-only quantisation issue, with a bias and a
 * ReLU fused before the clamp):
 *     y[n][k][p][q] = clamp(rint(relu(alpha_k * (float)acc + bias_k)), -128, 127)
 * one fp32 multiply, then one fp32 add, each rounded to nearest even (never
 * fused), relu(v) = max(v, 0) when asked for, rint half to even.  With
 * alpha = NULL and bias = NULL and relu = 0 this is the alpha-only epilogue of
 * i8c_plan_run.  Both arrays are DEVICE memory of K floats, 16-byte aligned,
 * read by the kernel (owned by the caller; not modified). */
typedef struct {
  const float* alpha;  /* per-channel scales, or NULL: the scalar alpha argument */
  const float* bias;   /* per-channel biases added after the scale, or NULL: none */
  int32_t relu;        /* 1: clamp below at 0 (ReLU) before the int8 clamp      */
} i8c_epilogue;

/* Read-only facts about a plan (for benchmarks and tests). */
typedef struct {
  int32_t P, Q;              /* output height and width                        */
  int64_t M;                 /* GEMM rows: N*P*Q                               */
  int32_t gemm_n, gemm_k;    /* GEMM columns (K) and reduction length (C*R*S)  */
  int32_t block_m, block_n;  /* tile shape (block_m 256 for a CTA pair's tile) */
  int32_t num_tiles;         /* M-tiles x N-tiles                              */
  int32_t num_ctas;          /* persistent grid size                           */
  int32_t num_chunks;        /* exact fp32 chunks per tile                     */
  int32_t chunk_slices;      /* K-slices per chunk                             */
  int32_t acc_buffers;       /* tensor-memory accumulator buffers              */
  int32_t smem_bytes;        /* dynamic shared memory per CTA                  */
  int32_t kernels_per_run;   /* kernel launches enqueued by one i8c_plan_run   */
  int64_t ops;               /* 2*N*K*P*Q*C*R*S                                 */
  int64_t workspace_bytes;   /* device memory owned by the plan                */
  int32_t kernel_variant;    /* 1 = per-tap gather kernel, 2 = halo kernel,
                                3 = halo kernel on CTA pairs, 4 = transposed
                                tiles (block_m = tile_px pixels, block_n = 128
                                output channels), 5 = transposed tiles on CTA
                                pairs (block_n = 256), 6 = stacked taps
                                (block_m = a pair's two row tiles of valid
                                outputs, block_n = 64; chunk_slices counts
                                filter rows)                                   */
  int32_t halo_staging;      /* halo kernel: int8 staging slots (0 = loads
                                straight into registers); 0 for the gather kernel */
  int32_t filter_run;        /* halo kernel: K-slices per filter stage (taps of
                                one filter row); 1 for the gather kernel       */
  int32_t filter_stages;     /* filter pipeline stages in shared memory        */
  int32_t tail_split;        /* channel-block units per last-wave tile (1: none) */
  int32_t work_units;        /* units of work the persistent CTAs share          */
  int32_t tail_halves;       /* 2 when last-wave tiles are halved along the output channels */
  int32_t flat_tiles;        /* 1 when tiles are 128 consecutive padded-row pixels */
  int32_t filter_resident;   /* halo kernel: 1 when the filter stages are loaded
                                once per CTA and kept (one output-channel tile,
                                whole-tile units, every stage fits)           */
} i8c_plan_info;

/* Shared- and tensor-memory layout of a plan's kernel, as the kernel will
 * use it: the numbers a host-side bounds check needs to show that every
 * matrix descriptor, TMA box and producer store stays inside its region.
 * Byte offsets are relative to the CTA's 1024-byte-aligned shared-memory
 * base (smem_bytes includes the 1024 bytes of slack for that alignment). */
typedef struct {
  int32_t kernel_variant;      /* as in i8c_plan_info                                  */
  int32_t cta_group;           /* CTAs per MMA tile (2: a CTA pair)                    */
  int32_t block_n;             /* output channels per tile (variants 4, 5: 128 per CTA) */
  int32_t smem_bytes;          /* dynamic shared memory requested per CTA              */
  int32_t tmem_cols;           /* tensor-memory columns allocated per CTA              */
  int32_t chunk_slices;        /* K-slices per exact fp32 chunk                        */
  int32_t num_chunks;
  /* halo and transposed-tile kernels (variants 2-5; 0 for the gather kernel) */
  int32_t flat_tiles;          /* 1: tiles of consecutive padded-row pixels            */
  int32_t tile_px;             /* flat tiles: output pixels per CTA and tile            */
  int32_t halo_rows, halo_cw;  /* halo rows; positions per halo row (flat: padded W)   */
  int32_t positions;           /* halo positions per channel block                     */
  int32_t plane_bytes;         /* one 8-channel fp16 plane of the halo                 */
  int32_t halo_bytes;          /* one halo stage: 4 planes                             */
  int32_t halo_stages;
  int32_t off_staging, staging_slots, staging_bytes;  /* int8 staging ring (may be empty) */
  int32_t off_filter;          /* first filter stage                                   */
  int32_t filter_stages;
  int32_t filter_run;          /* K-slices per filter stage                            */
  int32_t filter_stage_bytes;  /* filter_run x filter rows per CTA x 64 bytes          */
  int32_t off_out;             /* transposed tiles: the epilogue's output staging rows */
  int32_t off_bar, bar_bytes;  /* mbarriers and the CTA's control words                */
  int32_t phase_off[9];        /* halo: first position of column phase f, f <= stride_w */
  /* TMA-fed halos (halo_loads = 3): int8 slots of one TMA box each */
  int32_t tma_halo, x8_slots, off_x8, x8_bytes, box_w, box_h;
  /* per-tap gather kernel (variant 1; 0 otherwise) */
  int32_t gather_stages, gather_off_a, gather_stage_a, gather_off_b, gather_stage_b;
  int32_t gather_off_staging, gather_staging_slots, gather_staging_bytes, gather_off_bar;
  /* halo kernel, 2-D patches: 16x8 sub-tiles per patch (2 for 16x16 patches) */
  int32_t subtiles;
} i8c_layout;

/* The layout i8c_plan_create would give `shape` with `opts` (may be NULL) on
 * a GPU of `num_sms` SMs, computed on the host alone: no CUDA call is made,
 * so it works without a GPU (CTA pairs are assumed to fit one per two SMs,
 * which changes only the grid size, not the layout).  Errors as for
 * i8c_plan_create's argument and shape checks, and I8C_ERR_UNSUPPORTED when
 * a forced kernel form does not fit. */
i8c_status i8c_plan_layout(const i8c_conv_shape* shape, const i8c_options* opts, int32_t num_sms,
                           i8c_layout* out);

/* The same layout for an existing plan. */
i8c_status i8c_plan_get_layout(const i8c_plan* plan, i8c_layout* out);

/* Output height P and width Q for a shape (formula above).  Returns
 * I8C_ERR_INVALID_ARG for non-positive sizes or negative padding and
 * I8C_ERR_UNSUPPORTED when the dilated filter does not fit (P or Q < 1). */
i8c_status i8c_output_size(const i8c_conv_shape* shape, int32_t* P, int32_t* Q);

/* The argument check of the checked entry points (the CUTLASS Python API's
 * supports(), host-latency tutorial, "Bypassing argument checks"):
 * positive sizes, C % 32 == 0, K % 32 == 0, P, Q >= 1, C*R*S*16384 < 2^31
 * (so no int32 accumulator can overflow and saturating accumulation is moot),
 * and every tensor small enough for 32-bit element offsets per image plane. */
i8c_status i8c_supported(const i8c_conv_shape* shape);

/* Checked one-shot convolution: validates, then runs on `stream` using a
 * plan cached per (shape, device).  The first call for a shape creates the
 * plan (allocates and may synchronise the device); later calls do not.
 *   x: NCxHWx<32> int8 [N][C/32][H][W][32], read-only
 *   f: CxRSKx<32> int8 [C/32][R][S][K][32], read-only
 *   y: NCxHWx<32> int8 [N][K/32][P][Q][32], written */
i8c_status i8c_conv2d_fprop(const int8_t* x, const int8_t* f, int8_t* y, const i8c_conv_shape* shape,
                            float alpha, cudaStream_t stream);

/* As i8c_conv2d_fprop, but writes the int32 accumulators instead of the
 * epilogue result: acc is [N][K/32][P][Q][32] int32 (same interleave).
 * For parity checks of the contraction alone. */
i8c_status i8c_conv2d_fprop_acc(const int8_t* x, const int8_t* f, int32_t* acc, const i8c_conv_shape* shape,
                                cudaStream_t stream);

/* As i8c_conv2d_fprop, with the per-output-channel epilogue `ep` (see
 * i8c_epilogue; NULL: the alpha-only epilogue). */
i8c_status i8c_conv2d_fprop_ex(const int8_t* x, const int8_t* f, int8_t* y, const i8c_conv_shape* shape,
                               float alpha, const i8c_epilogue* ep, cudaStream_t stream);

/* Same convolution and arguments as i8c_conv2d_fprop, for callers that must
 * not allocate device memory.  The pages have no counterpart to this entry
 * point; it exists for code whose device memory is owned by someone else
 * (a framework's caching allocator or a fixed memory-pool budget), for
 * latency-critical paths where cudaMalloc's implicit synchronisation is not
 * acceptable, and for plug-ins that may use only the buffers they are given.
 *
 * It calls no cudaMalloc, cudaFree or other allocating routine.  Its scratch
 * (the fp16 copy of the filter and a status word) lives in one 8 MiB static
 * device array inside the library, which every GPU that loads the library
 * keeps until the process exits.  Limit: K*C*R*S <= 4,194,176 filter
 * elements; larger filters return I8C_ERR_UNSUPPORTED and nothing is
 * enqueued.  Other argument errors are as for i8c_conv2d_fprop.
 *
 * The first call on a device looks up the array's device address and sets up
 * the kernels for that device (host-side queries, no allocation); make that
 * first call before any stream capture.  All calls share the one array and
 * each call overwrites it, so calls that may overlap on the GPU (different
 * streams, or different host threads) race and must be serialised by the
 * caller.  A device-side wait that runs out is recorded in the array's
 * status word (zeroed at the start of every call); i8c_last_device_status
 * reads it back, without allocating, and the output is then undefined. */
i8c_status i8c_conv2d_fprop_noalloc(const int8_t* x, const int8_t* f, int8_t* y, const i8c_conv_shape* shape,
                                    float alpha, cudaStream_t stream);

/* Device status of the checked one-shot calls (the checked-call side of the
 * host-latency tutorial's split, "Bypassing argument checks": the checked
 * calls report what their kernels met).  Synchronises `stream`, then returns
 * and clears the device status words of the plans that i8c_conv2d_fprop,
 * i8c_conv2d_fprop_acc and i8c_conv2d_fprop_ex cached for (current device,
 * `stream`), and of i8c_conv2d_fprop_noalloc on the current device (one word
 * per device, shared by all streams: reliable when its last call was made on
 * `stream`).  I8C_OK, or I8C_ERR_TIMEOUT if a bounded wait in one of their
 * kernels ran out since the last read (the outputs of that call are then
 * undefined; the next call runs normally).  Allocates nothing.
 *
 * The one-shot calls keep at most 64 cached plans (one per device, stream
 * and shape); creating a 65th destroys the least recently used one, which
 * synchronises the device, and a status word not yet read goes with it. */
i8c_status i8c_last_device_status(cudaStream_t stream);

/* Number of plans the one-shot calls currently keep (at most 64). */
int64_t i8c_oneshot_cached_plans(void);

/* Test hook: destroys the one-shot calls' cached plans (synchronising the
 * device) and makes the plans they create from now on, and the
 * no-allocation entry point, run with these i8c_options debug_flags and
 * wait_timeout_us (0, 0: the defaults).  I8C_ERR_INVALID_ARG for negative
 * values.  Not for production use. */
i8c_status i8c_debug_set_oneshot(int32_t debug_flags, int32_t wait_timeout_us);

/* Compile-once / run-many (host-latency tutorial, "Compiling once"): a plan
 * holds the validated shape, the tile schedule, the filter staging buffer
 * and a device status word, allocated on the current device.  `opts` may be
 * NULL.  The plan must be used on that device and destroyed by the caller. */
i8c_status i8c_plan_create(const i8c_conv_shape* shape, const i8c_options* opts, i8c_plan** plan);

/* Unchecked run (host-latency tutorial, "Bypassing argument checks"): no
 * shape validation (only null and 16-byte alignment checks, since a
 * misaligned vector access would otherwise fault the device), no
 * allocation, no synchronisation, so it
 * can be captured in a CUDA graph (tutorial section "CUDA Graphs").  Runs
 * sharing one plan must be serialised on one stream: they share the plan's
 * filter staging buffer. */
i8c_status i8c_plan_run(const i8c_plan* plan, const int8_t* x, const int8_t* f, int8_t* y, float alpha,
                        cudaStream_t stream);

/* i8c_plan_run with the per-output-channel epilogue `ep` (NULL: the
 * alpha-only epilogue).  I8C_ERR_MISALIGNED if ep->alpha or ep->bias is not
 * 16-byte aligned.  Same scheduling rules as i8c_plan_run. */
i8c_status i8c_plan_run_ex(const i8c_plan* plan, const int8_t* x, const int8_t* f, int8_t* y, float alpha,
                           const i8c_epilogue* ep, cudaStream_t stream);

/* Unchecked run that writes int32 accumulators (layout as in _acc above). */
i8c_status i8c_plan_run_acc(const i8c_plan* plan, const int8_t* x, const int8_t* f, int32_t* acc,
                            cudaStream_t stream);

/* Weight prepacking.  The filter operand transform (int8 -> the fp16
 * operand copy, or the stacked-tap order) is done once, for filters that
 * stay fixed across runs (inference weights): i8c_plan_set_filter converts
 * the int8 CxRSKx<32> filter f (DEVICE, 16-byte aligned; read on `stream`
 * before the call's work completes) into plan-owned memory -- for plans
 * whose kernel writes its resident filter itself, an int8 copy of f that
 * every run converts in shared memory -- and i8c_plan_run_prepacked(_ex)
 * then run the convolution alone on x (DEVICE) into y (DEVICE), as
 * i8c_plan_run(_ex) would with that filter: one kernel launch per run.
 * The copy is the plan's: f may change or be freed after set_filter's work
 * is done.  Any i8c_plan_run* call that takes a filter replaces the copy;
 * run_prepacked then returns I8C_ERR_INVALID_ARG until set_filter is called
 * again (also before the first set_filter).  The convolution kernels are
 * dependent launches: a run's kernel starts on SMs as soon as the kernel
 * ahead of it frees them and waits for that kernel only before reading
 * memory it may have written (the activations; the filter copy right after
 * set_filter), so successive prepacked runs load their filter stages while
 * the previous run finishes.  Not thread-safe per plan, like every other
 * plan call. */
i8c_status i8c_plan_set_filter(const i8c_plan* plan, const int8_t* f, cudaStream_t stream);
i8c_status i8c_plan_run_prepacked(const i8c_plan* plan, const int8_t* x, int8_t* y, float alpha,
                                  cudaStream_t stream);
i8c_status i8c_plan_run_prepacked_ex(const i8c_plan* plan, const int8_t* x, int8_t* y, float alpha,
                                     const i8c_epilogue* ep, cudaStream_t stream);

/* End-to-end run on HOST buffers: copies x and f from host memory into the
 * plan's staging buffers, runs, and copies y back, all on `stream`.  The plan
 * must have been created with host_staging = 1.  Pinned (page-locked) host
 * memory makes the copies asynchronous; the caller synchronises `stream`
 * before reading y. */
i8c_status i8c_plan_run_host(const i8c_plan* plan, const int8_t* x_host, const int8_t* f_host, int8_t* y_host,
                             float alpha, cudaStream_t stream);

/* `steps` end-to-end runs on HOST buffers, pipelined: run i copies x_host[i]
 * and f_host[i] in, runs with alpha[i] and copies y out to y_host[i] (each
 * array holds `steps` host pointers; pinned memory makes the copies
 * asynchronous).  The plan must have been created with host_staging = 2: two
 * device staging sets and two copy streams owned by the plan, so that the
 * input copies of run i + 1 and the output copy of run i - 1 overlap run i
 * (the runs stay on `stream`, in order, sharing the plan's filter buffer).
 * Enqueues everything and returns; `stream` reaches the end of the call once
 * the last output copy has completed, so the caller synchronises `stream`
 * before reading any y_host[i].  Host buffers must stay untouched until
 * then.  I8C_ERR_INVALID_ARG for null pointers, steps < 0, or a plan
 * without the second staging set.  Not capturable (it records events on
 * the plan's own streams). */
i8c_status i8c_plan_run_host_pipelined(const i8c_plan* plan, const int8_t* const* x_host,
                                       const int8_t* const* f_host, int8_t* const* y_host, const float* alpha,
                                       int32_t steps, cudaStream_t stream);

/* Synchronises `stream`, then returns (and clears) the plan's device status
 * word: I8C_OK, or I8C_ERR_TIMEOUT if a bounded wait in a kernel ran out. */
i8c_status i8c_plan_status(const i8c_plan* plan, cudaStream_t stream);

i8c_status i8c_plan_get_info(const i8c_plan* plan, i8c_plan_info* info);

/* With timing_events > 0: synchronises on the last recorded event, returns
 * the summed device time (ms) of the convolution-kernel launches recorded
 * since the previous call and their count, and starts a new window.  Only
 * the last timing_events launches are kept. */
i8c_status i8c_plan_kernel_time(const i8c_plan* plan, double* total_ms, int64_t* launches);

/* With I8C_DEBUG_TRACE: copies up to `count` entries of the last run's trace
 * (synchronous): entry (role*4 + event)*512 + i is the SM clock at event
 * `event` of step i of role 0 MMA issuer, 1 filter TMA, 2 activation
 * producer, 3 epilogue; 0 where not reached.  Up to 32*512 entries: entries
 * from 16*512 on are only written by builds made for pipeline analysis. */
i8c_status i8c_plan_trace(const i8c_plan* plan, long long* out, int64_t count);

/* Frees the plan's device memory.  Synchronises the device first. */
i8c_status i8c_plan_destroy(i8c_plan* plan);

/* One candidate of i8c_plan_autotune: its options, the status of creating
 * and running its plan (I8C_OK, or why the candidate was skipped: e.g.
 * I8C_ERR_UNSUPPORTED for a kernel form the shape cannot use), and its mean
 * device time per i8c_plan_run in microseconds (0 unless status is I8C_OK). */
typedef struct {
  i8c_options options;
  int32_t status;
  float us;
} i8c_tune_entry;

/* Plan selection by measurement, the search step of the "[BYOC] CUTLASS
 * integration" pull request (apache/tvm #9261, tune_cutlass_kernels):
 * creates each plan of a fixed candidate list for `shape` (i8c_plan_create's
 * own choice first, then forced kernel forms, tile widths and CTA pairing),
 * runs it twice untimed and `iters` times between CUDA events on `stream`,
 * on the caller's tensors (layouts as for i8c_conv2d_fprop), and returns in
 * *best the options of the fastest and in *best_us its mean time per run
 * (filter staging + convolution).  Candidates whose plan cannot be created
 * for the shape, or whose bounded waits ran out, are skipped.  Since the
 * default comes first and ties keep the earlier candidate, the result is
 * never slower than the default on these inputs (within timing noise).
 *   entries / max_entries: optional (NULL, 0): the first max_entries
 *     candidates' results, in order; *num_entries (optional) gets how many
 *     were written.
 *   On return y holds the chosen plan's output.
 * Not for the hot path: it allocates and frees plans, synchronises the
 * device, and cannot be captured in a graph.  Pass *best to i8c_plan_create
 * to get the tuned plan.  Errors: I8C_ERR_INVALID_ARG (null pointer,
 * iters < 1), I8C_ERR_MISALIGNED, the i8c_supported status of the shape, or
 * the default candidate's status if no candidate could run. */
i8c_status i8c_plan_autotune(const i8c_conv_shape* shape, const int8_t* x, const int8_t* f, int8_t* y, float alpha,
                             int32_t iters, cudaStream_t stream, i8c_options* best, float* best_us,
                             i8c_tune_entry* entries, int32_t max_entries, int32_t* num_entries);

/* Layout helpers (device, byte permutations, not part of the timed path).
 * C (resp. K for filters) must be a multiple of 32 where it is interleaved. */
i8c_status i8c_pack_nchw_to_ncxhwx32(const int8_t* src, int8_t* dst, int32_t N, int32_t C, int32_t H, int32_t W,
                                     cudaStream_t stream);
i8c_status i8c_unpack_ncxhwx32_to_nchw(const int8_t* src, int8_t* dst, int32_t N, int32_t C, int32_t H, int32_t W,
                                       cudaStream_t stream);
i8c_status i8c_pack_kcrs_to_cxrskx32(const int8_t* src, int8_t* dst, int32_t K, int32_t C, int32_t R, int32_t S,
                                     cudaStream_t stream);
i8c_status i8c_unpack_cxrskx32_to_kcrs(const int8_t* src, int8_t* dst, int32_t K, int32_t C, int32_t R, int32_t S,
                                       cudaStream_t stream);

/* The fp32 direct convolution of the POPCORNBENCH kernel-benchmark trace
 * (problem l1_p80, nn.Conv2d on fp32 tensors; the trace's checker compares
 * with the framework's convolution at atol = rtol = 1e-4):
 *     y[n][k][p][q] = bias[k] + sum_{c,r,s} x[n][c][h][w] * w[k][c][r][s]
 * with h, w, P and Q as for the int8 convolution (zero padding, per-axis
 * stride and dilation).  Computed on the SIMT cores in IEEE fp32: one fused
 * multiply-add per product in the order (c, r, s), then the bias, so every
 * output is within the fp32 summation bound of the exact sum.
 *   x: NCHW fp32 [N][C][H][W]; w: KCRS fp32 [K][C][R][S]; bias: K floats or
 *   NULL (no bias); y: NCHW fp32 [N][K][P][Q], written.  All DEVICE memory,
 *   4-byte aligned, owned by the caller; any C and K >= 1.
 * The first call for a filter size on a device allocates a transposed copy of
 * the weight there (cudaMalloc; kept until exit); calls with the same filter
 * size share that copy and must be serialised on one stream.
 * Errors: I8C_ERR_INVALID_ARG (null pointer, bad sizes), I8C_ERR_MISALIGNED,
 * I8C_ERR_UNSUPPORTED (empty output, N > 65535, or a filter whose input
 * region and weights per input channel exceed the kernel's shared memory),
 * I8C_ERR_OVERFLOW_RISK (an image over 2^31 elements), I8C_ERR_NO_DEVICE. */
i8c_status i8c_conv2d_fprop_f32(const float* x, const float* w, const float* bias, float* y,
                                const i8c_conv_shape* shape, cudaStream_t stream);

/* Human-readable name of a status code (static string). */
const char* i8c_status_string(i8c_status status);

/* Number of kernel launches this library has enqueued in this process
 * (all entry points, all devices).  For launch accounting in benchmarks. */
int64_t i8c_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* I8CONV_H_ */
