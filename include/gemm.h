/*
 * gemm.h: C-ABI of the GB300 (sm_103a) dense GEMM library.
 *
 *     C = A · B (+ bias)
 *
 * The operation is the matrix product with an added bias row, "Output =
 * Input * Weight + Bias", which the FuseReductionEpilogue series
 * (kimm240.github.io/tvm, "[TIR][Schedule] Add FuseReductionEpilogue
 * primitive to fuse epilogue into reduction init", parts 1 and 2) fuses into the
 * reduction by starting it from the bias.  fp16 inputs are multiplied and summed
 * in fp32, the mixed-precision multiply-accumulate of the Tensor Core notes
 * (je-d.tistory.com, "tvm").  fp32 inputs run the CUDA-core path of the
 * "TVM Matrix Multiplication Optimization" ladder (kimm240.github.io/tvm,
 * Steps 1-7).  Small and skinny shapes use the Stream-K decomposition of the
 * leiblog.wang Stream-K post (Technical index).
 *
 * Conventions for every call:
 *   - A is M x K, B is K x N, C is M x N; sizes are element counts (>= 0).
 *   - Leading dimensions are packed: A row-major has lda = K, column-major lda = M;
 *     B row-major has ldb = N, column-major ldb = K; C is row-major, ldc = N.
 *   - A, B, bias, C are DEVICE pointers on the handle's device, owned by the
 *     caller; the library never frees or retains them past the call.
 *   - bias is NULL or N fp32 values, added to every row in fp32 before the
 *     single rounding to the output type.
 *   - stream is a cudaStream_t (NULL = the legacy default stream).
 *   - Every function returns a gemm_status_t; nothing aborts, traps or prints
 *     (set GEMM_LOG=1 in the environment to print each plan to stderr).
 */
#ifndef DGEMM_GB300_GEMM_H_
#define DGEMM_GB300_GEMM_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct gemm_ctx *gemm_handle_t;

typedef enum {
  GEMM_OK = 0,
  GEMM_ERR_INVALID_ARG = -1,    /* bad size, null pointer, unknown enum */
  GEMM_ERR_UNSUPPORTED = -2,    /* valid request this library does not run */
  GEMM_ERR_ALLOC = -3,          /* device or host allocation failed */
  GEMM_ERR_CUDA = -4,           /* a CUDA runtime/driver call failed */
  GEMM_ERR_DEVICE_TIMEOUT = -5  /* a bounded device-side wait expired */
} gemm_status_t;

enum { GEMM_F16 = 0, GEMM_F32 = 1 };
enum { GEMM_ROW_MAJOR = 0, GEMM_COL_MAJOR = 1 };

/* Storage and types.  a_major/b_major: GEMM_ROW_MAJOR or GEMM_COL_MAJOR.
 * in_dtype applies to both A and B.  Supported pairs: f16 -> f16, f16 -> f32,
 * f32 -> f32.  f32 -> f16 returns GEMM_ERR_UNSUPPORTED. */
typedef struct {
  uint8_t a_major;
  uint8_t b_major;
  uint8_t in_dtype;
  uint8_t out_dtype;
} gemm_layout_t;

/* Kernels the picker chooses among. */
enum {
  GEMM_KERNEL_TC = 0,       /* tcgen05/TMEM tensor-core GEMM, whole output tiles */
  GEMM_KERNEL_STREAMK = 1,  /* the same kernel with Stream-K (or hybrid) k-splitting */
  GEMM_KERNEL_SIMT = 2,     /* CUDA-core GEMM, fp32 accumulation: fp32 inputs, or fp16
                               inputs the tensor-core path cannot read */
  GEMM_KERNEL_FILL = 3,     /* K == 0: C = bias (or 0) */
  GEMM_KERNEL_NONE = 4,     /* M == 0 or N == 0: nothing to do */
  GEMM_KERNEL_TC2 = 5,      /* two-SM tcgen05 GEMM (CTA pairs, cta_group::2), 256 x 256
                               tiles, whole or with a Stream-K tail; tile_m = tile_n = 256,
                               grid = 2 x pairs; dp_tiles, sk_tiles and the work units
                               count pair tiles and pairs */
  GEMM_KERNEL_SPLITC = 6    /* one-SM tcgen05 GEMM with each tile's k-blocks split over a
                               cluster of cluster_split CTAs, whose fp32 partials are added
                               in distributed shared memory (no global workspace) */
};

/* What gemm_run will launch for a shape.  "MMA view": with swap_ab = 1 the
 * kernel computes Cᵀ = Bᵀ·Aᵀ, so its M side is the problem's N and vice versa. */
typedef struct {
  int32_t kernel;      /* GEMM_KERNEL_* */
  int32_t swap_ab;     /* 1: operands swapped (skinny M), C written transposed */
  int32_t tile_m;      /* CTA tile rows (MMA view): 256 (CTA pairs), 128, or 64 */
  int32_t tile_n;      /* CTA tile columns (MMA view) */
  int32_t tile_k;      /* k-block depth per pipeline stage */
  int32_t stages;      /* shared-memory pipeline stages (k-blocks the ring holds) */
  int32_t grid;        /* CTAs launched */
  int32_t tiles_m;     /* output tiles along the MMA M side */
  int32_t tiles_n;     /* output tiles along the MMA N side */
  int32_t k_iters;     /* k-blocks per output tile = ceil(K / tile_k) */
  int32_t dp_tiles;    /* tiles computed whole, tile c + u*grid by CTA c */
  int32_t sk_tiles;    /* tiles whose k-blocks are split evenly over all CTAs */
  int32_t a_mn_major;  /* MMA-view A operand is M-contiguous (else K-contiguous) */
  int32_t b_mn_major;  /* MMA-view B operand is N-contiguous (else K-contiguous) */
  int32_t group_m;     /* tile raster: groups of group_m tile rows */
  int32_t cluster_split; /* GEMM_KERNEL_SPLITC: CTAs per tile (2, 4 or 8), else 0 */
  int64_t workspace_bytes; /* fp32 partial-tile bytes the split needs */
  int32_t k_group;     /* k-blocks each TMA copy brings (the ring is taken k_group
                          stages at a time); 1 = one copy per operand and k-block */
  int32_t tma_store;   /* 1: row-major output tiles leave by TMA store (where C's base is
                          16-byte aligned and its row pitch a multiple of 16 bytes),
                          0: plain stores (always for gemm_run_noalloc) */
} gemm_plan_t;

/* Options for tests and tuning (gemm_set_option).  Values < 0 restore the default. */
enum {
  GEMM_OPT_FORCE_KERNEL = 0,     /* GEMM_KERNEL_TC / _STREAMK / _SIMT / _TC2 / _SPLITC, or -1 */
  GEMM_OPT_FORCE_TILE_N = 1,     /* 16, 32, 64, 128, 256 (tensor-core path), or -1 */
  GEMM_OPT_FORCE_GRID = 2,       /* CTA count for the split path, or -1 */
  GEMM_OPT_WAIT_LIMIT_NS = 3,    /* bound on each device-side wait (default 2e9 ns); the
                                    clean-up waits after one gave up are bounded by
                                    gemm_drain_limit_ns of it */
  GEMM_OPT_MIN_SPLIT_ITERS = 4,  /* fewest k-blocks per CTA when splitting (default: enough
                                    that a CTA reads 4x its fp32 partial tile in operands) */
  GEMM_OPT_FORCE_SWAP_AB = 5,    /* 0 or 1, or -1 for the picker's choice */
  GEMM_OPT_GROUP_M = 6,          /* tile rows per raster group (default: 4096 rows of A,
                                    16 pair tiles, on the two-SM kernel; 2048 rows, 16
                                    tiles, on the one-SM kernels) */
  GEMM_OPT_PAIR = 7,             /* two-SM kernel: 0 never, 1 whenever the shape allows
                                    (not swapped), -1 the picker's rule */
  GEMM_OPT_CLUSTER_SPLIT = 8,    /* cluster split: 0 never (Stream-K instead), 2/4/8 CTAs
                                    per tile when a split is chosen, -1 the picker's rule */
  GEMM_OPT_PDL = 9,              /* 1 (default): tensor-core kernels are launched so their
                                    prologue may overlap the previous kernel on the stream;
                                    they touch global memory only after it completed. 0: off */
  GEMM_OPT_PAIR_SPLIT = 10,      /* two-SM kernel: -1 (default) or 0 whole tiles only;
                                    1 every tile's k-blocks split evenly over the pairs
                                    (Stream-K); 2 the part-empty last wave of pair tiles and
                                    the wave before it split evenly over the pairs */
  GEMM_OPT_TMA_STORE = 11,       /* row-major output tiles leave the tensor-core kernels by
                                    TMA store when C is 16-byte aligned with a row pitch that
                                    is a multiple of 16 bytes: -1 (default) on launches with
                                    4 (fp32 output) or 10 (fp16 output) or more output tiles
                                    per CTA (per CTA pair on the two-SM kernel), 1 always, 0
                                    never (plain stores) */
  GEMM_OPT_BIAS_INIT = 12,       /* 1: the tensor-core kernels start each tile's fp32
                                    reduction from the bias (seeded into the accumulator
                                    before the first MMA) instead of adding it to the sum;
                                    0 (default): added to the finished fp32 sum */
  GEMM_OPT_DYNAMIC_TILES = 13,   /* two-SM kernel with whole tiles: 1 each pair takes its
                                    next tile from a counter in the handle at run time, so
                                    the tiles in flight stay in raster order (half the
                                    DRAM reads of the static schedule at 16384^3 with
                                    raster groups of 8); 0 (default) the static schedule
                                    gemm_work_units reports (pair c takes tiles c, c +
                                    pairs, ...), measured faster with raster groups of 16
                                    once operands come in two-k-block copies.  The split
                                    tail and the bias seeding always use the static
                                    schedule. */
  GEMM_OPT_STAGES = 14,          /* one-SM tensor-core kernel: shared-memory ring stages.
                                    -1 (default) the picker's: all the ring holds, or, for a
                                    cluster split over more than half the SMs, as many as
                                    let two CTAs share an SM (so the next launch's CTAs
                                    start beside this one's); n >= 1 forced (at most the
                                    ring's size) */
  GEMM_OPT_TILE_M = 15,          /* one-SM tensor-core kernel: rows per tile.  -1 (default)
                                    the picker's: 64 for a small, shallow product taken as
                                    whole tiles when 64-row tiles still fit one wave, else
                                    128; 64 or 128 forced (64: whole tiles, operands not
                                    swapped, tile width 32, 64 or 128) */
  GEMM_OPT_K_GROUP = 16          /* k-blocks per TMA copy on the tensor-core kernels (the
                                    ring's stages are taken that many at a time): -1
                                    (default) the picker's, when K is a multiple of 64 or
                                    both operands are MN-major: up to 4 on the 64-row
                                    kernel, 2 on the two-SM kernel, 2 on the 128-row kernel
                                    when its ring holds 6 k-blocks or more, else 1; 1 to 4
                                    forced (rounded down to what the shape, kernel and ring
                                    allow: at most 3 on the two-SM kernel) */
};

/* Creates a handle on CUDA device `device`.  Allocates, on that device, the
 * Stream-K workspace (fp32 partial tiles, bounded by 2 x SM count tiles of
 * 128 x 256), the per-tile arrival counters and the device status word.
 * The caller's current device is restored before returning.
 * Errors: INVALID_ARG (h NULL, no such device), UNSUPPORTED (device is not
 * compute capability 10.3), ALLOC, CUDA. */
int gemm_create(gemm_handle_t *h, int device);

/* Frees everything gemm_create allocated.  The caller must have synchronised
 * every stream the handle was used on.  NULL is accepted (no-op). */
int gemm_destroy(gemm_handle_t h);

/* Enqueues C = A·B (+bias) on `stream` and returns without waiting.
 * Picks the kernel with the rules gemm_query_plan reports.
 * Alignment: none is required.  fp16 inputs go to the tensor cores (operands
 *   read by TMA) when A and B are 16-byte aligned and each leading dimension
 *   is a multiple of 8 elements; otherwise (and for operands with 2^31 or more
 *   rows or columns) to the CUDA-core kernel, fp16 widened to fp32 with fp32
 *   accumulation, which is much slower.  gemm_query_plan assumes aligned bases.
 * M == 0 or N == 0: nothing is launched.  K == 0: C = bias (or 0).
 * One handle must not run on two streams at once: its workspace is shared.
 * Device-side wait timeouts are not seen here; call gemm_status.
 * Errors: INVALID_ARG (negative size, NULL pointer with non-empty operand,
 * unknown enum), UNSUPPORTED, CUDA (launch failed). */
int gemm_run(gemm_handle_t h, int64_t M, int64_t N, int64_t K, const void *A,
             const void *B, const float *bias, void *C, gemm_layout_t layout,
             void *stream);

/* gemm_run for operands and output in HOST memory.  A, B, bias (NULL or N
 * fp32) and C are host pointers owned by the caller, laid out as for
 * gemm_run.  Enqueued on `stream`, in this order: A, B and bias copied to
 * device buffers the handle owns, gemm_run on them, C copied back.  The call
 * returns once the work is enqueued; C holds the result when the stream has
 * reached that point (gemm_status, or a stream synchronisation).  With
 * page-locked host memory (cudaHostAlloc, or pinned torch tensors) the
 * copies are asynchronous; pageable memory works, but each copy then
 * completes before the call returns.  The device buffers grow to the largest
 * problem seen on the handle (a call that grows them first waits for the
 * handle's previous gemm_run_host call to finish) and are freed by
 * gemm_destroy.  gemm_run_host calls on one handle run in call order
 * whatever their streams: each call's copies wait (on the device) for the
 * previous gemm_run_host call's work, so they never overwrite buffers still
 * in use.  That ordering covers gemm_run_host calls only: a gemm_run on the
 * same handle shares its workspace and counters with no such ordering, so,
 * as for gemm_run, one handle must not run on two streams at once unless the
 * caller orders the streams.  For one step's copies to overlap another's
 * compute, use two handles on two streams.  Not for stream capture.
 * Errors: gemm_run's, ALLOC, and CUDA (a copy, event or stream call failed). */
int gemm_run_host(gemm_handle_t h, int64_t M, int64_t N, int64_t K, const void *A,
                  const void *B, const float *bias, void *C, gemm_layout_t layout,
                  void *stream);

/* Synchronises `stream`, then reads and clears the device status word.
 * Returns GEMM_OK, GEMM_ERR_DEVICE_TIMEOUT (a bounded wait inside a kernel
 * expired; the kernel stopped early and C is unspecified; the handle's
 * counters are reset so the handle stays usable), or GEMM_ERR_CUDA (the
 * stream reported an error). */
int gemm_status(gemm_handle_t h, void *stream);

/* Raw device status word read by the last gemm_status call (0 = none;
 * otherwise 1 + the role whose wait expired: 1 TMA producer, 2 MMA issuer
 * waiting for data, 3 MMA issuer waiting for an accumulator, 4 epilogue,
 * 5 drain, 6 the self-test below). */
int gemm_status_detail(gemm_handle_t h);

/* Failure injection for tests of the error paths: with n > 0, the n-th
 * device allocation this library makes from now on (1 = the next one; in any
 * thread, on any handle) fails as if the device memory were exhausted, so the
 * call that makes it returns GEMM_ERR_ALLOC.  gemm_create makes three (the
 * workspace, the tile counters, the status word) and frees whatever it made
 * before the failure; gemm_run_host makes one when its buffers grow, and the
 * handle stays usable (its buffers are then empty and grow on the next call).
 * n == 0 disarms.  gemm_run_noalloc makes no allocation and is not affected.
 * Errors: INVALID_ARG (n < 0). */
int gemm_inject_alloc_failure(int64_t n);

/* Phase tracing for the tensor-core kernels.  dev_buf: NULL (tracing off) or a
 * caller-owned DEVICE buffer of ctas x 12 uint64 values; while set, every
 * tensor-core launch whose grid fits in `ctas` CTAs writes, for CTA i,
 * %globaltimer nanoseconds to dev_buf[12*i + p] at phase p: 8 kernel entry,
 * 0 setup done (barriers, TMEM, the wait for the previous kernel on the
 * stream), 1 first TMA load issued, 2 first stage landed (MMA issuer), 3 last
 * accumulator committed, 4 last accumulator received by the epilogue,
 * 5 epilogue done, 10 cluster split: every CTA of the cluster parked its
 * partial, 11 cluster split: this CTA's share of the reduction stored (by
 * thread 64), 7 cluster split: the whole cluster done, 9 TMEM freed (about to
 * return); slot 6 holds the CTA's work-unit count.  Slots a CTA
 * never reaches (e.g. the MMA slots of the second CTA of a pair) are not
 * written.  Launches with more CTAs than `ctas` are not traced.
 * Errors: INVALID_ARG. */
int gemm_set_trace(gemm_handle_t h, uint64_t *dev_buf, int64_t ctas);

/* Failure-path self-test: enqueues one CTA whose wait on an mbarrier that
 * nothing completes gives up after limit_ns nanoseconds, records the expiry
 * in the device status word and returns normally (no trap, no fault).  The
 * next gemm_status call on `stream` must report GEMM_ERR_DEVICE_TIMEOUT with
 * detail 6; the handle stays usable.  Errors: INVALID_ARG, CUDA. */
int gemm_selftest_wait_timeout(gemm_handle_t h, int64_t limit_ns, void *stream);

/* C = A·B (+bias) for callers that cannot allocate device memory.
 * (The pages have no counterpart to this entry point.)
 *
 * Some callers cannot call cudaMalloc: a plugin inside a host application whose
 * own caching allocator has reserved the device memory (an outside cudaMalloc
 * may fail, or bypasses that allocator's accounting), or a latency-critical
 * path where cudaMalloc/cudaFree would synchronise the device.  gemm_create
 * allocates; this call does not, and needs no handle.  It runs the same
 * tensor-core kernel and picker as gemm_run, with the split path's scratch in
 * a fixed array compiled into the library: 16 MiB of fp32 partial tiles, 4096
 * split-tile counters and one status word.  Every GPU that loads the library
 * holds that array until the process exits.
 *
 * Arguments are gemm_run's, minus the handle: A, B, bias, C are device pointers
 * on the CURRENT device, owned by the caller; stream belongs to that device.
 * dev_status: NULL, or a device int the caller owns that the kernel sets to a
 * nonzero site code (as gemm_status_detail reports) if a bounded device-side
 * wait expires; the caller clears it.  With NULL a timeout CANNOT be detected:
 * the kernel stops early, C is incomplete, and nothing reports it (the expiry
 * goes to a word inside the array, which each such call clears before its
 * kernel and nothing reads).  Pass a status word wherever a wrong C matters.
 *
 * The first call on a device looks up the array's device address with that
 * device current (cudaGetSymbolAddress) and caches it; make that first call
 * before any stream capture.  Calls never call cudaMalloc, cudaFree or any
 * allocating routine.
 *
 * All calls share the one array, which keeps the last call's contents; each
 * call clears the counters it uses (cudaMemsetAsync on `stream`) before its
 * kernel.  Calls whose kernels overlap on the GPU (different streams, no
 * ordering between them) race on the array and give wrong results: order them.
 *
 * Limits: fp16 inputs only (fp32 inputs return GEMM_ERR_UNSUPPORTED; use
 * gemm_run).  A Stream-K split whose partial tiles exceed 16 MiB runs on fewer
 * CTAs so that they fit; a Stream-K split over more than 4096 output tiles is
 * refused with GEMM_ERR_UNSUPPORTED (the counters would not fit).  Cluster
 * splits and whole-tile plans use neither.  Other errors as gemm_run:
 * INVALID_ARG, UNSUPPORTED (alignment, device not compute capability 10.3),
 * CUDA. */
int gemm_run_noalloc(int64_t M, int64_t N, int64_t K, const void *A, const void *B,
                     const float *bias, void *C, gemm_layout_t layout, void *stream,
                     int *dev_status);

/* Sets an option (GEMM_OPT_*) on the handle. Errors: INVALID_ARG. */
int gemm_set_option(gemm_handle_t h, int option, int64_t value);

/* Fills *out with the plan gemm_run would launch for this shape on the
 * handle's device with its current options.  Errors as gemm_run's checks. */
int gemm_query_plan(gemm_handle_t h, int64_t M, int64_t N, int64_t K,
                    gemm_layout_t layout, gemm_plan_t *out);

/* Human-readable name of a gemm_status_t (static storage). */
const char *gemm_strerror(int code);

/* ---- Host-only functions: need no GPU, no handle. ---------------------- */

/* The tile picker for a device with `num_sms` SMs and default options. */
int gemm_plan_for(int64_t M, int64_t N, int64_t K, gemm_layout_t layout,
                  int num_sms, gemm_plan_t *out);

/* The work units CTA `cta` of `plan` processes, in order: writes up to
 * `max_units` triples (tile, k_begin, k_end) to out (3 int32 each) and returns
 * the count (which may exceed max_units), or a negative gemm_status_t. */
int gemm_work_units(const gemm_plan_t *plan, int cta, int32_t *out, int max_units);

/* For split tile `sk_tile` (0-based within the split region): the first and
 * last contributing CTA, in ascending k order.  Returns 0 or INVALID_ARG. */
int gemm_split_contributors(const gemm_plan_t *plan, int sk_tile, int32_t *first,
                            int32_t *last);

/* The bound on the clean-up waits of a kernel whose device-side wait gave up
 * (its TMA copies and MMAs still in flight must land before it frees its TMEM
 * and exits), for a GEMM_OPT_WAIT_LIMIT_NS of wait_limit_ns (<= 0: the
 * default): the limit itself, but never less than one second, so that a limit
 * short enough to stop a launch early cannot also cut its clean-up short. */
int64_t gemm_drain_limit_ns(int64_t wait_limit_ns);

/* Shared-memory row strides (in floats) of the fp32 CUDA-core kernel's A and B
 * staging tiles, padded as storage_align(factor 32, offset 4) pads them. */
int gemm_simt_smem_strides(int32_t *a_stride, int32_t *b_stride);

#ifdef __cplusplus
}
#endif
#endif /* DGEMM_GB300_GEMM_H_ */
