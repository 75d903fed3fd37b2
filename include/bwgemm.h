/*
 * bwgemm.h -- C ABI of the GB300 (sm_103a) dense GEMM library libbwgemm.so.
 *
 * The operation (the one all the source pages build):
 *
 *     C[M x N] = A[M x K] * B[N x K]^T
 *
 *   A, B : bf16 or fp16, both stored K-major (row-major A; B stored N x K,
 *          i.e. "B already transposed" -- "Matrix Multiplication on NVIDIA's
 *          Blackwell", optimisation roadmap section and the naive Kernel 1,
 *          which reads b[col, k]).
 *   accumulation in fp32 ("BF16 in and out, converted to FP32 to accumulate",
 *          same page, Kernel 1 section; the CuTeDSL post's K-loop,
 *          "Writing a Blackwell GEMM by hand", step 1 equation).
 *   C    : same type as A and B, rounded to nearest even from fp32.
 *
 * All sizes and leading dimensions are in elements.  Matrices are row-major
 * with row strides lda / ldb / ldc (lda >= K, ldb >= K, ldc >= N).
 *
 * Alignment (the TMA rules the kernels rely on): A, B, C 16-byte aligned;
 * lda, ldb, ldc multiples of 8 elements.  Violations return
 * BWGEMM_ERR_ALIGNMENT; nothing is launched.
 *
 * Threading: a plan may be used from one host thread at a time and on one
 * stream at a time (its split-K workspace and status word are shared by its
 * launches).  Different plans are independent.
 *
 * Nothing is thrown across this boundary; every entry point returns a status.
 */
#ifndef BWGEMM_H
#define BWGEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define BWGEMM_VERSION_MAJOR 0
#define BWGEMM_VERSION_MINOR 2

/* Regions of the fixed device array behind bwgemm_run_splitk_noalloc. */
#define BWGEMM_NOALLOC_PARTIAL_BYTES (8u << 20) /* fp32 partial tiles of the K slices */
#define BWGEMM_NOALLOC_COUNTER_BYTES (64u << 10) /* 32-bit arrival counters           */

typedef struct bwgemm_plan_s* bwgemm_plan_t;

typedef enum {
    BWGEMM_BF16 = 0, /* bfloat16 inputs and output */
    BWGEMM_FP16 = 1  /* IEEE binary16 inputs and output */
} bwgemm_dtype_t;

typedef enum {
    BWGEMM_OK = 0,
    BWGEMM_ERR_INVALID_ARG = 1, /* bad size, stride, dtype, NULL pointer or handle      */
    BWGEMM_ERR_ALIGNMENT = 2,   /* pointer not 16-byte aligned or ld not a multiple of 8 */
    BWGEMM_ERR_UNSUPPORTED = 3, /* device is not sm_103 / size beyond the supported range */
    BWGEMM_ERR_NO_DEVICE = 4,   /* no CUDA device / driver                                */
    BWGEMM_ERR_CUDA = 5,        /* a CUDA runtime or driver call failed                   */
    BWGEMM_ERR_TIMEOUT = 6,     /* a device-side wait ran out (see bwgemm_get_status)     */
    BWGEMM_ERR_WORKSPACE = 7    /* split-K workspace too small for the forced options     */
} bwgemm_status_t;

typedef enum {
    BWGEMM_VARIANT_AUTO = 0, /* choose from the shape                                  */
    BWGEMM_VARIANT_1SM = 1,  /* one CTA per tile: 128 x BN tiles, tcgen05 cta_group::1 */
    BWGEMM_VARIANT_2SM = 2   /* CTA pair per tile: 256 x BN tiles, cta_group::2        */
} bwgemm_variant_t;

typedef enum {
    BWGEMM_SCHEDULE_AUTO = 0,     /* stream-K when whole tiles leave workers idle         */
    BWGEMM_SCHEDULE_TILES = 1,    /* whole tiles, or split_k slices of every tile          */
    BWGEMM_SCHEDULE_STREAM_K = 2, /* K iterations of the last tiles divided evenly among
                                     the workers; the earlier full waves as whole tiles    */
    BWGEMM_SCHEDULE_CLC = 3       /* whole tiles, one cluster per tile in the grid; running
                                     clusters take over the tiles of clusters not yet
                                     launched through cluster launch control               */
} bwgemm_schedule_t;

/* Plan options.  Zero means "choose automatically" for every field; get the
 * defaults with bwgemm_default_options(). */
typedef struct {
    int32_t variant;          /* bwgemm_variant_t                                       */
    int32_t tile_n;           /* 0 = auto, 64, 128, 224, 256, 320 or 384: columns per
                                 work unit (224, 320, 384: CTA-pair form, operands not
                                 swapped, no multicast; 320 and 384 issue two MMAs,
                                 N = 256 and N = tile_n - 256, into one accumulator)    */
    int32_t split_k;          /* 0 = auto, 1 = off, s >= 2: s K-slices per tile         */
    int32_t raster_group;     /* 0 = auto; m-blocks walked before stepping along N      */
    int32_t max_ctas;         /* 0 = fill the GPU; else cap on the persistent grid      */
    int32_t stall_kblock;     /* test hook, keep -1: the producer of CTA 0 never fills
                                 this k-block of its first unit, so a bounded wait runs
                                 out and the call reports BWGEMM_ERR_TIMEOUT            */
    uint64_t timeout_ns;      /* bound on every device-side wait; 0 = 4 s               */
    uint64_t workspace_bytes; /* split-K / stream-K workspace of the plan; 0 = 64 MiB   */
    int32_t schedule;         /* bwgemm_schedule_t                                       */
    int32_t pdl_off;          /* nonzero: launch without programmatic dependent launch  */
    int32_t trace;            /* nonzero: record a per-CTA timeline of every launch
                                 (read back with bwgemm_plan_read_trace)                */
    int32_t prefetch;         /* K blocks of the streamed operand (the one with more
                                 rows) prefetched into L2 ahead of the shared-memory
                                 loads: 0 or -1 = none (measured slower on every shape),
                                 n = n K blocks ahead                                    */
    int32_t swap_ab;          /* 0 = auto, 1 = never, 2 = always: compute C^T = B A^T so
                                 that B's rows fill the 128-row MMA side (small M)       */
    int32_t multicast;        /* 0 = auto, 1 = off, 2 = on: clusters of two CTA pairs on
                                 adjacent column blocks; each A tile is read from L2
                                 once and multicast to both pairs (CTA-pair variant,
                                 operands not swapped)                                   */
    int32_t copy_kblocks;     /* K blocks per TMA operand copy: 0 = auto (two for
                                 compute-bound shapes, four in the whole-K kernel),
                                 1 = one, 2 = two (where K holds at least two whole
                                 64-element chunks; either selects the main kernel)      */
    int32_t cluster_split;    /* 0 = auto, 1 = off, 2 = required: the two K slices of a
                                 one-wave split-K tile run in one cluster and exchange
                                 partials through distributed shared memory (when a
                                 cluster per tile fits at once)                          */
    int32_t tuned_table;      /* 0 = apply the library's table of tuned options when the
                                 shape matches one of its entries exactly and every
                                 option the entry sets is left automatic, 1 = plan
                                 from the rules alone                                   */
    int32_t skinny;           /* 0 = auto, 1 = off, 2 = required: for at most 64 rows of A
                                 (operands swapped) and ceil(N / 64) <= SMs, the whole-K
                                 kernel with 64 weight rows per CTA (MMA M = 64) and no
                                 split of K; auto takes it unless another option asks
                                 for something only the main kernel does              */
    int32_t wholek;           /* 0 = auto, 1 = off, 2 = required: for 129 to 256 rows of
                                 A (operands not swapped), the whole-K kernel on CTA
                                 pairs with all rows of A on the MMA's M side (256 over
                                 the pair) and a block of weight rows (96-192) sized so
                                 that the blocks fill the pairs once, no split of K;
                                 auto takes it where the main kernel would use a pair
                                 tile wider than 256 columns and no other option asks
                                 for the main kernel                                  */
    int32_t reserved[1];      /* must be zero                                            */
} bwgemm_plan_options_t;

/* The launch configuration chosen for a shape (for inspection and tests). */
typedef struct {
    int32_t variant;      /* BWGEMM_VARIANT_1SM or BWGEMM_VARIANT_2SM            */
    int32_t tile_m;       /* rows of C per work unit (128 or 256)                */
    int32_t tile_n;       /* columns of C per work unit                          */
    int32_t tile_k;       /* K elements per pipeline stage (64)                  */
    int32_t stages;       /* depth of the shared-memory ring                     */
    int32_t split_k;      /* K slices per tile (1 = none)                        */
    int32_t raster_group; /* m-blocks per raster group                           */
    int32_t num_tiles;    /* output tiles                                        */
    int32_t num_units;    /* whole-tile / split-K units (dp_tiles x split_k)     */
    int32_t grid;         /* CTAs launched (persistent, or one cluster per tile
                             with BWGEMM_SCHEDULE_CLC)                           */
    int64_t workspace_bytes; /* partial-tile bytes used by this shape            */
    int32_t schedule;     /* BWGEMM_SCHEDULE_TILES, _STREAM_K or _CLC            */
    int32_t dp_tiles;     /* tiles computed whole (or as split_k slices)         */
    int32_t sk_tiles;     /* tiles whose K iterations are spread by stream-K     */
    int32_t workers;      /* clusters (CTAs, CTA pairs or pairs of pairs) of the
                             persistent grid                                     */
    int32_t split_scatter; /* 1: the split_k slices of each tile run in one wave
                              and reduce-scatter their partials                  */
    int32_t swap_ab;      /* 1: operands swapped (tiles over C^T: tile_m along N,
                             tile_n along M)                                     */
    int32_t multicast;    /* CTA pairs per cluster sharing each A tile (1 or 2);
                             a tile then spans tile_n x multicast columns        */
    int32_t copy_kblocks; /* K blocks per TMA operand copy (1 or 2; 2 applies
                             where K holds at least two whole 64-element chunks;
                             the whole-K kernel: 4 where K holds four, else 1)   */
    int32_t prefetch_kblocks; /* L2 prefetch distance of the streamed operand (0: off) */
    int32_t prefetch_b;   /* the streamed operand: 1 = B (the kernel's), 0 = A   */
    int32_t cluster_split; /* 1: split_k = 2 slices per tile inside one cluster,
                              partials exchanged in distributed shared memory    */
    int32_t tuned;         /* 1: an entry of the tuned-options table was applied */
    int32_t skinny;        /* 1: the whole-K kernel for a few rows of A (tile_m =
                              64 weight rows per CTA, tile_n = the MMA's N)      */
    int32_t wholek;        /* 1: the whole-K pair kernel for 129-256 rows of A
                              (tile_m = 256, tile_n = weight rows per pair)      */
} bwgemm_config_t;

/* Fill *opts with the defaults (all automatic, stall_kblock = -1). */
void bwgemm_default_options(bwgemm_plan_options_t* opts);

/*
 * Create a plan on CUDA device `device` (an ordinal; the library makes it
 * current for the calls it makes).  Checks that the device is compute
 * capability 10.3 (sm_103) and returns BWGEMM_ERR_UNSUPPORTED otherwise --
 * there is no fallback path.  Allocates the plan's device status word and
 * split-K workspace.  `opts` may be NULL (defaults).  On failure *plan is NULL.
 */
bwgemm_status_t bwgemm_create_plan(bwgemm_plan_t* plan, int device,
                                   const bwgemm_plan_options_t* opts);

/* Free a plan and its device memory.  NULL is accepted.  Synchronises the
 * device first, so no launch of the plan may still be running. */
bwgemm_status_t bwgemm_destroy(bwgemm_plan_t plan);

/*
 * C = A * B^T on `stream` (a cudaStream_t; NULL = the legacy default stream).
 *
 *   A : device pointer, M x K, row stride lda (read only)
 *   B : device pointer, N x K, row stride ldb (read only; may alias A)
 *   C : device pointer, M x N, row stride ldc (written; must not overlap A or B)
 *
 * A, B and C must be device (or managed) memory of the plan's device: an
 * operand in host memory or on another GPU is refused with
 * BWGEMM_ERR_INVALID_ARG before anything is encoded or launched (A and B are
 * not checked when K == 0).  The caller owns A, B and C and keeps them alive
 * until the stream reaches the launch.  Asynchronous: returns after enqueueing one kernel (none when
 * M == 0 or N == 0; a zero fill of C when K == 0, the empty sum).  No host
 * synchronisation and no device allocation, so it may be captured in a CUDA
 * graph.  Argument errors are returned synchronously and launch nothing.
 * Device-side timeouts are reported by bwgemm_get_status().
 */
bwgemm_status_t bwgemm_run(bwgemm_plan_t plan, const void* A, const void* B, void* C, int64_t M,
                           int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                           bwgemm_dtype_t dtype, void* stream);

/*
 * Same product with HOST operands: copies A and B (host memory, pinned for
 * full speed) to plan-owned device buffers, runs the GEMM, copies C back to
 * host memory, and synchronises `stream` before returning.  The device
 * buffers grow on demand and are kept for later calls.  Returns the device
 * status of the launch (as bwgemm_get_status would).
 */
bwgemm_status_t bwgemm_run_host(bwgemm_plan_t plan, const void* A_host, const void* B_host,
                                void* C_host, int64_t M, int64_t N, int64_t K, int64_t lda,
                                int64_t ldb, int64_t ldc, bwgemm_dtype_t dtype, void* stream);

/*
 * Synchronise `stream`, then read and clear the plan's device status word:
 * BWGEMM_OK, or BWGEMM_ERR_TIMEOUT when a bounded device-side wait of an
 * earlier launch ran out (that launch's C is then undefined), or
 * BWGEMM_ERR_CUDA.  Clearing also re-arms the split-K turn counters.
 */
bwgemm_status_t bwgemm_get_status(bwgemm_plan_t plan, void* stream);

/*
 * Raw device status bits of the last bwgemm_get_status() call (0 = fine):
 * 1, 2, 4, 8 = a bounded wait of the producer, the MMA warp, the epilogue or
 * the split-K exchange ran out; 16 = a kernel variant was handed a unit it
 * cannot run (a ring-staged or clustered split-K variant given a second or a
 * non-split unit: a planning error, never produced by the planner).  Any bit
 * makes bwgemm_get_status return BWGEMM_ERR_TIMEOUT.
 */
uint32_t bwgemm_last_device_status(bwgemm_plan_t plan);

/*
 * Host-only argument check of a bwgemm_run() call (no device access):
 * returns the status bwgemm_run would return for these arguments before
 * launching anything.
 */
bwgemm_status_t bwgemm_check_args(const void* A, const void* B, const void* C, int64_t M,
                                  int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                                  bwgemm_dtype_t dtype);

/*
 * Host-only: the configuration a plan with `opts` (NULL = defaults) would
 * pick for this shape on a GPU with `num_sms` SMs that can hold
 * `max_pairs` co-resident CTA pairs (0 = num_sms / 2) and `max_quads`
 * co-resident clusters of two pairs (0 = max_pairs / 2; the multicast form
 * and the clustered split-K).  No device access.
 */
bwgemm_status_t bwgemm_select_config(int32_t num_sms, int32_t max_pairs, int32_t max_quads,
                                     int64_t M, int64_t N, int64_t K, bwgemm_dtype_t dtype,
                                     const bwgemm_plan_options_t* opts, bwgemm_config_t* out);

/* The configuration of the plan's most recent bwgemm_run / bwgemm_run_host. */
bwgemm_status_t bwgemm_plan_last_config(bwgemm_plan_t plan, bwgemm_config_t* out);

/*
 * Timeline of the plan's most recent launch (plans created with opts.trace):
 * synchronises the device, then copies ctas x slots %globaltimer stamps
 * (nanoseconds; 0 = not reached) into `out`, row per CTA.  Slots: 0 kernel
 * entry, 1 prologue and dependency wait done, 2 first TMA load issued,
 * 3 last TMA load issued, 4 epilogue finished, 5 exit, 6 barriers, TMEM and
 * the prologue's cluster barrier done, 7 producer's first unit worked out
 * (before the dependency wait); from slot 8 on, four
 * per work unit (at most 14 units): MMA start, MMA end, epilogue start,
 * epilogue end.  *ctas and *slots receive the dimensions; `capacity` is the
 * size of `out` in elements.  BWGEMM_ERR_INVALID_ARG if tracing is off or
 * `out` is too small.  Each CTA clears its own row as it starts, so tracing
 * adds nothing to the stream between launches; two launches of one traced
 * plan that overlap (programmatic dependent launch) write the same rows, so
 * for a timeline of back-to-back launches alternate two traced plans.
 */
bwgemm_status_t bwgemm_plan_read_trace(bwgemm_plan_t plan, uint64_t* out, int64_t capacity,
                                       int32_t* ctas, int32_t* slots);

/* Number of GEMM kernels the plan has enqueued since it was created. */
uint64_t bwgemm_plan_launch_count(bwgemm_plan_t plan);

/*
 * Dense tensor-pipe rate of one SM, measured: one CTA per SM of `device`
 * issues 4096 tcgen05.mma (M = 128, N = 256, K = 16, bf16 in, fp32 in TMEM)
 * on operands held in shared memory and times them in SM cycles.  Writes
 * the median FLOP per SM clock to *flop_per_clock_per_sm and the device's
 * SM count to *sm_count, from which a nominal dense peak is
 * SMs x rate x clock ("Matrix Multiplication on NVIDIA's Blackwell",
 * Kernel 2, and the CuTeDSL post's MMA step define the instruction; the
 * pages state no per-SM rate).  Synchronises the device.  Errors:
 * BWGEMM_ERR_INVALID_ARG (NULL output), BWGEMM_ERR_NO_DEVICE,
 * BWGEMM_ERR_UNSUPPORTED (not sm_103), BWGEMM_ERR_CUDA, BWGEMM_ERR_TIMEOUT
 * (the bounded wait for the MMAs ran out).
 */
bwgemm_status_t bwgemm_probe_tensor_rate(int device, double* flop_per_clock_per_sm, int32_t* sm_count);

/*
 * Load-path microbenchmark ("Writing a Blackwell GEMM by hand", step 4: a
 * benchmark that isolates the load path, with no MMA, moving the same bytes
 * with the same copies and changing only the shared-memory layout).  `ctas`
 * CTAs (0 = one per SM of `device`; at most one per SM) run the GEMM's ring
 * of `stages` (1..6) stages of 32 KiB: per K block the producer copies a
 * 128-row x 64-element bf16 tile of A and one of B by TMA and a consumer
 * warp frees the stage as soon as it lands, for `kblocks` (1..2^20) K blocks
 * per CTA.  `source`: 0 = a 16 MiB matrix that stays in L2 (the L2 ->
 * shared-memory path), 1 = a 2 GiB matrix of which every CTA streams rows
 * of its own (the HBM -> shared-memory path; 256 K blocks per row block
 * before a CTA wraps).  `layout`: 0 = 128B swizzle (the GEMM's layout, one
 * copy of box {64, 128} per tile), 1 = no swizzle with the same copies
 * (plain 128-byte rows), 2 = no swizzle in the tensor cores' interleaved
 * K-major layout (8 x 16-byte core matrices, eight copies of box {8, 128}
 * per tile), 3 = 128B swizzle with one copy of box {64, 256} per K block
 * (the same bytes in half the copies), 4 = 128B swizzle in clusters of two
 * CTAs that share A: each copies half of the A tile with cluster multicast
 * into both and its own B tile (the same bytes landed, three quarters
 * issued; an even number of CTAs), 5 = 128B swizzle, two K blocks of one
 * 128-row block per copy (box {64, 128, 2} of a 3-D view: 256 contiguous
 * bytes of each row; A only), 6 = 128B swizzle, stages of two K blocks of
 * A and B (64 KiB, `stages` at most 3) in clusters of two CTAs sharing A:
 * each copies half of A's rows (box {64, 64, 2}) with cluster multicast and
 * its own B (box {64, 128, 2}), 7 = the same stages without multicast.  For
 * layouts 6 and 7 `kblocks` counts stages of two K blocks.  Writes the
 * bytes landed by all CTAs per second (GB/s, one
 * timed launch after a warm-up launch, CUDA events) to *gbytes_per_s and the
 * launch's time to *ms.  Allocates and frees its source matrix; synchronises
 * the device.  Errors: BWGEMM_ERR_INVALID_ARG (NULL output or an argument
 * out of range, more CTAs than SMs), BWGEMM_ERR_NO_DEVICE,
 * BWGEMM_ERR_UNSUPPORTED (not sm_103), BWGEMM_ERR_CUDA, BWGEMM_ERR_TIMEOUT (a
 * bounded wait ran out).
 */
bwgemm_status_t bwgemm_bench_load_path(int device, int32_t layout, int32_t source, int32_t ctas,
                                       int32_t stages, int32_t kblocks, double* gbytes_per_s,
                                       double* ms);

/*
 * Shape-keyed tuning ("Matrix Multiplication on NVIDIA's Blackwell", the
 * Gemma-shape experiment, chooses pipeline and MMA shapes per shape with an
 * autotuner).  Times a fixed list of candidate configurations -- the plan's
 * options with the schedule, split-K slices, variant, tile width, K blocks
 * per copy, clustered split, raster group or operand order overridden -- on
 * the caller's A, B and C (the same arguments and rules as bwgemm_run), each
 * for `iters` launches (1..10000) after two warm-up launches, timed with CUDA
 * events on `stream`.  Candidates that fail to plan, plan to a configuration
 * already tried, or report a device-side error are skipped.  The fastest is
 * recorded in the plan for this (M, N, K, dtype): later bwgemm_run /
 * bwgemm_run_host calls with that shape use it.  C is left holding the
 * chosen configuration's result (every candidate computes the same C).
 * Synchronises `stream`.  *best (may be NULL) receives the chosen
 * configuration.  Not thread-safe with other calls on the same plan.
 * The timing is back to back on the caller's operands, which stay in L2
 * when they are smaller than it: the choice is the fastest for multiplying
 * those operands repeatedly, not necessarily for operands streamed from HBM.
 * (The library's own table of tuned options comes from a sweep that
 * re-times each choice in steady state on rotated inputs.)
 */
bwgemm_status_t bwgemm_tune(bwgemm_plan_t plan, const void* A, const void* B, void* C, int64_t M,
                            int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                            bwgemm_dtype_t dtype, void* stream, int32_t iters, bwgemm_config_t* best);

/* Number of shapes the plan holds tuned options for. */
int32_t bwgemm_plan_tuned_count(bwgemm_plan_t plan);

/*
 * C = A * B^T with split-K, allocating no device memory (the source pages
 * have no counterpart to this entry point).
 *
 * For callers that cannot call cudaMalloc -- code running under a memory
 * manager that has already reserved the device's memory, code whose device
 * footprint must stay fixed after start-up, or loops that must not risk the
 * device-wide synchronisation cudaMalloc / cudaFree can cause -- and so
 * cannot create a plan.  Needs no plan: the split-K scratch (fp32 partial
 * tiles, arrival counters, a status word) lives in one fixed device array of
 * BWGEMM_NOALLOC_PARTIAL_BYTES + BWGEMM_NOALLOC_COUNTER_BYTES + 256 B inside
 * the library, present on every GPU that loads it until the process exits.
 *
 *   A, B, C, M, N, K, lda, ldb, ldc, dtype : as for bwgemm_run (caller-owned
 *          pointers, device or managed memory of the current device; same
 *          alignment rules and error codes)
 *   split_k : K slices per output tile, 2..16 (capped at the number of
 *          64-wide K blocks; with one K block the call runs unsplit and uses
 *          no partials or counters); the partial tiles of all slices must
 *          fit the partial region (tiles x split_k x 128 KiB for the
 *          256-column tiles) and their arrival counters the counter region,
 *          else BWGEMM_ERR_WORKSPACE is returned and nothing is launched
 *          (bwgemm_noalloc_scratch answers this on the host beforehand)
 *   stream : cudaStream_t (NULL = legacy default stream)
 *
 * The first call on a device (with that device current) resolves the
 * array's device address and occupancy limits; make that first call before
 * any stream capture.  Every call shares the array, which keeps the previous
 * call's contents; each call clears the counters and status word it uses on
 * `stream` first.  Calls whose kernels may overlap on the GPU (other streams,
 * other host threads) race on the array: serialise them.  Device-side wait
 * timeouts of this entry point are not reported (there is no plan to hold
 * the status); use the plan API when that matters.
 */
bwgemm_status_t bwgemm_run_splitk_noalloc(const void* A, const void* B, void* C, int64_t M,
                                          int64_t N, int64_t K, int64_t lda, int64_t ldb,
                                          int64_t ldc, bwgemm_dtype_t dtype, int32_t split_k,
                                          void* stream);

/*
 * Host-only (no device access): the parts of the fixed array that
 * bwgemm_run_splitk_noalloc would use for these sizes on a GPU with
 * `num_sms` SMs holding `max_pairs` co-resident CTA pairs (0 = num_sms / 2).
 * *partial_bytes and *counter_bytes receive the bytes of the partial-tile
 * and counter regions the call writes (both 0 when it runs unsplit or
 * launches nothing).  Returns BWGEMM_ERR_WORKSPACE (the sizes still filled
 * in) when they exceed BWGEMM_NOALLOC_PARTIAL_BYTES or
 * BWGEMM_NOALLOC_COUNTER_BYTES, BWGEMM_ERR_INVALID_ARG for a NULL output,
 * negative sizes or split_k outside 2..16.
 */
bwgemm_status_t bwgemm_noalloc_scratch(int32_t num_sms, int32_t max_pairs, int64_t M, int64_t N,
                                       int64_t K, int32_t split_k, uint64_t* partial_bytes,
                                       uint64_t* counter_bytes);

/* Static text for a status code ("unknown status" for anything else). */
const char* bwgemm_status_string(bwgemm_status_t status);

/* Library version as (major << 16) | minor. */
int32_t bwgemm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* BWGEMM_H */
