/*
 * clcgemm — C ABI of a GB300 (sm_103a) bf16 GEMM whose output tiles are scheduled at run
 * time by Cluster Launch Control work stealing, with static-persistent and non-persistent
 * modes of the same kernel for comparison.
 *
 * Operation (all entry points):  C = A * B
 *   A  bf16, M x K, row-major (element (i, k) at A[i*K + k])
 *   B  bf16, K x N, row-major (element (k, j) at B[k*N + j])
 *   C  fp32, M x N, row-major; every element is the sum over k of A[i][k]*B[k][j]
 *      accumulated in fp32 by the tensor cores (summation order is the hardware's).
 * The pages this follows ("CUTLASS CLC dynamic persistent kernel", section "From one tile
 * per block to one worker working continuously") fix each task as one complete output
 * tile of a GEMM, with no split-K or Stream-K; the scheduling modes change who computes
 * a tile, never its value.
 *
 * Conventions shared by every call:
 *   - Return value: GEMM_OK (0) or a negative GEMM_ERR_* code; gemm_strerror() names it.
 *   - Pointers named "device" are CUDA device pointers owned by the caller; "host"
 *     pointers are ordinary (preferably pinned) host memory owned by the caller.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *     Runs are asynchronous on that stream; device-side failures (a wait that ran out
 *     of time) are reported by gemm_sync().
 *   - A handle is bound to one device and is not thread-safe.  It owns its workspace
 *     (ownership log, error word, trace buffer, grouped-problem tables, staging buffers
 *     for gemm_run_host) and frees it in gemm_destroy().  A run that needs more
 *     workspace than earlier runs grows it, and growing synchronises the device first
 *     (it waits for every stream, including kernels of other libraries).
 *   - Shape rules: M, N, K >= 0; K and N multiples of 8 and all pointers 16-byte aligned
 *     (TMA needs 16-byte row strides and base addresses).  M, N and K need NOT be
 *     multiples of the tile: partial tiles are zero-filled on load and clipped on store.
 *     M == 0 or N == 0 is a no-op; K == 0 writes C = 0.
 */
#ifndef CLCGEMM_H
#define CLCGEMM_H

#include <stdint.h>

#if defined(__GNUC__)
#define CLCGEMM_API __attribute__((visibility("default")))
#else
#define CLCGEMM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- error codes */
#define GEMM_OK                       0
#define GEMM_ERR_INVALID_ARG         -1  /* null pointer, bad enum, bad tile/cluster, negative size */
#define GEMM_ERR_UNSUPPORTED_DEVICE  -2  /* device is not compute capability 10.3 */
#define GEMM_ERR_ALIGNMENT           -3  /* pointer not 16-byte aligned, or K / N not a multiple of 8 */
#define GEMM_ERR_LAUNCH              -4  /* the kernel launch was refused */
#define GEMM_ERR_TIMEOUT             -5  /* a device-side wait exceeded its bound (see gemm_sync) */
#define GEMM_ERR_OOM                 -6  /* workspace allocation failed */
#define GEMM_ERR_CUDA                -7  /* another CUDA runtime / driver error */
#define GEMM_ERR_NO_DEVICE           -8  /* no CUDA device / driver in this process */
#define GEMM_ERR_TOO_LARGE           -9  /* a tile or worker count exceeds 2^31 - 1 */
#define GEMM_ERR_SCRATCH_LIMIT      -10  /* gemm_run_noalloc: more tiles or workers than its fixed scratch holds */
#define GEMM_ERR_MULTICAST          -11  /* a cluster shape that loads operands by TMA multicast was asked for
                                            where it is not allowed: the handle was created with
                                            multicast = 0, or the process sees more than one GPU */
#define GEMM_ERR_BOUNDS             -12  /* library built with bounds checks: a tile coordinate fell outside
                                            its problem; the tile was skipped (see gemm_sync) */

/* ---------------------------------------------------------------- types */
typedef struct gemm_handle *gemm_handle_t;

/* Tile schedulers ("CUTLASS CLC dynamic persistent kernel", table in section "From one
 * tile per block to one worker working continuously"):
 *   CLC            grid over all tiles; a running worker takes the next tile by cancelling
 *                  a cluster launch that has not started (clusterlaunchcontrol.try_cancel);
 *                  it stops at the first failed cancel.
 *   STATIC         grid over `num_workers` workers; worker w computes tiles w, w+W, ...
 *   NONPERSISTENT  grid over all tiles; each CTA computes its own tile and exits. */
typedef enum {
    GEMM_SCHED_CLC = 0,
    GEMM_SCHED_STATIC = 1,
    GEMM_SCHED_NONPERSISTENT = 2
} gemm_sched_t;

/* Output tile per CTA and cluster shape.  Supported: {128, 256, 64} and {128, 128, 64} with
 * cluster {1,1,1}; {128, 256, 64} with cluster {2,1,1} (a 256 x 256 tile per cluster,
 * computed by a CTA-pair MMA, or with gemm_opts_t.cluster_b_multicast by two 128 x 256
 * MMAs sharing B) and with cluster {4,1,1} (a 512 x 256 tile per cluster: four CTAs on
 * consecutive row blocks, each loading a quarter of the B tile and multicasting it to
 * the others) and with cluster {2,2,1} (a 256 x 512 tile per cluster: four CTAs, each on
 * one 128 x 256 quarter; the two CTAs of a row share their A tile and the two of a column
 * their B tile, each loading half and multicasting it).  A successful cancel takes a
 * whole cluster; with clusters {x,1,1} CTA rank r computes row block r of the cluster
 * tile, with {2,2,1} rank r computes row block r / 2 and column block r % 2.  The cluster
 * tiles of a problem (its rows and columns divided by the cluster tile's, rounded up) are
 * numbered in raster order; that number is the launch coordinate of the cluster that owns
 * the tile.  bk must be 64; the library picks the k depth of its ring stages
 * (32 when a CTA runs its own 128 x 256 MMA, which keeps nine stages in flight, 64
 * otherwise). */
typedef struct { int bm, bn, bk; } gemm_tile_t;
typedef struct { int x, y, z; } gemm_cluster_t;

typedef struct {
    int     log_enable;        /* 1 (default): write the per-tile ownership log every run */
    int     trace_enable;      /* 1: record per-tile start/end time and SM id (default 0) */
    int64_t timeout_ns;        /* bound on every device-side wait; <= 0 selects 2 s */
    int     inject_fail_after; /* CLC test hook: after this many successful fetches the
                                  scheduler reports a failed fetch without issuing a cancel;
                                  < 0 (default) disables it */
    int     raster_group;      /* tile rows per raster band; <= 0 selects 16; 1 = row-major */
    int     l2_prefetch;       /* k-blocks (of 64) the producer prefetches into L2 ahead of its
                                  loads; 0 = off (default), < 0 selects the default */
    int     hold_scheduler;    /* test hook (default 0): in CLC mode the scheduler issues no
                                  cancel and signals nothing, so every response wait runs out
                                  after timeout_ns; each worker computes its own tile and
                                  gemm_sync reports GEMM_ERR_TIMEOUT */
    int     cluster_b_multicast; /* clusters of 2: 0 (default) = CTA-pair MMA; 1 = each CTA runs
                                  its own 128 x 256 MMA and the pair shares the B tile by TMA
                                  multicast (clusters of 4 always work this way) */
    int     pdl;               /* 1: launch as a programmatic dependent of the previous kernel
                                  on the stream: the CTAs' prologue (barrier setup, tensor-memory
                                  allocation) may overlap that kernel's tail, and every access to
                                  global memory waits until it has completed.  Default 0 */
    int     fetch_ahead;       /* CLC throttle: 0 (default) = a worker fetches its next tile once
                                  its current tile has started (one tile ahead); 1 or 2 = that many
                                  tiles further ahead (held in reserve, which can unbalance the
                                  tail when tiles differ in cost).  Clamped to [0, 2] */
    int     multicast;         /* read by gemm_create only.  1 (default): the cluster shapes whose
                                  CTAs share operand tiles by TMA multicast (clusters {4,1,1} and
                                  {2,2,1}, and {2,1,1} with cluster_b_multicast) may run, provided
                                  the process sees exactly one GPU.  0: the handle never loads or
                                  launches those kernels and refuses those shapes with
                                  GEMM_ERR_MULTICAST; set it in every process of a multi-GPU job.
                                  The CTA pair and one-CTA shapes issue no multicast load */
} gemm_opts_t;

/* Description of the last launch, filled by gemm_last_launch(). */
typedef struct {
    int64_t n_tiles;      /* CTA tiles = entries of the ownership log */
    int64_t n_cluster_tiles; /* cluster tiles = launch coordinates of CLC / non-persistent */
    int64_t n_workers;    /* workers launched (clusters): entries of the first-tile log */
    int64_t grid_ctas;    /* CTAs in the launch */
    int     smem_bytes;   /* dynamic shared memory per CTA */
    int     cluster;      /* CTAs per cluster */
    int     sched;        /* gemm_sched_t of the launch */
    int     launched;     /* 0 when the call had nothing to launch (M == 0 or N == 0) */
} gemm_launch_info_t;

/* ---------------------------------------------------------------- lifetime */

/* gemm_opts_default: fill `opts` with the defaults listed above.  Not in the pages (a
 * deployment convenience). */
CLCGEMM_API void gemm_opts_default(gemm_opts_t *opts);

/* gemm_create: open a handle on CUDA device `device` (makes it current on this thread).
 * The handle holds what "CUTLASS CLC dynamic persistent kernel", section "Following the
 * CUTLASS source: issuing requests and consuming responses", has the kernel set up once
 * per worker and reuse across tiles (the device-side workspace the schedulers write);
 * the call itself is not in the pages.  opts may be NULL (defaults).  Fails with
 * GEMM_ERR_NO_DEVICE when there is no usable device, GEMM_ERR_UNSUPPORTED_DEVICE when the
 * device is not sm_103.  It loads every kernel the handle may launch (those of the TMA
 * multicast cluster shapes only when opts->multicast is 1 and the process sees one GPU),
 * so that no later launch waits for code loading (under CUDA's lazy loading a first
 * launch can wait until other kernels have finished, which never happens while the SM
 * occupier waits for the host). */
CLCGEMM_API int gemm_create(int device, const gemm_opts_t *opts, gemm_handle_t *out);

/* gemm_destroy: release the handle's SM occupier if it still runs, synchronise the device
 * and free the handle's workspace.  NULL is a no-op.  Not in the pages. */
CLCGEMM_API void gemm_destroy(gemm_handle_t h);

/* gemm_set_opts: replace the handle's options (NULL = defaults).  The `multicast` field
 * keeps the value the handle was created with.  Not in the pages. */
CLCGEMM_API int gemm_set_opts(gemm_handle_t h, const gemm_opts_t *opts);

/* ---------------------------------------------------------------- compute */

/* gemm_run: C = A * B on `stream` (see the file header for layouts and shape rules).
 * The operation of "CUTLASS CLC dynamic persistent kernel", section "From one tile per
 * block to one worker working continuously" (one task = one output tile, three
 * schedulers); the signature follows the problem statement gemm_run(M, N, K, A, B, C,
 * tile, cluster, sched_mode), since the pages define no user API (their
 * clc_fetch_and_wait is a placeholder).
 *   A, B, C      device pointers (bf16, bf16, fp32) into memory of the handle's own
 *                device (cudaMalloc / torch); host, managed or another GPU's memory is
 *                refused with GEMM_ERR_INVALID_ARG before any tensor map is made
 *   tile/cluster see gemm_tile_t
 *   sched        gemm_sched_t
 *   num_workers  STATIC only: workers (clusters) to launch; 0 = SM count / cluster size.
 *                Ignored by CLC and NONPERSISTENT, which launch one cluster per tile.
 * Asynchronous; returns after the launch.  A call may be captured into a CUDA graph once
 * the handle has run the same shape outside the capture (so its workspace is allocated);
 * capture with log_enable = 0: a replay reuses the log tag of the capture. */
CLCGEMM_API int gemm_run(gemm_handle_t h, int64_t M, int64_t N, int64_t K,
             const void *A, const void *B, float *C,
             gemm_tile_t tile, gemm_cluster_t cluster, gemm_sched_t sched,
             int num_workers, void *stream);

/* gemm_run_grouped: G independent problems C_g = A_g * B_g (A_g M_g x K, B_g K x N,
 * C_g M_g x N) in one launch over a single flat tile grid: problem g's tiles follow
 * problem g-1's, and the raster map applies inside each problem.  Not in the pages as an
 * API: the grouped workload of the problem statement (64 problems of uneven height),
 * with the flat tile index decoded to a work tile as in "CUTLASS CLC dynamic persistent
 * kernel", section "Following the CUTLASS source".
 *   M_g              host array of G row counts (each >= 0)
 *   A_g, B_g, C_g    host arrays of G device pointers, each into the handle's device
 *                    memory (checked when the problem set changes; see gemm_run)
 * The per-problem tables live in the handle; a call whose problem set differs from the
 * previous grouped call synchronises `stream` before replacing them. */
CLCGEMM_API int gemm_run_grouped(gemm_handle_t h, int G, const int64_t *M_g, int64_t N, int64_t K,
                     const void *const *A_g, const void *const *B_g, float *const *C_g,
                     gemm_tile_t tile, gemm_cluster_t cluster, gemm_sched_t sched,
                     int num_workers, void *stream);

/* gemm_run_grouped_v: like gemm_run_grouped, but every problem has its own shape (not in
 * the pages: the variable-cost grouped workload; "B200 Cluster Persistent Scheduler"
 * names uneven tile cost as where dynamic scheduling pays):
 * C_g (M_g x N_g) = A_g (M_g x K_g) * B_g (K_g x N_g); each N_g and K_g a multiple of 8.
 * Tiles of different problems then cost different amounts of work (K_g / 64 k-steps),
 * which is where run-time work stealing pays.  The ownership log indexes each problem's
 * CTA tiles row-major over (M_g / 128) x (N_g / bn), problems in order. */
CLCGEMM_API int gemm_run_grouped_v(gemm_handle_t h, int G, const int64_t *M_g, const int64_t *N_g,
                                   const int64_t *K_g, const void *const *A_g, const void *const *B_g,
                                   float *const *C_g, gemm_tile_t tile, gemm_cluster_t cluster,
                                   gemm_sched_t sched, int num_workers, void *stream);

/* gemm_run_host: the same product from HOST buffers (not in the pages: the end-to-end
 * path of a caller whose operands live on the host).  A and B are copied to device
 * staging buffers owned by the handle in blocks (row bands of A, column bands of B, up
 * to 8 each, about 2048 wide); the GEMM of each C block starts as soon as its A and B
 * bands have arrived, and each C block is copied back to C_host while later blocks
 * compute, so host-to-device and device-to-host copies run at the same time (handle-owned
 * streams, ordered after earlier work on `stream`; `stream` waits for the last copy).
 * Pinned host memory makes the copies asynchronous.  The first call (or a larger
 * problem) allocates the staging buffers.  The ownership log afterwards describes the
 * last block. */
CLCGEMM_API int gemm_run_host(gemm_handle_t h, int64_t M, int64_t N, int64_t K,
                  const void *A_host, const void *B_host, float *C_host,
                  gemm_tile_t tile, gemm_cluster_t cluster, gemm_sched_t sched,
                  int num_workers, void *stream);

/* gemm_sync: wait for `stream`, then report and clear the device error word.
 * Returns GEMM_ERR_TIMEOUT if any wait of the finished runs gave up (a worker whose wait
 * ran out stops, like a worker whose cancel failed in "CUTLASS CLC dynamic persistent
 * kernel", section "Cluster granularity and exit after failure", but its tile may be
 * unfinished, so the run is reported), GEMM_ERR_BOUNDS if a library built with bounds
 * checks skipped a tile. */
CLCGEMM_API int gemm_sync(gemm_handle_t h, void *stream);

/* gemm_device_error: the raw device error word of the finished runs (synchronises the
 * device): bits (1 = a wait ran out, 2 = a bounds check failed), wait site (or 100 +
 * the failed check), block of the first failure.  Does not clear it.  Not in the pages. */
CLCGEMM_API int gemm_device_error(gemm_handle_t h, int32_t out3[3]);

/* ---------------------------------------------------------------- ownership log */

/* gemm_last_launch: shape of the most recent launch (its log sizes).  Not in the pages. */
CLCGEMM_API int gemm_last_launch(gemm_handle_t h, gemm_launch_info_t *info);

/* gemm_get_log: copy-out of the most recent run's ownership log; waits for that run's
 * stream only (pageable `owner`/`claims`/`first` memory is fine).  It records the
 * invariant of "CUTLASS CLC dynamic persistent kernel", section "What is cancelled is a
 * launch, what is obtained is a work coordinate": each tile is computed exactly once,
 * either by the launch whose coordinate it is or by the one worker whose cancel
 * obtained that coordinate, and a worker's first tile is its own launch coordinate.
 *   owner[n_tiles]     worker (cluster launch id) that computed each CTA tile, -1 if
 *                      no worker did
 *   claims[n_tiles]    how many times each CTA tile was computed (1 when correct;
 *                      counts saturate at 255)
 *   first[n_workers]   linear id of each worker's first tile, -1 if the worker never ran
 * CTA tiles are indexed row-major over (M / 128) x (N / bn) per problem (both rounded up
 * to whole cluster tiles), problems in order.  Any output pointer may be NULL.  n_tiles / n_workers must equal the values
 * gemm_last_launch() reports.  On the device every entry carries a tag of the launch
 * that wrote it, so logging needs no clearing pass before a launch; this call keeps
 * only the entries of the most recent launch.  GEMM_ERR_INVALID_ARG if the most recent
 * launch wrote no log (log_enable was 0 when it ran, or nothing was launched). */
CLCGEMM_API int gemm_get_log(gemm_handle_t h, int32_t *owner, int32_t *claims, int32_t *first,
                 int64_t n_tiles, int64_t n_workers);

/* gemm_get_trace: (not in the pages: the measurement of where a tile's time goes and of
 * the response wait of "CUTLASS CLC dynamic persistent kernel", section "Following the
 * CUTLASS source") copy-out of the trace of the most recent run, waiting for its stream (that
 * run must have had trace_enable set; GEMM_ERR_INVALID_ARG otherwise): 8 x uint64 per CTA
 * tile (out holds n_tiles * 8):
 *   [0] start ns (the producer begins the tile; device globaltimer)  [1] end ns (the
 *   epilogue issued the tile's last store)  [2] SM id  [3] worker  [4] ns the producer
 *   spent obtaining this tile after finishing the loads of its previous one (CLC: waiting
 *   for the response that named it; static: its next-tile arithmetic; 0 for a worker's
 *   first tile)  [5] ns from the try_cancel that returned this tile to the
 *   scheduler seeing its response (CLC, rank-0 tile only)  [6] ns when the epilogue saw
 *   the finished accumulator  [7] ns when the MMA warp issued the tile's last MMA
 *   (rank 0 for CTA pairs). */
CLCGEMM_API int gemm_get_trace(gemm_handle_t h, uint64_t *out, int64_t n_tiles);

/* ---------------------------------------------------------------- occupancy */

/* gemm_max_active_clusters: how many clusters of the given configuration can be
 * resident at once on the whole device (cudaOccupancyMaxActiveClusters): the resident
 * worker count of "CUTLASS CLC dynamic persistent kernel", section "Why a fixed task
 * sequence has a tail".  GEMM_ERR_MULTICAST for a shape the handle may not launch. */
CLCGEMM_API int gemm_max_active_clusters(gemm_handle_t h, gemm_tile_t tile, gemm_cluster_t cluster,
                             int *clusters);

/* gemm_sm_count: number of SMs of the handle's device.  Not in the pages. */
CLCGEMM_API int gemm_sm_count(gemm_handle_t h, int *sms);

/* SM occupier: launches `n_ctas` CTAs on `stream`, each holding one whole SM (large
 * shared-memory footprint) and spinning until gemm_occupy_stop() or `limit_ns` elapses.
 * It stands for the other kernel of "CUTLASS CLC dynamic persistent kernel", section "Why
 * a fixed task sequence has a tail" (fewer workers resident than planned); the calls are
 * not in the pages (the problem statement's partially-occupied workload).  gemm_occupy_wait_resident() blocks the host until all CTAs run (or
 * `wait_ms` passes: GEMM_ERR_TIMEOUT).  gemm_occupy_stop() releases them; its `status`
 * (may be NULL) is 1 if the spinners hit their time limit. */
CLCGEMM_API int gemm_occupy_start(gemm_handle_t h, int n_ctas, int64_t limit_ns, void *stream);
CLCGEMM_API int gemm_occupy_wait_resident(gemm_handle_t h, int wait_ms);
CLCGEMM_API int gemm_occupy_stop(gemm_handle_t h, int *status);

/* ---------------------------------------------------------------- no-allocation variant */

/* gemm_run_noalloc: the product of gemm_run, for callers that cannot allocate device
 * memory (a process whose device memory belongs to its own pool allocator or sits under
 * a hard cap, or a latency-critical path that cannot afford a cudaMalloc).  The paper
 * has no counterpart: this is a deployment convenience, not part of the method.
 *   - No handle: it runs on the current device with the default options (ownership log
 *     on, 2 s wait bound, the default raster band of 16 tile rows).  Same arguments,
 *     shape rules and pointer checks as gemm_run; the TMA multicast cluster shapes run
 *     only when the process sees one GPU (GEMM_ERR_MULTICAST otherwise).
 *   - Its scratch (device error word and ownership log) is one fixed file-scope device
 *     array of 1 MiB + 16 B, held by every GPU that loads the library until the process
 *     exits.  At most 65536 CTA tiles and 65536 launched workers per call; larger
 *     problems return GEMM_ERR_SCRATCH_LIMIT and launch nothing.
 *   - It calls no cudaMalloc / cudaFree and no allocating library routine.
 *   - The first call on a device (that device current) resolves the array's address and
 *     launches every kernel once over an empty problem on a private stream, waiting for
 *     them (see gemm_create); make that first call before any stream capture begins.
 *   - All calls share the array: each clears what must start at zero on its own stream,
 *     but calls that overlap on the GPU (different streams or threads) race: serialise
 *     them.  gemm_noalloc_status reads back the error word and log of the latest call.
 * Asynchronous on `stream`; returns launch-time errors only (device-side ones through
 * gemm_noalloc_status). */
CLCGEMM_API int gemm_run_noalloc(int64_t M, int64_t N, int64_t K,
                                 const void *A, const void *B, float *C,
                                 gemm_tile_t tile, gemm_cluster_t cluster, gemm_sched_t sched,
                                 int num_workers, void *stream);

/* gemm_noalloc_status: what the most recent gemm_run_noalloc call on the current device
 * left in the fixed scratch, read without allocating device memory.  Waits for `stream`
 * (pass the call's stream), then copies:
 *   out3[3]            the device error word: bits (1 = a wait ran out, 2 = a bounds check
 *                      failed), wait site, block of the first failure; all 0 when the
 *                      call finished normally (may be NULL)
 *   owner, claims, first  the call's ownership log, with the meaning of gemm_get_log (any
 *                      may be NULL); n_tiles and n_workers must equal the call's CTA
 *                      tiles and launched workers (GEMM_ERR_INVALID_ARG otherwise, and
 *                      when no call has run on this device)
 * Returns GEMM_OK, or GEMM_ERR_TIMEOUT / GEMM_ERR_BOUNDS when the error word is set: the
 * call's C is then incomplete.  Nothing is cleared (the next call clears the word).
 * Overlapping gemm_run_noalloc calls race with this read as with each other.  The paper
 * has no counterpart. */
CLCGEMM_API int gemm_noalloc_status(int32_t out3[3], int32_t *owner, int32_t *claims, int32_t *first,
                                    int64_t n_tiles, int64_t n_workers, void *stream);

/* ---------------------------------------------------------------- misc */

/* gemm_strerror: static string for a return code.  Not in the pages. */
CLCGEMM_API const char *gemm_strerror(int code);

/* gemm_version: library version as 10000*major + 100*minor + patch.  Not in the pages. */
CLCGEMM_API int gemm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CLCGEMM_H */
