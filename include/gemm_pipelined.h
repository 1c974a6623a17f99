/*
 * gemm_pipelined.h -- C ABI of the software-pipelined tiled GEMM library for
 * NVIDIA GB300 (sm_103a).
 *
 * The operation is the matrix product C = A x B, computed by a tiled K-loop
 * whose global-to-shared tile loads are software-pipelined: a prologue fills
 * the first buffers, the steady state loads tile k+1 .. k+S-1 while the MMA
 * consumes tile k, and an epilogue drains the buffers
 * ("CUDA Kernel Study: Pipelining", Background, Case 1 "Ping-Pong Double
 * Buffering" and Case 2 "cp.async Multi-Stage Pipeline";
 * "pipeline-gpu-kernel", Step 3 "restructure the K loop").  The arithmetic is
 * the plain definition of the product ("Part 4 -- Pipelining and Occupancy",
 * section 4.3): pipelining reorders loads, not arithmetic.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Dimensions: C is M x N, the sum runs over K.  M, N, K >= 0.
 *  - Layouts (elements, no padding; leading dimension = the contiguous extent):
 *      A      row-major M x K (K contiguous);
 *      B      GP_A_ROW_B_COL: column-major K x N, i.e. stored N x K with K
 *             contiguous (both operands K-major);
 *             GP_A_ROW_B_ROW: row-major K x N (N contiguous);
 *      C      row-major M x N.
 *  - Pointers are DEVICE pointers owned by the caller; the library neither
 *    allocates nor frees operand memory and keeps no reference after a call
 *    returns (it caches tensor-map descriptors keyed by pointer and shape,
 *    which hold no ownership).  Every base pointer must be 16-byte aligned.
 *  - Calls are asynchronous on the caller's CUDA stream (a cudaStream_t passed
 *    as void*; NULL is the legacy default stream).  Nothing synchronises
 *    unless a function says so.  The tcgen05 kernels are launched as
 *    programmatic dependents of the work before them in the stream: they may
 *    start their set-up (barriers, tensor memory, descriptor prefetch) while
 *    that work drains, but touch no global memory until it has completed, so
 *    stream order is kept exactly as for an ordinary launch.
 *  - Device workspace: split K-loops (stream-K tails of the tcgen05 kernels,
 *    split FFMA K-loops) and the FP16 copies of INT8 operands live in a
 *    workspace the library allocates per (device, stream) on first need,
 *    grows when a larger plan needs it and keeps until gemm_release
 *    (gp_plan.workspace_bytes is the size a call uses).  Growing it
 *    synchronises that stream and frees and allocates device memory
 *    (cudaFree / cudaMalloc, which may synchronise the device).  The library
 *    tracks up to 64 streams at once; a call on a 65th stream takes over the
 *    least recently used stream's workspace after a device-wide
 *    synchronisation.  gemm_pipelined_noalloc uses a fixed static array
 *    instead.
 *  - Status: each call has its own status record, tagged with the call, in a
 *    static per-device ring of 4096 slots; gemm_stats(sync=1) reads it on the
 *    call's stream only.  A call's record can be lost only if 4096 later calls
 *    on the device are made before it is read and the one sharing its slot
 *    also fails.
 *  - Return value: GP_OK (0) or a negative GP_ERR_* code.  Argument errors are
 *    detected on the host before anything is launched; the output is then
 *    untouched.  gemm_strerror() names every code.
 *  - Thread safety: the per-thread "last call" record read by gemm_stats() is
 *    thread-local; everything else may be called from several host threads
 *    (calls on different streams report their own errors).
 */
#ifndef GEMM_PIPELINED_H
#define GEMM_PIPELINED_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element types: inputs -> accumulator -> output. */
typedef enum {
    GP_I8_I32 = 0,              /* int8 x int8 -> int32 sums (two's-complement wrap) -> int32 C */
    GP_F16_F32ACC_F16OUT = 1,   /* fp16 x fp16 -> fp32 sums -> fp16 C (round to nearest even) */
    GP_BF16_F32ACC_BF16OUT = 2, /* bf16 x bf16 -> fp32 sums -> bf16 C (round to nearest even) */
    GP_F32 = 3                  /* fp32 x fp32 -> fp32 sums (FFMA, no tensor cores) -> fp32 C */
} gp_dtype;

typedef enum {
    GP_A_ROW_B_COL = 0, /* A row-major, B column-major: both K-major */
    GP_A_ROW_B_ROW = 1  /* A row-major, B row-major */
} gp_layout;

/* How the K-loop moves tiles from global to shared memory.  The MMA engine
 * follows the dtype: tcgen05 UMMA with TMEM accumulators for FP16/BF16; FFMA on
 * the CUDA cores for FP32; for INT8, sm_103a has no tcgen05 integer kind, so
 * GP_PIPELINED runs it on tcgen05 with the operands converted exactly to FP16
 * and the FP32 accumulator restarted every 1024 K (all partial sums stay exact
 * integers below 2^24), while the ping-pong and no-overlap variants (and
 * GP_PIPELINED with gp_options.i8_engine = 1) use warp-level IMMA.  Variants of one
 * engine differ only in the data path. */
typedef enum {
    /* Register-staged double buffer: global loads into registers, compute on
     * the current shared buffer, then store the registers into the other one
     * ("CUDA Kernel Study: Pipelining", Case 1; "pipeline-gpu-kernel", Step 3,
     * LDG-register variant).  stages must be 0 or 2. */
    GP_PINGPONG = 0,
    /* Warp-specialised S-stage ring: a TMA producer warp fills S shared-memory
     * slots guarded by mbarrier full/empty phases while the consumers run the
     * MMA ("CUDA Kernel Study: Pipelining", Case 2, with TMA and mbarrier in
     * place of cp.async commit/wait groups).  stages 1..8, 0 = default. */
    GP_PIPELINED = 1,
    /* No overlap: load, synchronise, compute, synchronise
     * ("CUDA Kernel Study: Pipelining", Background).  stages must be 0 or 1. */
    GP_NOPIPE = 2
} gp_variant;

/* Error codes. */
#define GP_OK 0
#define GP_ERR_ARG (-1)         /* null pointer with non-empty output, negative size, bad enum, stages out of range */
#define GP_ERR_UNSUPPORTED (-2) /* dtype x layout x variant not built, or an alignment rule broken */
#define GP_ERR_SMEM (-3)        /* no tile of this variant fits the per-CTA shared-memory budget at this stage count */
#define GP_ERR_CUDA (-4)        /* a CUDA runtime call or the launch failed (detail in gp_stats.cuda_error) */
#define GP_ERR_TIMEOUT (-5)     /* a bounded wait inside the kernel gave up; reported by gemm_stats(sync=1) */
#define GP_ERR_SIZE (-6)        /* a dimension exceeds what the variant can address (see gemm_pipelined) */
#define GP_ERR_SCRATCH (-7)     /* gemm_pipelined_noalloc: the plan needs more scratch than its fixed array holds */

/* Step of a call whose CUDA runtime call failed (gp_stats.cuda_error_site; 0 when nothing failed). */
#define GP_SITE_DEVICE 1        /* device query or the per-device set-up */
#define GP_SITE_EVENT 2         /* timing events (gp_options.time_kernel) */
#define GP_SITE_CAPACITY 3      /* occupancy query of a cluster kernel */
#define GP_SITE_WORKSPACE 4     /* device workspace allocation */
#define GP_SITE_TENSOR_MAP 5    /* TMA tensor-map encoding */
#define GP_SITE_SMEM_ATTR 6     /* opting a kernel into its dynamic shared memory */
#define GP_SITE_LAUNCH 7        /* the kernel launch itself */
#define GP_SITE_SYNC 8          /* gemm_stats(sync=1): reading the status record or synchronising */

/* Tile, stage and resource choice for one problem ("pipeline-gpu-kernel",
 * Step 1 "shared-memory budget" and Step 2 "compute/load ratio"; "Part 4 --
 * Pipelining and Occupancy", section 4.2). */
typedef struct gp_plan {
    int32_t dtype, layout, variant;
    int32_t stages;              /* shared-memory ring slots actually used */
    int32_t bm, bn, bk;          /* CTA output tile BM x BN, K step BK */
    int32_t threads;             /* threads per CTA */
    int32_t stage_bytes;         /* one slot: (BM*BK + BN*BK) * sizeof(input) */
    int32_t ring_bytes;          /* stages * stage_bytes */
    int32_t smem_bytes;          /* dynamic shared memory per CTA (ring + epilogue staging + barriers) */
    int32_t tmem_cols;           /* TMEM columns allocated per CTA (tcgen05 kernels), else 0 */
    int32_t persistent;          /* 1 if CTAs loop over output tiles */
    int32_t grid;                /* CTAs launched (0 when no device was queried) */
    int64_t tiles;               /* output tiles ceil(M/BM) * ceil(N/BN) */
    int64_t k_tiles;             /* ceil(K/BK) */
    double compute_load_ratio;   /* 2*BM*BN*BK / ((BM*BK + BK*BN) * sizeof(input)), FLOP per byte */
    const char* kernel;          /* kernel family name, static string */
    int32_t dp_tiles;            /* persistent kernels: tiles computed whole by one CTA (raster order first) */
    int32_t sk_tiles;            /* tiles after those whose K-loops are split evenly over all CTAs (stream-K) */
    int64_t workspace_bytes;     /* device workspace of the call (per device and stream, kept between calls):
                                    partial tiles of split K-loops; for INT8 on tcgen05 also the FP16 copies */
    int32_t cta_pair;            /* 1: two CTAs (a cluster on one TPC) share each BM x BN tile, each holding
                                    BM/2 rows of A and BN/2 rows of B; stage_bytes and smem_bytes are per CTA.
                                    3 (gp_options.pair_k_split): a cluster of four CTAs (two such pairs)
                                    shares each 256 x 128 tile, splitting its K-loop in two halves */
    int32_t k_splits;            /* FP32 FFMA path, tiles that would leave SMs idle (at most 3/4 of them busy,
                                    or a part-empty last wave): the tiles' K-loops are dealt out as equal
                                    ranges to `grid` CTAs (one per SM, fewer when a range would be under 256 K
                                    steps); k_splits = the CTAs sharing a tile: ceil(grid / tiles) when ranges
                                    are shorter than a K-loop, 2 when longer (each writes a partial tile; the
                                    CTA that completes a tile adds them in K order, so results do not depend
                                    on timing); 1 = whole K-loops */
    int32_t half_tiles;          /* INT8 on tcgen05: the last tiles (after dp_tiles whole ones), each run as two
                                    BM x BN/2 halves by two workers, when the whole tiles would leave a last
                                    wave at most half full; 0 = none */
    int32_t raster_gm;           /* tile order: groups of raster_gm consecutive BM-row blocks, each group swept
                                    over all N blocks (N block major inside a group), groups in turn */
    int32_t b_resident;          /* FP16/BF16 one-CTA ring whose K-loop fills the ring exactly (stages ==
                                    k_tiles, whole tiles only): each CTA takes a contiguous range of tiles in
                                    M-block-fastest order (raster_gm = all M blocks) and keeps the B tile in
                                    the ring while the N block repeats, so only A is loaded; 0 = off */
} gp_plan;

/* Record of the last gemm_pipelined call made by the calling host thread. */
typedef struct gp_stats {
    gp_plan plan;
    int32_t status;              /* return code of that call */
    int32_t cuda_error;          /* cudaError_t of the failing CUDA call, else 0 */
    int32_t regs_per_thread;     /* cudaFuncAttributes.numRegs of the kernel launched */
    int32_t local_bytes;         /* cudaFuncAttributes.localSizeBytes (register spills) */
    int32_t blocks_per_sm;       /* cudaOccupancyMaxActiveBlocksPerMultiprocessor at plan.smem_bytes */
    int32_t sm_count;            /* multiprocessors of the device used */
    uint32_t device_status;      /* the call's status record: 0 = clean, else code | wait site << 8;
                                    valid after gemm_stats(sync=1) */
    float last_ms;               /* kernel time from CUDA events if timing was requested, else -1 */
    int32_t cuda_error_site;     /* GP_SITE_* of the failing CUDA call when cuda_error != 0, else 0 */
} gp_stats;

/* Per-call options for gemm_pipelined_ex.  Zero-initialise and set what you need. */
typedef struct gp_options {
    int32_t bn;                  /* force the CTA tile width BN (0 = automatic); must be one the variant builds
                                    (FP16/BF16: 256, 128, 64; INT8: 256 on tcgen05, 128 or 64 on IMMA; FP32:
                                    128), else GP_ERR_UNSUPPORTED */
    int32_t time_kernel;         /* 1: record CUDA events around the launch; gemm_stats(sync=1) reports last_ms */
    uint64_t timeout_ns;         /* limit of every bounded wait inside the kernel (0 = 1 s) */
    int32_t inject_lost_load;    /* test hook: the TMA producer skips the last tile load of the problem, so a
                                    consumer wait runs out and the call reports GP_ERR_TIMEOUT (no GPU fault) */
    int32_t no_stream_k;         /* 1: never split K-loops across CTAs (every tile computed whole) */
    int32_t no_cta_pair;         /* 1: one CTA per output tile even where CTA pairs are available (INT8: use IMMA) */
    int32_t i8_engine;           /* INT8, GP_PIPELINED: 0 = default (2); 1 = warp-level IMMA ring; 2 = tcgen05
                                    after a separate int8 -> FP16 pass; 3 = tcgen05 in one kernel whose
                                    converter warps write the FP16 copies while the ring already consumes
                                    the K steps they have finished (stages <= 5, else engine 2).  Every
                                    engine gives the same exact int32 results; other values: GP_ERR_ARG */
    int32_t ffma_tm, ffma_tn;    /* FP32, GP_PIPELINED: outputs per thread, rows x columns (0, 0 = 8 x 8);
                                    built: 4x8, 8x4, 8x8, 8x16, 16x8, 16x16 (else GP_ERR_UNSUPPORTED) */
    int32_t plan_sms;            /* gemm_plan_ex only: plan for a device with this many SMs instead of the
                                    current one, all of them available (0 = query the current device); a
                                    launch always plans for the device it runs on */
    int32_t inputs_ready;        /* 1: the caller guarantees that no work still in flight on the stream writes A
                                    or B (they were in place before the previous call on this stream was made).
                                    INT8 on tcgen05 (two-pass engine) then converts them while the previous
                                    call's GEMM is still running, into the other of two FP16 copy buffers
                                    (pipelining successive calls); FP16/BF16 on tcgen05 then starts its loads
                                    and MMAs while the previous kernel on the stream is still finishing (only
                                    its stores wait).  The result is the same.  A promise the library cannot
                                    check: if it is false, A and B may be read too early */
    int32_t pair_k_split;        /* FP16/BF16 on 256 x 128 CTA-pair tiles (N <= 128): 1 = run each tile on a cluster
                                    of two pairs that split its K-loop in two halves, the second pair's FP32
                                    accumulator added by the first through distributed shared memory (at most
                                    5 stages; plan.cta_pair = 3; GP_ERR_UNSUPPORTED where it does not apply);
                                    0 = the planner's choice; -1 = never */
    int32_t one_tile_per_cta;    /* GP_PIPELINED, FP16/BF16 and INT8: 1 = launch one CTA per BM x BN output tile
                                    (grid = tiles), each computing its tile whole and exiting -- no CTA pairs, no
                                    persistent loop, no stream-K (INT8 then runs on the IMMA ring).  This is the
                                    launch shape of the ping-pong and no-overlap variants, so that the three data
                                    paths can be compared with nothing else changed ("CUDA Kernel Study:
                                    Pipelining", Benchmark Results).  0 = the planner's choice */
    int32_t raster_gm;           /* persistent tcgen05 rings: M blocks per raster group (gp_plan.raster_gm);
                                    0 = the planner's choice; negative: GP_ERR_ARG */
} gp_options;

/*
 * gemm_pipelined -- C = A x B on `stream`.
 *   A, B      device pointers to the inputs (layouts above); may be NULL when M*N == 0 or K == 0.
 *   C         device pointer to the output, written completely (every element of M x N); may be NULL
 *             when M*N == 0 (then no argument but the enums and sizes is looked at).
 *   M, N, K   sizes.  M == 0 or N == 0: nothing is launched.  K == 0: C is filled with zeros.
 *   dtype     gp_dtype.  layout: gp_layout.  variant: gp_variant.
 *   stages    shared-memory buffers in the K-loop ring; 0 picks the variant's default.
 *   stream    cudaStream_t (as void*).
 * Built combinations: dtype I8/F16/BF16 with GP_A_ROW_B_COL, dtype F32 with
 * GP_A_ROW_B_ROW; every variant for each.  Alignment rules (TMA and vector
 * loads need 16-byte rows): K % 16 == 0 for I8, K % 8 == 0 for F16/BF16,
 * K % 4 == 0 for F32; N % 4 == 0 for I8 and F32, N % 8 == 0 for F16/BF16.
 * M, N, K must each be below 2^31 (GP_ERR_SIZE).
 * Errors: GP_ERR_ARG, GP_ERR_UNSUPPORTED, GP_ERR_SMEM, GP_ERR_SIZE before any
 * launch; GP_ERR_CUDA if the launch fails.  A kernel that timed out is
 * reported only by gemm_stats(sync=1).
 */
int gemm_pipelined(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K, int dtype, int layout,
                   int stages, int variant, void* stream);

/* gemm_pipelined with options (opts may be NULL: same as gemm_pipelined). */
int gemm_pipelined_ex(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K, int dtype, int layout,
                      int stages, int variant, void* stream, const gp_options* opts);

/*
 * gemm_plan -- the tile / stage / shared-memory choice gemm_pipelined would
 * make, without touching the GPU (plan->grid is filled only if a device is
 * present).  bn: as gp_options.bn.  Returns the same argument / budget errors
 * gemm_pipelined would (alignment and pointer checks excepted).
 */
int gemm_plan(int64_t M, int64_t N, int64_t K, int dtype, int layout, int stages, int variant, int bn,
              gp_plan* out);

/* gemm_plan with the same options as gemm_pipelined_ex (opts may be NULL). */
int gemm_plan_ex(int64_t M, int64_t N, int64_t K, int dtype, int layout, int stages, int variant,
                 const gp_options* opts, gp_plan* out);

/*
 * gemm_stats -- copy the calling thread's last-call record into *out.
 *   sync != 0: first read that call's status record on the call's stream and
 *   synchronise that stream (no other stream), and compute last_ms if timing
 *   was requested.  If the kernel reported a timed-out wait, the record's
 *   status becomes GP_ERR_TIMEOUT and so does the return value.
 * Returns GP_OK, GP_ERR_ARG (out == NULL) or the code described above.
 */
int gemm_stats(gp_stats* out, int sync);

/* Static, human-readable name of an error code. */
const char* gemm_strerror(int code);

/* Version of this ABI: major * 10000 + minor * 100 + patch. */
int gemm_abi_version(void);

/*
 * gemm_release -- free every device workspace the library holds for
 * `device` (the stream-K partial tiles, split-K counters and INT8 FP16 copies
 * of all streams that called it).  Synchronises the device first, so nothing
 * in flight still uses them; later calls allocate afresh.  The fixed array of
 * gemm_pipelined_noalloc and the status slots are static and not affected.
 * Returns GP_OK, GP_ERR_ARG (no such device) or GP_ERR_CUDA.
 */
int gemm_release(int device);

/*
 * gemm_pipelined_noalloc -- the FP16/BF16 TMA-ring GEMM (GP_PIPELINED,
 * GP_A_ROW_B_COL) without any device memory allocation.  The pages describe
 * no such call; it exists for callers that cannot allocate device memory
 * while they run: a framework that owns all device memory through its own
 * pool and forbids allocations behind its back, a serving loop where the
 * implicit device-wide synchronisation of cudaMalloc would stall other
 * streams, or a process whose memory budget is fixed at start-up.
 *
 *   A, B, C, M, N, K, stages, stream: as gemm_pipelined; dtype must be
 *   GP_F16_F32ACC_F16OUT or GP_BF16_F32ACC_BF16OUT (else GP_ERR_UNSUPPORTED).
 *
 * gemm_pipelined keeps the stream-K partial tiles of a split launch in a
 * workspace it allocates on first use for each stream.  This entry point
 * uses instead a fixed array compiled into the library: 40 MiB of partial
 * tiles and 64 KiB of counters, held by every GPU that loads the library until
 * the process exits.  That covers every split plan on a 152-SM GB300; a plan
 * needing more returns GP_ERR_SCRATCH before anything is launched.
 *
 * The first call on a device looks up the array's device address and zeroes
 * its counters (cudaGetSymbolAddress, cudaMemset; neither allocates), so make
 * that first call before any stream capture.  All calls on a device share the
 * one array and it keeps the previous call's contents: calls whose kernels
 * overlap on the GPU (different streams, no ordering between them) race on
 * it and may produce wrong results; calls ordered on one stream are safe.
 * Returns and stats as gemm_pipelined.
 */
int gemm_pipelined_noalloc(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K, int dtype,
                           int stages, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_PIPELINED_H */
