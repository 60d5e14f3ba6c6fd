/*
 * gemm07.h -- C ABI of libgemm07.so, dense GEMM C = A * B on one NVIDIA
 * GB300 (sm_103a).
 *
 * The operation (every entry point below computes it):
 *   C[i][j] = sum_{k=0}^{K-1} A[i][k] * B[k][j],   0 <= i < M, 0 <= j < N,
 * with A (M x K), B (K x N) and C (M x N) row-major: element (r, c) of a
 * matrix with leading dimension ld sits at base + r*ld + c.
 *   - "GEMM" (inference-book, Part 4), opening section: the element formula.
 *   - "GEMM Optimization" (infra.bea.ai), section 1 "The Problem".
 *   - "How a Matrix Multiply Runs on a GPU", "Level 0": the row-major
 *     indexing A[row*K + k], B[k*N + col], C[row*N + col].
 * C is overwritten (the _ex variants below add alpha, beta, a bias and an
 * activation).  K == 0 writes zeros into C (the empty
 * sum); M == 0 or N == 0 is a no-op.  Out-of-range rows and columns of a
 * ragged edge tile contribute zero and are never written ("A06 -- Tiled
 * Matrix Multiply (GEMM)", section 3, the guarded tiled kernel and ": 0.0f").
 *
 * Conventions shared by every entry point:
 *   - Sizes and leading dimensions are element counts (int64_t).  Required:
 *     M, N, K >= 0, lda >= max(K, 1), ldb >= max(N, 1), ldc >= max(N, 1),
 *     M, N, K < 2^31, and each matrix's rows x leading dimension (M x lda,
 *     K x ldb, M x ldc) at most 2^60 elements.
 *   - Pointers are DEVICE pointers on the calling thread's current device,
 *     owned by the caller; the library keeps none of them after the call
 *     returns, and never frees caller memory.  A null pointer is allowed only
 *     for an operand with no elements.  C must not overlap A or B
 *     (unchecked).
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Calls only enqueue work and return without synchronising;
 *     a device-side failure (a bounded wait that ran out) is reported by
 *     gemm_get_device_status().
 *   - Results are deterministic: the same inputs, sizes and device give the
 *     same bits on every call (no atomics in any reduction).
 *   - Calls are thread-safe.  The library may hold per-device state (a
 *     status word, a workspace pool, scratch blocks kept per stream) until
 *     gemm_shutdown() or process exit.  Scratch is reused by later calls on
 *     the same stream handle, which the stream orders after the earlier
 *     ones; work still queued on a destroyed stream must have finished
 *     before a new stream that may reuse its handle calls the library.
 *     The device-buffer entry points can be captured in a CUDA graph; a
 *     replay must not run concurrently with other library work on the
 *     stream it was captured from (it uses that stream's scratch).
 *
 * Errors: every entry point returns a gemm_status_t.  Argument errors are
 * detected on the host before anything is enqueued and leave C untouched.
 */
#ifndef GEMM07_H
#define GEMM07_H

#include <stdint.h>

#if defined(__GNUC__)
#define GEMM07_API __attribute__((visibility("default")))
#else
#define GEMM07_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gemm_status {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = 1,        /* negative size, short ld, null pointer */
    GEMM_ERR_MISALIGNED = 2,         /* reserved, never returned: any alignment and
                                        leading dimension is handled internally */
    GEMM_ERR_UNSUPPORTED_DEVICE = 3, /* no device, or not compute capability 10.3 */
    GEMM_ERR_LAUNCH = 4,             /* a CUDA call or kernel launch failed */
    GEMM_ERR_TIMEOUT = 5,            /* a device-side bounded wait ran out */
    GEMM_ERR_INTERNAL = 6,           /* tensor-map encoding rejected a layout */
    GEMM_ERR_NO_MEMORY = 7,          /* workspace or staging allocation failed */
    GEMM_ERR_SCRATCH_TOO_SMALL = 8   /* gemm_bf16_f32acc_noalloc: request exceeds its fixed scratch */
} gemm_status_t;

/*
 * gemm_f32 -- FP32 inputs, FP32 output, FP32 arithmetic on the CUDA cores
 * (no tensor cores).
 *   Method: the register-blocked, shared-memory-tiled kernel of "GEMM,
 *   step by step" (section "Concept", register blocking: each thread owns an
 *   8 x 8 patch of C, 128 x 128 blocks) and "A06 -- Tiled Matrix Multiply",
 *   section 3 (transposed A tile with padding, vectorised shared reads,
 *   double buffering).  Each product is fused into its running FP32 sum
 *   (FMA); the order of the sum over k is increasing k.
 *   A: M x K floats, row stride lda.  B: K x N floats, row stride ldb.
 *   C: M x N floats, row stride ldc; columns N..ldc-1 are not touched.
 *   Any alignment and any leading dimension are accepted; 16-byte aligned
 *   bases with ld a multiple of 4 take the vectorised loads.
 */
GEMM07_API gemm_status_t gemm_f32(int64_t M, int64_t N, int64_t K,
                       const float *A, int64_t lda,
                       const float *B, int64_t ldb,
                       float *C, int64_t ldc, void *stream);

/*
 * gemm_bf16_f32acc -- BF16 inputs, FP32 accumulation, FP32 output, on the
 * tensor cores (tcgen05.mma, accumulators in tensor memory).
 *   Method: the tensor-core rung of "GEMM, step by step" (section
 *   "Concept": BF16 inputs, FP32 sums, large 128 x 256 tiles, neighbouring
 *   blocks kept on the same rows and columns so their loads hit L2) and the
 *   block-order swizzle of "GEMM Optimization", section "L2 Cache and Wave
 *   Analysis".  Every BF16 x BF16 product is exact in FP32; the sums are
 *   FP32.
 *   A, B: arrays of BF16 values, passed as their 16-bit patterns (uint16_t,
 *   bit-compatible with __nv_bfloat16).  A: M x K, row stride lda.
 *   B: K x N, row stride ldb.  C: M x N floats, row stride ldc.
 *   Fast path: A and B 16-byte aligned with lda and ldb multiples of 8 (the
 *   operands are then read directly by the tensor-memory accelerator).
 *   Other layouts are first copied on the GPU into an aligned workspace
 *   taken from a library-owned, stream-ordered memory pool.
 */
GEMM07_API gemm_status_t gemm_bf16_f32acc(int64_t M, int64_t N, int64_t K,
                               const uint16_t *A, int64_t lda,
                               const uint16_t *B, int64_t ldb,
                               float *C, int64_t ldc, void *stream);

/*
 * Fused epilogue ("How a Matrix Multiply Runs on a GPU", "Level 2": the
 * output step alpha * acc + beta * C, plus bias and activation, applied while
 * the accumulators are still on chip):
 *   C[i][j] := act(alpha * (A*B)[i][j] + beta * C[i][j] + bias[j])
 * evaluated in FP32 as v = alpha*acc; v = fma(beta, C_old, v); v += bias;
 * v = act(v).  beta == 0: the prior contents of C are not read (they may be
 * uninitialised).  bias: DEVICE pointer to N floats, or NULL.  A NULL
 * epilogue pointer means alpha = 1, beta = 0, no bias, no activation: the
 * plain product, bit for bit.
 */
typedef enum gemm_activation {
    GEMM_ACT_NONE = 0,
    GEMM_ACT_RELU = 1,     /* max(x, 0) */
    GEMM_ACT_GELU = 2      /* x * Phi(x) = 0.5 x (1 + erf(x / sqrt 2)), FP32 erff;
                              the element-wise GELU of "GEMM Optimization" */
} gemm_activation_t;

typedef struct gemm_epilogue {
    float alpha;
    float beta;
    const float *bias;
    int32_t activation;    /* a gemm_activation_t */
} gemm_epilogue_t;

/* gemm_f32 / gemm_bf16_f32acc with a fused epilogue; an unknown activation
 * returns GEMM_ERR_INVALID_ARG. */
GEMM07_API gemm_status_t gemm_f32_ex(int64_t M, int64_t N, int64_t K,
                          const float *A, int64_t lda,
                          const float *B, int64_t ldb,
                          float *C, int64_t ldc,
                          const gemm_epilogue_t *epilogue, void *stream);
GEMM07_API gemm_status_t gemm_bf16_f32acc_ex(int64_t M, int64_t N, int64_t K,
                                  const uint16_t *A, int64_t lda,
                                  const uint16_t *B, int64_t ldb,
                                  float *C, int64_t ldc,
                                  const gemm_epilogue_t *epilogue, void *stream);

/*
 * gemm_bf16_f32acc_noalloc -- the same operation, arguments and results as
 * gemm_bf16_f32acc, for callers that must not allocate device memory.
 *   The pages describe no such entry point; it has no counterpart there.
 *   Who needs it: code that runs inside a host application which owns every
 *   byte of device memory through its own allocator and forbids plug-ins
 *   from calling cudaMalloc, and latency-critical loops where an allocation
 *   could synchronise the device or wait on the allocator.  This call never
 *   calls cudaMalloc, cudaFree, a pool or any other allocating routine.
 *   Scratch: one fixed array of GEMM07_NOALLOC_SCRATCH_BYTES that the
 *   library declares in device memory; every device that loads the library
 *   holds it until the process exits.  A call may put in it, in this order:
 *     1. the aligned copy of A, when A has to be copied (base not 16-byte
 *        aligned, or lda not a multiple of 8);
 *     2. the aligned copy of B, likewise;
 *     3. for M > 128 when the schedule splits tiles along K over several SM
 *        pairs (the default schedule does so at 4096 x 4096 x 4096, even
 *        with aligned operands): the split tiles' partial sums and their
 *        synchronisation words (tickets, ready and cleared flags).
 *   A request whose copies (1 and 2) need more than the array returns
 *   GEMM_ERR_SCRATCH_TOO_SMALL before anything is enqueued; when 3 does not
 *   fit after them, the call runs without the K split instead.  M <= 128
 *   (M = 1 included) and N <= 128 < M run on the small-M and narrow-N
 *   kernels, which reduce through shared memory and put nothing in the
 *   array beyond 1 and 2.
 *   Sharing: every call on a device uses the same array and it keeps the
 *   last call's contents.  ANY two calls whose kernels may overlap on the
 *   GPU (on different streams without ordering between them) race on it,
 *   whether or not their operands are aligned: the results can be wrong, or
 *   a bounded wait can run out and gemm_get_device_status reports
 *   GEMM_ERR_TIMEOUT.  Order the calls on one stream or with events.
 *   Set-up: the first call on each device looks up the array's device
 *   address (with that device current); later calls reuse it.
 */
#define GEMM07_NOALLOC_SCRATCH_BYTES (64ull << 20)
GEMM07_API gemm_status_t gemm_bf16_f32acc_noalloc(int64_t M, int64_t N, int64_t K,
                                        const uint16_t *A, int64_t lda,
                                        const uint16_t *B, int64_t ldb,
                                        float *C, int64_t ldc, void *stream);

/*
 * gemm_f32_ladder -- the teaching rungs that lead up to gemm_f32, for
 * measuring the ladder of the pages on this GPU (not a production path):
 *   rung 0: one thread per output, coalesced mapping ("How a Matrix Multiply
 *           Runs on a GPU", "Level 0"), 0.25 FLOP/byte;
 *   rung 1: 32 x 32 shared-memory tiles, one output per thread, zero-filled
 *           edges ("Level 1"; "A06", section 3), 8 FLOP/byte; double
 *           buffered with one barrier per tile;
 *   rung 2: one-dimensional register tiling, 8 outputs per thread in one
 *           column ("GEMM" (inference-book), 1D register tiling).
 * Same operands, conventions and errors as gemm_f32; rung outside 0..2 or
 * M > 524280 returns GEMM_ERR_INVALID_ARG.
 */
GEMM07_API gemm_status_t gemm_f32_ladder(int rung, int64_t M, int64_t N, int64_t K,
                              const float *A, int64_t lda,
                              const float *B, int64_t ldb,
                              float *C, int64_t ldc, void *stream);

/*
 * Host-buffer variants: the same operations with A, B and C in HOST memory
 * (pinned memory gives the fastest copies; pageable memory works).  The
 * call stages A and B in device buffers from the library's memory pool,
 * runs the GEMM and copies C back, and returns once C is in host memory
 * (it synchronises `stream`).  A is split into row blocks (up to 3 for
 * FP32, 4 for BF16, boundaries on whole 128-row tiles; for FP32, when a
 * block of 30-60 % of the rows fills whole waves of the GPU's resident
 * 128 x 128 tiles, that block and the rest); uploads run on a
 * library-owned upload stream, each block's product is computed on
 * `stream` as soon as its operands arrive, and each block of C is copied
 * back on a library-owned download stream while the next block computes,
 * so uploads, downloads and compute overlap.  For FP32 with K >= 2048 and
 * several blocks, B and the first block of A go up in 4 pieces along K and
 * the first block's product is accumulated piece by piece, so its GEMM
 * starts after a quarter of B has arrived; those rows' sums are then taken
 * in that order (within the FP32 bound, not bit-identical to gemm_f32).
 * Work already queued on `stream` completes before any of this starts.
 */
GEMM07_API gemm_status_t gemm_f32_host(int64_t M, int64_t N, int64_t K,
                            const float *A, int64_t lda,
                            const float *B, int64_t ldb,
                            float *C, int64_t ldc, void *stream);
GEMM07_API gemm_status_t gemm_bf16_f32acc_host(int64_t M, int64_t N, int64_t K,
                                    const uint16_t *A, int64_t lda,
                                    const uint16_t *B, int64_t ldb,
                                    float *C, int64_t ldc, void *stream);

/* Static English text for a status code (never NULL). */
GEMM07_API const char *gemm_status_string(gemm_status_t status);

/*
 * Synchronises `stream`, then reads and clears the current device's
 * device-side status word.  Returns GEMM_ERR_TIMEOUT if any kernel since the
 * last call gave up on a bounded wait (its output is then incomplete),
 * GEMM_ERR_LAUNCH if the stream reports a CUDA error, GEMM_OK otherwise.
 */
GEMM07_API gemm_status_t gemm_get_device_status(void *stream);

/*
 * Test hook for failure detection, on the current device (synchronises it).
 *   wait_ns: limit of every bounded wait inside the tensor-core kernels
 *            (0 restores the default of 2 s).
 *   mode 0:  normal operation.
 *   mode 1:  BF16 tensor-core GEMMs (paired-SM path, small-M and narrow-N
 *            cluster paths, M == 1 included) withhold the copy of their first k-slice
 *            (first stage), so a bounded wait runs out: the kernels unwind,
 *            return, and gemm_get_device_status() reports GEMM_ERR_TIMEOUT
 *            (C is then incomplete).  Nothing faults, traps or hangs.
 * Returns GEMM_ERR_INVALID_ARG for an unknown mode.  Not for production use.
 */
GEMM07_API gemm_status_t gemm_debug_inject(int mode, uint64_t wait_ns);

/* Releases per-device state held by the library (pools, status words). */
GEMM07_API void gemm_shutdown(void);

/* ABI version of this header: 5.  Status codes are numbered as in the
 * boundary definition (MISALIGNED = 2 reserved, UNSUPPORTED_DEVICE = 3,
 * LAUNCH = 4, TIMEOUT = 5, INTERNAL = 6), with NO_MEMORY = 7 and
 * SCRATCH_TOO_SMALL = 8 added (since version 3).  Since version 4, M == 1 is
 * planned as GEMM_PATH_BF16_SKINNY, GEMM_PATH_BF16_GEMV is never returned,
 * and N <= 128 < M is planned as GEMM_PATH_BF16_NARROW.  Since version 5,
 * M > 128 and N > 128 with at most 76 tiles of 128 x 128 and K >= 1536 are
 * planned as GEMM_PATH_BF16_NARROW too, under GEMM_SCHEDULE_AUTO. */
GEMM07_API int gemm_abi_version(void);

/*
 * Number of CUDA kernels this library has launched in this process, across
 * all entry points and devices (for accounting, e.g. kernels per step).
 */
GEMM07_API uint64_t gemm_launch_count(void);

/*
 * Host-only helpers (no GPU needed), exported so that the tile scheduling
 * and the path selection can be checked without a device.
 *
 * gemm_tile_order: the block-order swizzle.  Maps the linear tile index
 * `linear` (0 <= linear < tiles_m * tiles_n) to the tile (*tile_m, *tile_n)
 * it computes.  Tiles are visited in bands of `group` tile-rows; inside a
 * band the index runs down a column of tiles before moving to the next
 * column, so tiles computed at the same time share rows of A and columns of
 * B ("GEMM Optimization", section "L2 Cache and Wave Analysis").  Returns
 * GEMM_ERR_INVALID_ARG when an argument is out of range.
 */
GEMM07_API gemm_status_t gemm_tile_order(int64_t tiles_m, int64_t tiles_n, int64_t group,
                              int64_t linear, int64_t *tile_m, int64_t *tile_n);

/* Which kernel path a call with these arguments takes (no GPU needed). */
typedef enum gemm_path {
    GEMM_PATH_NONE = 0,         /* M == 0 or N == 0: nothing to do          */
    GEMM_PATH_ZERO_FILL = 1,    /* K == 0: C := 0                           */
    GEMM_PATH_F32_SIMT = 2,     /* gemm_f32 register-blocked kernel         */
    GEMM_PATH_BF16_TMA = 3,     /* tcgen05 kernel reading the operands      */
    GEMM_PATH_BF16_PACKED = 4,  /* operands copied to aligned workspace first */
    GEMM_PATH_BF16_SKINNY = 5,  /* 1 <= M <= 128: 128-column tiles, K split
                                   over a cluster, B streamed once (A/B may
                                   also be copied first: see pack_a / pack_b) */
    GEMM_PATH_BF16_GEMV = 6,    /* reserved, never returned: ABI version 3's
                                   M == 1 kernel (B streamed on the CUDA
                                   cores); M == 1 now takes
                                   GEMM_PATH_BF16_SKINNY, which was faster at
                                   every shape measured */
    GEMM_PATH_BF16_SMALL = 7,   /* few multiply-adds (gemm_set_bf16_small_limit):
                                   64 x 64 tiles on the CUDA cores, operands
                                   read in place at any alignment (no
                                   copies), K split into split_k ranges added
                                   in range order (not used by the
                                   no-allocation entry point) */
    GEMM_PATH_BF16_NARROW = 8   /* N <= 128 < M: 128-row tiles by all N
                                   columns, K split over a cluster, A
                                   streamed once (A/B may also be copied
                                   first: see pack_a / pack_b).  Also
                                   M, N > 128 with few tiles and a long K
                                   (at most 76 tiles of 128 x 128, K >= 1536,
                                   under GEMM_SCHEDULE_AUTO): 128 x 128 tiles,
                                   K split over clusters of 2 to 8 CTAs */
} gemm_path_t;

typedef struct gemm_plan {
    int32_t path;          /* a gemm_path_t                                  */
    int32_t tile_m;        /* output tile rows                               */
    int32_t tile_n;        /* output tile columns                            */
    int32_t tile_k;        /* k-slice per pipeline stage                     */
    int32_t stages;        /* shared-memory ring depth                       */
    int32_t split_k;       /* slices of K reduced afterwards (1 = none)      */
    int64_t tiles;         /* output tiles (x split_k work units)            */
    int64_t workspace_bytes; /* device scratch the call takes from the pool */
    int32_t pack_a;        /* 1 if A is first copied to aligned workspace    */
    int32_t pack_b;        /* 1 if B is first copied to aligned workspace    */
    /* BF16 paired-SM path only (0 elsewhere); reported for the 76 resident
     * SM pairs of a 152-SM GB300 under the current gemm_set_bf16_schedule: */
    int64_t dp_tiles;      /* tiles computed whole, round-robin over pairs   */
    int64_t sk_tiles;      /* tiles after them split into runs of k-slices
                              shared evenly by sk_pairs pairs (stream-K)     */
    int32_t sk_pairs;      /* pairs sharing the stream-K slices              */
    int32_t pairs;         /* SM pairs launched                              */
} gemm_plan_t;

/*
 * How the BF16 paired-SM kernel (M > 128) shares out a partial last wave of
 * 256 x 256 tiles ("GEMM Optimization", section "L2 Cache and Wave Analysis":
 * a partial last wave leaves SMs idle).  Under GEMM_SCHEDULE_AUTO, calls
 * with few tiles and a long K run on the narrow-N kernel instead (see
 * GEMM_PATH_BF16_NARROW); the other two schedules keep them on SM pairs.
 *   GEMM_SCHEDULE_AUTO: the estimated fastest of running the last wave as
 *       it is, as 256 x 128 units (when it fills at most half of the SM
 *       pairs), with each of its tiles halved along K over two pairs, or
 *       as GEMM_SCHEDULE_STREAM_K; a split along K is taken only when it is
 *       estimated to save more than about 2.5 us.  Default.
 *   GEMM_SCHEDULE_STREAM_K: wherever it applies (a last wave at most 85 %
 *       full, K at least 8 slices), the last wave's tiles -- and, after one
 *       or more whole waves, also the last whole wave's -- are cut into
 *       equal runs of k-slices, one per pair; a tile cut into segments is
 *       finished by adding the segments' partial sums in k order.
 *   Splits along K need 512 KB of device scratch per SM pair that shares
 *   them, kept per stream between calls.
 *   GEMM_SCHEDULE_COLUMN_SPLIT: never split along K.
 * Every schedule gives the same results up to the order of FP32 additions
 * across a split tile; each is deterministic run to run.
 */
typedef enum gemm_schedule {
    GEMM_SCHEDULE_AUTO = 0,
    GEMM_SCHEDULE_STREAM_K = 1,
    GEMM_SCHEDULE_COLUMN_SPLIT = 2
} gemm_schedule_t;

/*
 * gemm_set_bf16_schedule: choose the schedule (a gemm_schedule_t) for BF16
 * calls issued after it returns, process-wide.  Returns the previous
 * schedule, or -1 (nothing changed) for an unknown value.  No GPU needed.
 */
GEMM07_API int gemm_set_bf16_schedule(int schedule);

/*
 * gemm_set_bf16_small_limit: the largest number of multiply-adds (M * N * K)
 * of a BF16 call that takes GEMM_PATH_BF16_SMALL, for calls issued after it
 * returns, process-wide.  That path also needs M >= 2, and M >= 64 or
 * N * K <= 2^19, and is capped below the limit: at 2^26 when the
 * tensor-core kernels would first copy an operand and K <= 512, else at
 * 2^24 (the measured crossovers on a GB300).  0 sends every call to the
 * tensor-core kernels.  Default 2^27.  Returns the previous limit, or -1
 * (nothing changed) for a negative value.  No GPU needed.
 */
GEMM07_API int64_t gemm_set_bf16_small_limit(int64_t max_macs);

/*
 * gemm_pair_units: the work units that SM pair `pair` computes in the BF16
 * paired-SM kernel for an M x N x K problem when `max_pairs` pairs are
 * resident, under `schedule` (a gemm_schedule_t), in the order it computes
 * them (no GPU needed; a test hook for the work sharing).  Unit i is written
 * to out[9*i .. 9*i+8] as
 *   tile (index in the tile order), k0, k1 (64-deep k-slices [k0, k1)),
 *   slot (-1 unless the unit is a segment of a split tile, else the pair's
 *   partial-sum slot 0/1), first pair and number of segments of the tile
 *   (pair, 1 when not split along K), 1 if the unit belongs to the stream-K
 *   part, else 0, and the unit's first column within the tile and its
 *   width (0 and 256, or 0 / 128 and 128 for the halves of a column-split
 *   tile),
 * for i < cap (out may be NULL when cap is 0).  Returns the number of units,
 * or -1 for an argument out of range (sizes, max_pairs < 1, pair outside
 * [0, max_pairs), unknown schedule).  Tiles are 256 x 256.
 */
GEMM07_API int64_t gemm_pair_units(int64_t M, int64_t N, int64_t K,
                                   int32_t max_pairs, int32_t schedule,
                                   int32_t pair, int64_t *out, int64_t cap);

/*
 * gemm_plan_bf16 / gemm_plan_f32: fill *plan with the path that the
 * corresponding entry point takes for these arguments.  Pointers are only
 * inspected for their alignment, never dereferenced.  Returns the status
 * the entry point would return from argument checking.
 */
GEMM07_API gemm_status_t gemm_plan_bf16(int64_t M, int64_t N, int64_t K,
                             const void *A, int64_t lda,
                             const void *B, int64_t ldb,
                             const void *C, int64_t ldc, gemm_plan_t *plan);
GEMM07_API gemm_status_t gemm_plan_f32(int64_t M, int64_t N, int64_t K,
                            const void *A, int64_t lda,
                            const void *B, int64_t ldb,
                            const void *C, int64_t ldc, gemm_plan_t *plan);

#ifdef __cplusplus
}
#endif

#endif /* GEMM07_H */
