/*
 * gemm.h: C ABI of the GB300 (sm_103a) dense tiled GEMM library.
 *
 * The library computes C = A·B for FP16, BF16 or FP8 (E4M3, E5M2) operands.
 * It accumulates in FP32 in tensor memory and casts on store to FP16, BF16
 * or FP32. The operation is the tiled GEMM of "Two Waves, One Stage Apart:
 * Warp-Pipelining Triton GEMMs on AMD Instinct" (opening paragraph: compute
 * on one pair of operand tiles while the next pair is prepared). The FP8
 * form is the GEMM of "Porting High-Performance HIP Kernels to FlyDSL"
 * (section "A More Complex Kernel"): E4M3 operands whose block scales are
 * all 1.0, so that C is the plain product. Throughput is counted as
 * 2·M·N·K / elapsed time, as in the first page's Table 1 caption.
 *
 * Conventions shared by every entry point:
 *   - A is M x K, row-major (K contiguous, leading dimension K).
 *   - B is stored in one of two ways:
 *       GEMM_K_MAJOR : N x K, K contiguous (the transposed "B_T" operand of
 *                      "Porting High-Performance HIP Kernels to FlyDSL",
 *                      section "A More Complex Kernel");
 *       GEMM_MN_MAJOR: K x N, N contiguous (plain row-major B).
 *   - C is M x N, row-major, densely packed (leading dimension N).
 *   - Every matrix is dense; there are no leading-dimension arguments.
 *   - The caller owns all operand memory. The library never frees it.
 *   - C must not overlap A or B. This is not checked.
 *   - Calls are asynchronous on the given stream, except where stated.
 *     `stream` is a cudaStream_t passed as void*; NULL means the legacy
 *     default stream.
 *   - Host-side argument errors are reported by the return value before
 *     anything is enqueued. They never abort the process.
 *   - The stream-taking calls (gemm, gemm_ex, gemm_mx, gemm_mx_ex,
 *     gemm_no_alloc) may be captured into a CUDA graph once one call on the
 *     device has run outside the capture (per-device setup). A replay runs
 *     the captured launch again, with the captured pointers, and gives the
 *     same result as a new call on the same inputs.
 */
#ifndef DENSE_TILED_GEMM_GEMM_H
#define DENSE_TILED_GEMM_GEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element types. F16 and BF16 serve as input or output types, F32 only as an
 * output type, E4M3 and E5M2 only as input types, E2M1 only as the input
 * type of gemm_mx. E4M3 is the OCP 8-bit "FN" format (bias 7, no
 * infinities, largest finite 448); E5M2 is the OCP 8-bit IEEE-style format
 * (bias 15); E2M1 is the OCP 4-bit format (bias 1, largest 6), stored two per
 * byte, the lower K index in the low nibble, each row padded to whole bytes. */
typedef enum {
    GEMM_F16 = 0,
    GEMM_BF16 = 1,
    GEMM_F32 = 2,
    GEMM_E4M3 = 3,
    GEMM_E5M2 = 4,
    GEMM_E2M1 = 5
} gemm_dtype_t;

typedef enum {
    GEMM_K_MAJOR = 0,
    GEMM_MN_MAJOR = 1
} gemm_layout_t;

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = 1,    /* null pointer, non-positive size, unknown enum */
    GEMM_ERR_UNSUPPORTED = 2,    /* valid request the library does not implement */
    GEMM_ERR_CUDA = 3,           /* a CUDA runtime or driver call failed */
    GEMM_ERR_TIMEOUT = 4,        /* a kernel wait ran past its limit (device status) */
    GEMM_ERR_NO_DEVICE = 5,      /* no usable sm_100-family GPU is current */
    GEMM_ERR_OUT_OF_MEMORY = 6   /* a workspace allocation failed */
} gemm_status_t;

/*
 * gemm: C = A·B on the current CUDA device.
 *
 *   A, B, C   device pointers (layouts above). A and B share one type,
 *             dtype_in. C has type dtype_out.
 *   M, N, K   sizes, each >= 1. K = 0 is rejected (GEMM_ERR_INVALID_ARG).
 *   dtype_in  GEMM_F16, GEMM_BF16, GEMM_E4M3 or GEMM_E5M2: the type of both
 *             A and B (GEMM_F32 gives GEMM_ERR_UNSUPPORTED).
 *   dtype_out GEMM_F16, GEMM_BF16 or GEMM_F32. The FP32 accumulator is
 *             rounded to nearest-even when it is cast. An FP8 output type
 *             gives GEMM_ERR_UNSUPPORTED.
 *   layoutA   must be GEMM_K_MAJOR (GEMM_MN_MAJOR gives GEMM_ERR_UNSUPPORTED).
 *   layoutB   GEMM_K_MAJOR or GEMM_MN_MAJOR; FP8 operands need GEMM_K_MAJOR
 *             (GEMM_MN_MAJOR gives GEMM_ERR_UNSUPPORTED).
 *   stream    cudaStream_t as void*.
 *
 * Tile choice: the library runs the tile shape (256 x 256 or 256 x 224 per CTA
 * pair; 128 x 256, 128 x 128 or 128 x 64 per single CTA), the schedule below
 * and the epilogue width that its time model predicts fastest for the
 * problem. Narrow single-CTA tiles serve problems of few tiles, which wide
 * tiles would leave most SMs idle for. gemm_plan reports the choice and
 * gemm_ex overrides it.
 *
 * Tail scheduling: the grid is persistent, one unit (CTA or CTA pair) per
 * resident slot. When the tile count leaves the last wave part-empty, the
 * planner may split the last tiles along K (stream-K): each unit then gets an
 * equal share of their k-blocks, and the units that end a split tile add the
 * FP32 partial sums of the others before the cast. The partial sums and their
 * flags (plan->workspace_bytes) live in the library's scratch (below). For a
 * given device and problem the split points are fixed, so results are
 * reproducible from run to run. The split tiles are run first, so that the
 * whole tiles after them proceed in step across the machine.
 *
 * Alignment: the tensor-memory-access engine needs 16-byte-aligned bases and
 * row pitches. When A or B misses this (for example K*2 bytes, or K bytes for
 * FP8, not a multiple of 16), the call first copies that operand into the
 * library's scratch with rows padded to a multiple of 128 bytes. When C
 * misses it, the epilogue writes C with ordinary stores instead of bulk
 * tensor stores. Results do not depend on either path.
 *
 * Scratch: the library keeps, per device, one scratch buffer for each of up
 * to 8 streams (told apart by cudaStreamGetId), for stream-K partial sums,
 * re-pitched operands and repacked MX scales. A call reuses its stream's
 * buffer, which stream order makes safe, so consecutive calls on a stream
 * put no allocation between their kernels; a buffer that is too small is
 * replaced by cudaFreeAsync and cudaMallocAsync on its own stream. Calls on
 * further streams, and calls made during a stream capture (whose graph then
 * owns the memory), take stream-ordered scratch per call (cudaMallocAsync /
 * cudaFreeAsync on the call's stream). gemm_release_workspace frees the
 * buffers.
 *
 * Per-call host work: the library keeps, per device, the plans and the TMA
 * tensor maps of its most recent launches (GEMM_LAUNCH_CACHE_ENTRIES of
 * each). A call whose sizes, types, layouts, options and pointer alignment
 * match a cached plan skips the planner; one whose operand, scratch and C
 * addresses also match skips the tensor-map encoding. A tensor map holds only
 * the numbers it was encoded from (addresses, sizes, pitches, tile shape), so
 * a cached one is the same bytes as a fresh encoding of the same call.
 * gemm_cache_stats counts hits and misses; gemm_cache_clear empties the
 * cache.
 *
 * Errors: returns GEMM_ERR_INVALID_ARG, GEMM_ERR_UNSUPPORTED,
 * GEMM_ERR_NO_DEVICE, GEMM_ERR_OUT_OF_MEMORY or GEMM_ERR_CUDA before or at
 * launch. A kernel that stalls past the wait limit (2 s per wait) sets the
 * library's device status word and exits; gemm_last_device_status reports it.
 */
#define GEMM_LAUNCH_CACHE_ENTRIES 32
gemm_status_t gemm(const void *A, const void *B, void *C,
                   int64_t M, int64_t N, int64_t K,
                   gemm_dtype_t dtype_in, gemm_dtype_t dtype_out,
                   gemm_layout_t layoutA, gemm_layout_t layoutB,
                   void *stream);

/*
 * gemm_mx: block-scaled (MX) C = (SFA ∘ A)·(SFB ∘ B) on the current device.
 *
 * The MXFP8 and MXFP4 GEMMs of "Two Waves, One Stage Apart" (section "MI450",
 * Table 1), in the OCP Microscaling form: every run of 32 consecutive K
 * elements of a row of A, and of a column of B, shares one E8M0 scale
 * 2^(e-127); the product accumulates in FP32 and is cast on store.
 *
 *   A, B      device pointers. A is M x K, B is N x K (layoutB must be
 *             GEMM_K_MAJOR; GEMM_MN_MAJOR gives GEMM_ERR_UNSUPPORTED).
 *             Elements are dtype_in: GEMM_E4M3 or GEMM_E5M2 (MXFP8, one byte
 *             each, row pitch K bytes) or GEMM_E2M1 (MXFP4, packed, row pitch
 *             ceil(K/2) bytes).
 *   SFA, SFB  device pointers to the E8M0 scale exponents, one byte per 32 K:
 *             SFA is M x ceil(K/32) bytes, SFB is N x ceil(K/32) bytes, both
 *             row-major and densely packed. NULL gives GEMM_ERR_INVALID_ARG.
 *             The value 0xFF (NaN) is not handled specially.
 *   C, M, N, K, dtype_out, layoutA, stream: as for gemm.
 *
 * The call first repacks the scales into the kernel's per-stage layout, in
 * the library's scratch (as for gemm; (M + N) x ceil(K / stage K) x 16
 * bytes), and re-pitches A or B like gemm when their row pitch is not a
 * multiple of 16 bytes. Tiles are 256 x 224, computed by CTA pairs. Errors as
 * for gemm.
 */
gemm_status_t gemm_mx(const void *A, const void *B, const uint8_t *SFA, const uint8_t *SFB, void *C,
                      int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype_in, gemm_dtype_t dtype_out,
                      gemm_layout_t layoutA, gemm_layout_t layoutB, void *stream);

/*
 * gemm_options_t: overrides for gemm_ex and gemm_mx_ex. A zero field means the library
 * chooses that value.
 *   cta_group     1: each output tile is 128 x block_n and one CTA owns it.
 *                 2: tiles are 256 x block_n, and a cluster of two CTAs
 *                 shares each one (paired tensor-core issue).
 *   block_n       the tile width: 256 or 224 for cta_group 2; 256, 128 or 64
 *                 for cta_group 1 (128 and 64 for the FP16/BF16 and FP8
 *                 products only). 224 is valid only for a K-major B. A width
 *                 no variant offers for the other settings gives
 *                 GEMM_ERR_UNSUPPORTED.
 *   max_clusters  upper bound on the persistent grid, counted in CTAs
 *                 (cta_group 1) or in pairs (cta_group 2). A small value
 *                 makes each CTA loop over many tiles.
 *   group_m       raster group height in tiles, for the swizzled tile order.
 *   timeout_ms    per-wait limit inside the kernel (default 2000).
 *   k_stage       K depth of one shared-memory ring stage, in elements: one or
 *                 two 128-byte slabs, so 64 or 128 for FP16/BF16 and 128 or
 *                 256 for FP8 (and for MXFP8), 256 or 512 for packed FP4.
 *                 The default (0) is two slabs for CTA pairs, one slab for
 *                 single CTAs and for the block-scaled kinds. Other values
 *                 give GEMM_ERR_UNSUPPORTED.
 *   stream_k      tail scheduling: 0 lets the planner choose, 1 keeps every
 *                 tile whole (data-parallel), 2 forces stream-K on the last
 *                 tiles (see gemm_schedule_jobs). Other values give
 *                 GEMM_ERR_INVALID_ARG (negative) or GEMM_ERR_UNSUPPORTED.
 *   cluster_pairs CTA pairs per thread-block cluster (cta_group 2 only):
 *                 1 keeps each pair on its own; 2 clusters two pairs on
 *                 tiles side by side in N, which share their A tiles: each
 *                 CTA loads half of its A rows and multicasts them to the
 *                 other pair, so A is read from L2 once per two tiles. Only
 *                 the FP16/BF16 and FP8 products with 256-wide tiles offer
 *                 it. Other values give GEMM_ERR_INVALID_ARG (negative) or
 *                 GEMM_ERR_UNSUPPORTED.
 *   clock_trace   NULL, or a device pointer to 4 writable, 8-byte aligned
 *                 uint64 words. The launch's first CTA then writes the
 *                 global timer (ns) and its SM cycle counter as it starts
 *                 work ([0], [1]) and again as it finishes ([2], [3]), so
 *                 that ([3]-[1]) / ([2]-[0]) is the SM clock, in GHz, that
 *                 the launch ran at. The words are written by the kernel,
 *                 asynchronously on the call's stream; the caller owns them.
 *                 It does not change the plan or the result. The global
 *                 timer advances in steps, so for a launch of a few
 *                 microseconds pool the words of many launches.
 *   epilogue_warps warps per CTA that drain the accumulators: 4, or 8 (two
 *                 per TMEM lane quarter, each taking half of a tile's
 *                 columns). The default (0) takes 8 where a CTA's last
 *                 epilogue, which nothing overlaps, is a large share of its
 *                 work (at most two tiles, or four with a 16-bit C), and 4
 *                 otherwise. Other values give GEMM_ERR_INVALID_ARG
 *                 (negative) or GEMM_ERR_UNSUPPORTED.
 *   reserved      must be 0 (GEMM_ERR_INVALID_ARG otherwise).
 */
typedef struct {
    int32_t cta_group;
    int32_t block_n;
    int32_t max_clusters;
    int32_t group_m;
    int32_t timeout_ms;
    int32_t k_stage;
    int32_t stream_k;
    int32_t cluster_pairs;
    uint64_t *clock_trace;
    int32_t epilogue_warps;
    int32_t reserved;       /* must be 0 */
} gemm_options_t;

/* gemm with overrides. opts may be NULL. An unsupported override combination
 * gives GEMM_ERR_UNSUPPORTED. */
gemm_status_t gemm_ex(const void *A, const void *B, void *C,
                      int64_t M, int64_t N, int64_t K,
                      gemm_dtype_t dtype_in, gemm_dtype_t dtype_out,
                      gemm_layout_t layoutA, gemm_layout_t layoutB,
                      const gemm_options_t *opts, void *stream);

/* gemm_mx with overrides (cta_group must be 0 or 2, block_n 0 or 224,
 * k_stage 0 or one of the offered depths: 128 or 256 for MXFP8, 256 or 512
 * for MXFP4). */
gemm_status_t gemm_mx_ex(const void *A, const void *B, const uint8_t *SFA, const uint8_t *SFB, void *C,
                         int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype_in, gemm_dtype_t dtype_out,
                         gemm_layout_t layoutA, gemm_layout_t layoutB, const gemm_options_t *opts,
                         void *stream);

/*
 * gemm_plan_t: the launch gemm_ex would make for a problem. Filled by
 * gemm_plan, which launches nothing.
 */
typedef struct {
    int32_t cta_group;     /* CTAs per output tile */
    int32_t block_m;       /* rows per output tile (128 * cta_group) */
    int32_t block_n;       /* columns per output tile */
    int32_t block_k;       /* K per pipeline stage (64/128 16-bit, 128/256 FP8) */
    int32_t stages;        /* shared-memory ring depth */
    int32_t num_tiles;     /* output tiles */
    int32_t grid_ctas;     /* persistent CTAs launched */
    int32_t group_m;       /* raster group height */
    int32_t realign_a;     /* 1 if A goes through the padded copy */
    int32_t realign_b;     /* 1 if B goes through the padded copy */
    int32_t direct_store;  /* 1 if C is written with ordinary stores */
    int32_t smem_bytes;    /* dynamic shared memory per CTA */
    int32_t num_sms;       /* multiprocessors on the current device */
    int32_t sk_tiles;      /* leading scheduling units split along K (stream-K); 0 = none.
                              A unit is one tile, or two side by side in N when
                              cluster_pairs is 2 */
    int32_t workspace_bytes; /* stream-K partial sums and flags, taken per call */
    int32_t cluster_pairs;   /* CTA pairs per cluster sharing A (1 or 2) */
    int32_t epilogue_warps;  /* epilogue warps per CTA (4 or 8) */
} gemm_plan_t;

/* Fill *plan for a problem on the current device. Same validation and
 * errors as gemm_ex. Needs a GPU, for the SM count and cluster occupancy. */
gemm_status_t gemm_plan(int64_t M, int64_t N, int64_t K,
                        gemm_dtype_t dtype_in, gemm_dtype_t dtype_out,
                        gemm_layout_t layoutA, gemm_layout_t layoutB,
                        const void *A, const void *B, const void *C,
                        const gemm_options_t *opts, gemm_plan_t *plan);

/* gemm_plan for the block-scaled product of gemm_mx_ex (same arguments; the
 * scale pointers do not affect the plan). workspace_bytes counts the
 * stream-K partial sums only, not the repacked scales. */
gemm_status_t gemm_mx_plan(int64_t M, int64_t N, int64_t K,
                           gemm_dtype_t dtype_in, gemm_dtype_t dtype_out,
                           gemm_layout_t layoutA, gemm_layout_t layoutB,
                           const void *A, const void *B, const void *C,
                           const gemm_options_t *opts, gemm_plan_t *plan);

/*
 * gemm_from_host: C = A·B with A, B and C in HOST memory (pinned or
 * pageable). It copies A and B to a device workspace, runs gemm on `stream`,
 * copies C back, and synchronises the stream before returning: C_host is
 * complete when the call returns GEMM_OK. The workspace belongs to the
 * library: two staging slots per device, each cached and grown to the
 * largest problem seen; gemm_release_workspace frees them. The errors are
 * gemm's, plus GEMM_ERR_OUT_OF_MEMORY when a slot cannot grow.
 */
gemm_status_t gemm_from_host(const void *A_host, const void *B_host, void *C_host,
                             int64_t M, int64_t N, int64_t K,
                             gemm_dtype_t dtype_in, gemm_dtype_t dtype_out,
                             gemm_layout_t layoutA, gemm_layout_t layoutB,
                             void *stream);

/*
 * gemm_from_host_async: gemm_from_host without the final synchronisation.
 * The uploads of A and B run on a copy stream of the library, in the next of
 * the two staging slots, once that slot's previous call has finished with
 * it; the product and the read-back of C run on `stream`, after the uploads.
 * So consecutive calls overlap: one call's uploads run while the previous
 * call's product and read-back run. C_host is complete once `stream` has
 * passed the call (cudaStreamSynchronize, or an event recorded after it);
 * A_host and B_host must stay unchanged until then. With pinned host memory
 * the call returns without waiting for the copies. Arguments and errors are
 * gemm_from_host's.
 */
gemm_status_t gemm_from_host_async(const void *A_host, const void *B_host, void *C_host,
                                   int64_t M, int64_t N, int64_t K,
                                   gemm_dtype_t dtype_in, gemm_dtype_t dtype_out,
                                   gemm_layout_t layoutA, gemm_layout_t layoutB,
                                   void *stream);

/* Free the gemm_from_host staging slots and the per-stream scratch buffers of
 * the current device and empty its launch cache. Synchronises the device
 * first. */
gemm_status_t gemm_release_workspace(void);

/* Launch-cache counters of this process, over all devices: plan lookups that
 * hit or missed, and tensor-map lookups that hit or missed. Any pointer may
 * be NULL. */
void gemm_cache_stats(uint64_t *plan_hits, uint64_t *plan_misses, uint64_t *map_hits,
                      uint64_t *map_misses);

/* Empty the launch cache of the current device (the counters keep counting). */
gemm_status_t gemm_cache_clear(void);

/*
 * gemm_last_device_status: synchronise `stream`, then read and clear the
 * device status word of the current device. Returns GEMM_OK, or
 * GEMM_ERR_TIMEOUT if any kernel of this library timed out a wait since the
 * last call. If detail is not NULL, *detail gets the wait site that timed
 * out (role << 8 | barrier kind), or 0.
 */
gemm_status_t gemm_last_device_status(void *stream, uint32_t *detail);

/*
 * gemm_selftest_wait_timeout: launch one CTA that waits, through the
 * kernel's own bounded wait, on a shared-memory barrier that nothing ever
 * arrives at, with a limit of timeout_ms. The kernel records a timeout in
 * the device status word and returns. It does not hang, trap or fault.
 * Check the result with gemm_last_device_status. Exists so that tests can
 * prove that a stalled wait ends.
 */
gemm_status_t gemm_selftest_wait_timeout(int32_t timeout_ms, void *stream);

/*
 * gemm_selftest_withheld_load: run the real GEMM kernel (gemm's arguments,
 * whole tiles only, cta_group 1 or 2) with the tile producer of the first
 * unit withholding one stage: for k-block withhold_kb of its first tile it
 * issues neither the expected-bytes arrive nor the tensor loads. Every
 * address stays valid and no copy is left in flight; the stage simply never
 * fills, so the matrix issuer and the epilogue behind it wait until
 * timeout_ms runs out. The kernel then records GEMM_ERR_TIMEOUT with the
 * site of the first wait that ran out in the device status word, every role
 * stops issuing, and the launch returns. C is left partly written. Exists so
 * that tests can prove that the product kernel's abort path ends.
 *   withhold_kb  0 <= withhold_kb < the number of ring stages K spans
 *                (ceil(K / block_k)); otherwise GEMM_ERR_INVALID_ARG.
 *   timeout_ms   1 .. 10000; otherwise GEMM_ERR_INVALID_ARG.
 *   cta_group    1 or 2; otherwise GEMM_ERR_INVALID_ARG.
 * Other errors are gemm's.
 */
gemm_status_t gemm_selftest_withheld_load(const void *A, const void *B, void *C,
                                          int64_t M, int64_t N, int64_t K,
                                          gemm_dtype_t dtype_in, gemm_dtype_t dtype_out,
                                          gemm_layout_t layoutB, int32_t cta_group,
                                          int32_t withhold_kb, int32_t timeout_ms, void *stream);

/*
 * gemm_no_alloc: gemm for callers that must not allocate device memory.
 *
 * The pages have no counterpart to this entry point; it exists for callers
 * such as a serving runtime that has already handed all of the GPU's memory
 * to its own pool, or a latency-critical loop in which a cudaMalloc or
 * cudaFree could synchronise the device or fail. gemm itself needs scratch
 * whenever A or B must be re-pitched (a base or row pitch that is not a
 * multiple of 16 bytes, for example K*2 bytes not a multiple of 16) and
 * whenever its plan splits tiles along K (the stream-K partial sums and
 * flags), and takes it with cudaMallocAsync/cudaFreeAsync: on a stream's
 * first such call, when that stream's buffer must grow, and per call on
 * streams beyond its cache or during a capture. gemm_no_alloc takes the same arguments
 * and computes the same result, but it never allocates or frees: the
 * re-pitched copies and the stream-K workspace go into one fixed device
 * array that the library holds on every GPU that loads it,
 * GEMM_NO_ALLOC_SCRATCH_BYTES (32 MiB) in size, until the process exits.
 *
 *   - Limit: the padded copies (rows x row bytes rounded up to 128, A then B,
 *     each started on a 256-byte boundary) must fit in
 *     GEMM_NO_ALLOC_SCRATCH_BYTES. Otherwise the call returns
 *     GEMM_ERR_UNSUPPORTED and launches nothing. When no operand needs
 *     re-pitching the array is not used for them, and there is no size limit
 *     beyond gemm's.
 *   - Stream-K: when the plan splits tiles along K, the partial sums and
 *     flags go into the same array after the copies. When they do not fit,
 *     the call keeps every tile whole instead (same result bound).
 *   - Set-up: the first call on a device (whether or not it needs the
 *     array) looks up the array's device address (cudaGetSymbolAddress) with
 *     that device current. Make this first call before any stream capture.
 *   - Sharing: every call on a device uses the same array, and the array
 *     keeps the previous call's contents. Nothing in it has to start at zero:
 *     each call writes every element it later reads. Calls whose work
 *     overlaps on the GPU (for example on two streams at once) race on the
 *     array, so serialise them.
 * Other errors are as for gemm.
 */
#define GEMM_NO_ALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

gemm_status_t gemm_no_alloc(const void *A, const void *B, void *C,
                            int64_t M, int64_t N, int64_t K,
                            gemm_dtype_t dtype_in, gemm_dtype_t dtype_out,
                            gemm_layout_t layoutA, gemm_layout_t layoutB,
                            void *stream);

/*
 * gemm_no_alloc_scratch: the current device's fixed array of gemm_no_alloc,
 * for tests and debuggers that check what the calls write into it.
 * *ptr receives its device address and *bytes its size
 * (GEMM_NO_ALLOC_SCRATCH_BYTES). The address is looked up as on a first
 * gemm_no_alloc call on the device. The array belongs to the library: a
 * caller may read it, or fill it between calls that are not in flight,
 * since no call depends on its previous contents.
 * Errors: GEMM_ERR_INVALID_ARG (ptr or bytes NULL), GEMM_ERR_NO_DEVICE,
 * GEMM_ERR_CUDA.
 */
gemm_status_t gemm_no_alloc_scratch(void **ptr, size_t *bytes);

/*
 * gemm_schedule_jobs: the work list that unit `unit` of a launch walks, as
 * computed by the kernel itself (no GPU needed). Tiles [0, sk_tiles) (the
 * first in the swizzled raster order) are laid end to end in k-blocks
 * (k_blocks per tile) and cut into `units` equal ranges, one per unit; tiles
 * [sk_tiles, num_tiles) are whole and dealt round-robin to the units. Each
 * job covers k-blocks [kb_begin, kb_end) of one tile and is
 *   GEMM_JOB_FULL   the whole K range: the unit stores C for the tile;
 *   GEMM_JOB_WRITER a leading or middle part: the unit leaves an FP32 partial;
 *   GEMM_JOB_OWNER  the trailing part: the unit adds the writers' partials
 *                   (units unit-1, unit-2, ... that share the tile) and stores C.
 * Jobs are listed in the order the unit runs them: the writer job, the whole
 * stream-K tiles, the owner job, then the whole round-robin tiles. Writes at most max_jobs
 * entries to `jobs` and the full count to *n_jobs. Returns
 * GEMM_ERR_INVALID_ARG for inconsistent sizes (num_tiles < 1, units < 1,
 * unit outside [0, units), k_blocks < 1, sk_tiles outside [0, num_tiles],
 * jobs NULL with max_jobs > 0, or n_jobs NULL). The planner always makes
 * num_tiles - sk_tiles a multiple of units, so that every unit gets the same
 * number of whole tiles.
 */
typedef enum { GEMM_JOB_FULL = 0, GEMM_JOB_WRITER = 1, GEMM_JOB_OWNER = 2 } gemm_job_kind_t;

typedef struct {
    int32_t tile;
    int32_t kb_begin;
    int32_t kb_end;
    int32_t kind;
} gemm_job_t;

gemm_status_t gemm_schedule_jobs(int32_t num_tiles, int32_t units, int32_t k_blocks, int32_t sk_tiles,
                                 int32_t unit, gemm_job_t *jobs, int32_t max_jobs, int32_t *n_jobs);

/* Human-readable name of a status code. Never NULL. */
const char *gemm_status_string(gemm_status_t status);

/* Number of GEMM kernel launches (main kernel and operand copies) this
 * process made on any device. Used to count launches in a timed region. */
uint64_t gemm_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* DENSE_TILED_GEMM_GEMM_H */
