/*
 * gemm_f16.h -- C ABI of the GB300 (sm_103a) dense fp16 GEMM library.
 *
 * The operation ("Building a Tiled GEMM", MLC Modern GPU Programming for
 * MLSys, section "GEMM"):
 *
 *     D[m,n] = sum_{k<K} A[m,k] * B[n,k]        i.e.  D = A * B^T
 *
 * A is M x K and B is N x K, both row-major fp16 (IEEE binary16).  B is the
 * linear-layer weight layout and is read as stored: it is never transposed
 * or repacked.  Products accumulate in fp32 (same section: fp16 storage, fp32
 * accumulator); D is written as fp16, converted from the fp32 sum with
 * round-to-nearest-even.  The throughput figure the library is measured by
 * is TFLOPS = 2*M*N*K / (t * 1e12) (same section, and the headline table of
 * the Croqtile tutorial "dense GEMM fp16 from naive").
 *
 * Conventions for every entry point below:
 *   - A, B and D are DEVICE pointers (cudaMalloc memory or a CUDA tensor's
 *     storage) owned by the caller; the library never frees or keeps them.
 *   - Rows are dense: the leading dimension of A and B is K elements, of D
 *     it is N elements.
 *   - Calls are asynchronous on `stream` (NULL = the legacy default stream):
 *     they validate their arguments on the host, enqueue the kernel(s) and
 *     return.  A returned GEMM_OK means "enqueued"; device-side failures are
 *     reported by gemm_f16_nt_check().
 *   - Argument errors are returned synchronously and nothing is enqueued.
 *   - The library uses the CUDA device that is current on the calling thread.
 *
 * Scratch memory.  Two kernels keep fp32 partial sums and per-tile counters
 * in global memory: the 2-CTA tiles with a split K loop
 * (GEMM_VARIANT_TILE_2CTA_SPLITK) and the stream-K small-M kernel
 * (GEMM_VARIANT_SKINNY_STREAMK; the default small-M kernel sums its partials
 * on chip and needs none).  That workspace is allocated with cudaMalloc on
 * the first call that needs it for a given (device, stream) pair, grows when
 * a larger problem needs more, and is kept until the process exits: a caller
 * that runs these variants on many short-lived streams keeps one workspace
 * per stream (each as large as the largest problem it ran).  Calls on the
 * same stream are ordered and share that workspace safely; calls on
 * different streams get different workspaces.
 *
 * CUDA graphs.  A call may be recorded by stream capture (and the graph
 * replayed on new contents of the same buffers) once one uncaptured call of
 * the same kind has run on that stream: the first call on a device sets the
 * device up, and a call that has to grow its stream's workspace allocates
 * (and may synchronise the stream), which a capture does not allow.  The
 * recorded kernels keep the pointers, sizes and scalars of the captured call.
 */
#ifndef GEMM_F16_H_
#define GEMM_F16_H_

#include <stdint.h>

#if defined(__GNUC__)
#define GEMM_API __attribute__((visibility("default")))
#else
#define GEMM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream; NULL means the legacy default stream. */
typedef struct CUstream_st* gemm_stream_t;

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_VALUE = 1,      /* negative or > INT32_MAX size, NULL pointer with a
                                        non-empty problem, D overlapping A or B, or a variant
                                        that cannot run this shape */
    GEMM_ERR_MISALIGNED = 2,         /* a pointer not 16-byte aligned, or K or N not a
                                        multiple of 8 (TMA needs 16-byte row pitches) */
    GEMM_ERR_UNSUPPORTED_DEVICE = 3, /* the current device is not compute capability 10.3 */
    GEMM_ERR_LAUNCH = 4,             /* the kernel launch itself failed */
    GEMM_ERR_TIMEOUT = 5,            /* a kernel gave up waiting on one of its barriers
                                        (reported by gemm_f16_nt_check) */
    GEMM_ERR_CUDA = 6                /* another CUDA runtime call failed (no device,
                                        out of memory for the workspace, ...) */
} gemm_status_t;

/* Kernel choices.  GEMM_VARIANT_AUTO picks one from the shape. */
typedef enum {
    GEMM_VARIANT_AUTO = 0,
    GEMM_VARIANT_TILE_2CTA_256x256 = 1, /* persistent, 2-CTA cluster, 256x256 tile per pair */
    GEMM_VARIANT_TILE_1CTA_128x128 = 2, /* persistent, one CTA per 128x128 tile */
    GEMM_VARIANT_TILE_1CTA_128x256 = 3, /* persistent, one CTA per 128x256 tile */
    GEMM_VARIANT_SKINNY_SPLITK = 4,     /* M <= 64: operands swapped; N in column ranges, each
                                           range's K loop split over the CTAs of one cluster,
                                           partials summed in distributed shared memory */
    GEMM_VARIANT_TILE_2CTA_SPLITK = 5   /* 2-CTA 256x256 tiles with each tile's K loop split over
                                           several CTA pairs (for shapes with few tiles); falls
                                           back to GEMM_VARIANT_TILE_2CTA_256x256 when the tiles
                                           already fill the GPU */,
    GEMM_VARIANT_SKINNY_STREAMK = 6,    /* M <= 64: operands swapped; (tile, K block) units dealt
                                           in equal contiguous ranges to all SMs, split tiles
                                           summed through the fp32 workspace (the kernel of
                                           gemm_f16_nt_noalloc) */
    GEMM_VARIANT_TILE_2CTA_512x256 = 7, /* persistent, 2-CTA cluster, 512x256 tile per pair: two
                                           MMA consumers per CTA share each staged B tile, each
                                           with its own accumulator and epilogue warpgroup */
    GEMM_VARIANT_TILE_1CTA_SPLITK = 8   /* 1-CTA 128x256 tiles with each tile's K loop split over
                                           a cluster of up to 8 CTAs (for shapes with few tiles);
                                           falls back to GEMM_VARIANT_TILE_1CTA_128x256 when the
                                           tiles already fill the GPU */
} gemm_variant_t;

/* Element type of A and B; both operands share it and the MMA accumulates in
 * fp32.  D (and C, bias) is fp16 for GEMM_DTYPE_F16 and bf16 for the others.
 * The 8-bit types are the FP8 layouts of the GEMM blog post (section 2.2), as
 * the tensor cores define them:
 *   E4M3  1 sign, 4 exponent (bias 7), 3 fraction bits; no infinities,
 *         S.1111.111 is NaN; largest finite 448
 *   E5M2  1 sign, 5 exponent (bias 15), 2 fraction bits; IEEE-like with
 *         infinities and NaNs; largest finite 57344
 * They are stored one byte per element.  Quantisation scales are applied in
 * the fused epilogue: a per-tensor scale through alpha, a per-output-column
 * (per weight row) scale through gemm_epilogue_t.scale_n. */
typedef enum {
    GEMM_DTYPE_F16 = 0,
    GEMM_DTYPE_BF16 = 1,
    GEMM_DTYPE_E4M3 = 2,
    GEMM_DTYPE_E5M2 = 3
} gemm_dtype_t;

typedef enum {
    GEMM_ACT_NONE = 0,
    GEMM_ACT_RELU = 1
} gemm_activation_t;

/*
 * Fused output transform, applied in fp32 to the fp32 accumulator before the
 * single rounding of D:
 *     D = act(alpha * scale_n[n] * (A B^T) + beta * C + bias[n])
 * (the scaled update C = alpha A B + beta C and the bias/activation fusion of
 * the GEMM blog post, sections 2.1 and 5.4; scale_n is the per-output-channel
 * weight scale of its 8-bit quantisation, section 4.2).
 *   alpha       scale of A B^T
 *   beta        scale of C; 0 means C is not read
 *   C           [M][N] row-major, same dtype as D, 16-byte aligned; may be D
 *               itself (in-place update) but may not partly overlap it;
 *               required when beta != 0
 *   bias        [N], same dtype as D, 16-byte aligned, added to every row;
 *               NULL = none
 *   activation  a gemm_activation_t, applied last
 *   reserved    unused
 *   scale_n     [N] fp32, device memory, 16-byte aligned, must not overlap D;
 *               multiplies column n of A B^T; NULL = none.  Any dtype.
 */
typedef struct {
    float alpha;
    float beta;
    const void* C;
    const void* bias;
    int32_t activation;
    int32_t reserved;
    const float* scale_n;
} gemm_epilogue_t;

/*
 * gemm_f16_nt -- D = A * B^T, the operation above.
 *
 *   A  const __half[M][K], row-major, device memory, 16-byte aligned
 *   B  const __half[N][K], row-major, device memory, 16-byte aligned
 *   D  __half[M][N], row-major, device memory, 16-byte aligned; every element
 *      is overwritten, nothing outside it is written; must not overlap A or B
 *   M, N, K  sizes, 0 <= each <= INT32_MAX; K and N multiples of 8
 *   stream   the stream the work is ordered on
 *
 * M == 0 or N == 0 is a no-op (GEMM_OK).  K == 0 writes D = 0 (the empty sum).
 * The kernel path is hand-written sm_103a code (TMA, tcgen05.mma with a TMEM
 * accumulator); there is no CPU or library fallback.
 */
GEMM_API gemm_status_t gemm_f16_nt(const void* A, const void* B, void* D,
                          int64_t M, int64_t N, int64_t K, gemm_stream_t stream);

/*
 * gemm_f16_nt_variant -- gemm_f16_nt with the kernel chosen by the caller.
 * Same arguments and semantics; `variant` selects the kernel.  Returns
 * GEMM_ERR_INVALID_VALUE when the variant cannot run the shape (the skinny
 * variant needs M <= 64).  The split-K variants keep fp32 partial sums in
 * the per-stream workspace described above.  All variants compute the same D up to the order
 * of fp32 additions.
 */
GEMM_API gemm_status_t gemm_f16_nt_variant(const void* A, const void* B, void* D,
                                  int64_t M, int64_t N, int64_t K,
                                  gemm_variant_t variant, gemm_stream_t stream);

/*
 * gemm_bf16_nt -- the same operation for bf16 A, B and D (fp32 accumulation,
 * D rounded to nearest even).  The pages list bf16 beside fp16 (the GEMM blog
 * post, section 2.2: same storage size, fp32's exponent range).  Arguments,
 * layout, ownership and errors as for gemm_f16_nt.
 */
GEMM_API gemm_status_t gemm_bf16_nt(const void* A, const void* B, void* D,
                                    int64_t M, int64_t N, int64_t K, gemm_stream_t stream);

/*
 * gemm_nt_ex -- the general entry point: element type, an optional fused
 * epilogue (NULL = plain D = A B^T) and the kernel variant (GEMM_VARIANT_AUTO
 * to let the planner choose).  Arguments otherwise as for gemm_f16_nt, with
 * A and B of `dtype` and D of the output type that dtype implies (bf16 for
 * the 8-bit types).  For the 8-bit types K must be a multiple of 16 (rows of
 * 16-byte units).
 * Additional errors: GEMM_ERR_INVALID_VALUE for an unknown dtype or
 * activation, beta != 0 with C == NULL, C partly overlapping D, or bias or
 * scale_n overlapping D; GEMM_ERR_MISALIGNED for C, bias or scale_n not
 * 16-byte aligned.
 * With K == 0 the result is act(beta * C + bias) (the empty sum is zero).
 */
GEMM_API gemm_status_t gemm_nt_ex(gemm_dtype_t dtype, const void* A, const void* B, void* D,
                                  int64_t M, int64_t N, int64_t K, const gemm_epilogue_t* epilogue,
                                  gemm_variant_t variant, gemm_stream_t stream);

/*
 * gemm_f16_nt_check -- synchronise `stream`, then report and clear the
 * device-side status word of the current device.  Returns GEMM_OK,
 * GEMM_ERR_TIMEOUT if any kernel since the last check gave up waiting on a
 * barrier (its output is then incomplete), or GEMM_ERR_CUDA if the stream
 * reported an error.  After a timeout the skinny-kernel workspaces of the
 * device are reset.
 */
GEMM_API gemm_status_t gemm_f16_nt_check(gemm_stream_t stream);

/*
 * gemm_selftest_timeout -- failure-detection self-test.  Enqueues on `stream`
 * a one-thread kernel that waits, with the same bounded waits every GEMM
 * kernel uses, on an mbarrier phase that never completes and on a device
 * counter that nothing increments; each wait gives up after `timeout_us`
 * microseconds (1 .. 1000000) and records a timeout in the device status
 * word, and the kernel returns.  The next gemm_f16_nt_check on the stream
 * then reports GEMM_ERR_TIMEOUT and clears the word; the context stays
 * usable.  Returns GEMM_ERR_INVALID_VALUE for a timeout out of range.
 */
GEMM_API gemm_status_t gemm_selftest_timeout(int32_t timeout_us, gemm_stream_t stream);

/* A static, human-readable name for a status code (never NULL). */
GEMM_API const char* gemm_status_string(gemm_status_t status);

/* What a call would run, as decided by the host-side planner. */
typedef struct {
    int32_t variant;         /* the gemm_variant_t that runs (never AUTO) */
    int32_t cta_group;       /* CTAs per MMA (1 or 2) */
    int32_t tile_m;          /* output rows per tile (per CTA pair when cta_group == 2) */
    int32_t tile_n;          /* output columns per tile */
    int32_t tile_k;          /* K elements per pipeline stage */
    int32_t stages;          /* shared-memory pipeline depth in K blocks (the column-range
                                small-M kernel groups them into ring stages of up to 8) */
    int64_t m_tiles, n_tiles;/* tile grid (small M: m_tiles = 1; n_tiles = column ranges of
                                tile_n columns, or tiles of 128 for the stream-K kernel) */
    int64_t k_blocks;        /* ceil(K / tile_k) */
    int32_t grid_ctas;       /* CTAs launched */
    int32_t smem_bytes;      /* dynamic shared memory per CTA */
    int32_t tmem_cols;       /* TMEM columns allocated per CTA */
    int32_t max_tiles_per_cta; /* small M: column ranges per CTA (stream-K: partial-sum
                                  slots per CTA), else 0 */
    int64_t workspace_bytes; /* fp32 partials + counters of the stream-K small-M kernel,
                                else 0 */
    int64_t num_full_tiles;  /* tiled: tiles run whole (the persistent grid's full rounds) */
    int32_t tail_split;      /* tiled: the other tiles are cut into this many column pieces */
    int32_t group_m;         /* tiled: tile rows per raster group (L2 reuse of A) */
    int32_t k_split;         /* pieces per tile's K loop (1 = none): tiled split-K, or the
                                CTAs per cluster of the column-range small-M kernel */
    int32_t reserved;
} gemm_plan_t;

/*
 * gemm_f16_nt_plan -- fill *plan with what gemm_f16_nt_variant(...variant...)
 * would run for an M x N x K problem on a GPU with `num_sms` SMs.  Pure host
 * code: it touches no device when num_sms > 0 (pass num_sms <= 0 to query the
 * current device).  Returns the same argument errors as the GEMM call would
 * for these sizes (pointers are not checked), or GEMM_OK.
 */
GEMM_API gemm_status_t gemm_f16_nt_plan(int64_t M, int64_t N, int64_t K, gemm_variant_t variant,
                               int32_t num_sms, gemm_plan_t* plan);

/*
 * gemm_nt_plan_ex -- gemm_f16_nt_plan for the operand type `dtype` (what
 * gemm_nt_ex(dtype, ...variant...) would run).  The 8-bit types move 128 K
 * elements per pipeline stage (tile_k = 128) instead of 64.  Returns
 * GEMM_ERR_INVALID_VALUE for an unknown dtype or a NULL plan.
 */
GEMM_API gemm_status_t gemm_nt_plan_ex(gemm_dtype_t dtype, int64_t M, int64_t N, int64_t K,
                                       gemm_variant_t variant, int32_t num_sms, gemm_plan_t* plan);

/*
 * gemm_f16_nt_noalloc -- the small-M GEMM (M <= 64) without any device
 * allocation by the library.  (The pages have no counterpart: this entry
 * point exists for callers of this library, not for the method.)
 *
 * Who it is for: callers that cannot call cudaMalloc -- a framework or
 * serving engine that has handed (nearly) all device memory to its own pool,
 * or code that must not risk the device-wide synchronisation a cudaMalloc or
 * cudaFree can cause in the middle of a latency-critical sequence.
 * gemm_f16_nt's small-M path needs a workspace of fp32 partial sums and
 * per-tile counters that it allocates on first use; this entry point instead
 * uses one fixed array compiled into the library (GEMM_F16_NOALLOC_SCRATCH_BYTES,
 * 16 MiB), which every GPU that loads the library holds until the process exits.
 *
 * Arguments, layout, ownership and semantics are those of gemm_f16_nt; the
 * caller still passes A, B and D (device memory).  It runs the stream-K
 * kernel of GEMM_VARIANT_SKINNY_STREAMK on the array and gives the same D as
 * that variant (bitwise); against gemm_f16_nt, which runs the column-range
 * small-M kernel, D agrees up to the order of the fp32 additions.
 *
 * Errors: those of gemm_f16_nt, plus GEMM_ERR_INVALID_VALUE when M > 64 or when
 * the problem needs more scratch than the fixed array holds (nothing is then
 * enqueued).  Every M <= 64 with N <= 16384 fits, at any K; larger N fits for
 * smaller M (the check is exact: 256-byte-padded counters of 4 bytes per
 * 128 columns, plus 4 * 128 * MN bytes of partials per (CTA, tile) slot).
 *
 * Set-up: the first call on a device, with that device current, looks up the
 * array's device address (cudaGetSymbolAddress) and the library's per-device
 * kernel settings; make that first call before any stream capture.
 *
 * Sharing: every call on every stream uses the same array, and it keeps the
 * last call's contents.  Each call clears the counters it needs on `stream`
 * before its kernel runs.  Calls whose work overlaps on the GPU (e.g. issued
 * on two streams without ordering between them) race on the array and give
 * wrong results: order them on one stream or with events.
 */
#define GEMM_F16_NOALLOC_SCRATCH_BYTES (16u << 20)
GEMM_API gemm_status_t gemm_f16_nt_noalloc(const void* A, const void* B, void* D,
                                  int64_t M, int64_t N, int64_t K, gemm_stream_t stream);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* GEMM_F16_H_ */
