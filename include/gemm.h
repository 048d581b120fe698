/*
 * gemm.h -- C ABI of the GB300 dense-GEMM library (libtcgemm.so).
 *
 * One operation: C = A . B over row-major operands with an FP32 result,
 * computed on an NVIDIA GB300 (sm_103a) by hand-written CUDA kernels.
 *
 * Where the operation is defined:
 *   - "Shared memory and tensor cores" (ml-compiler-from-scratch ch. 13),
 *     section 13.1: C = A @ B, 2*M*N*K flops, traffic of a block tiling;
 *     sections 13.3-13.7: the shared-memory tiled SIMT kernel with barriers
 *     and register micro-tiles (the FP32 path here);
 *     section 13.8: tensor-core precision (exact products, FP32 sums).
 *   - "Learn CuTeDSL" README, sections 3 (TMA), 4.3 (tcgen05 MMA with the
 *     accumulator in Tensor Memory, 2-CTA MMA), 5.4 (TMA/MMA pipeline) and
 *     8.1 (static persistent tile scheduler): the TF32/BF16 tensor-core path.
 *   - The same README, section 2.2.1: a C entry point taking raw device
 *     pointers and sizes, called from a thin Python layer.
 *
 * Conventions for every entry point:
 *   - Matrices are row-major.  A is M x K, B is K x N, C is M x N.  Leading
 *     dimensions are in ELEMENTS: lda >= K, ldb >= N, ldc >= N.
 *   - A, B and C are DEVICE pointers owned by the caller; the library never
 *     frees or retains them past the call.  The stream is the caller's
 *     (NULL = the legacy default stream).  Work is enqueued on it and the call
 *     returns without synchronising; the result is ready once the stream is.
 *   - A status code (gemm_status_t) is returned.  On any non-zero status
 *     nothing was enqueued, except GEMM_ERR_CUDA raised by a launch, in which
 *     case the stream is in the state CUDA reports.  gemm_last_error() gives
 *     a human-readable message for the calling thread's last failure.
 *   - The library is thread-safe for concurrent calls on different streams.
 */
#ifndef TCGEMM_GEMM_H
#define TCGEMM_GEMM_H

#include <stdint.h>

#if defined(__GNUC__)
#define GEMM_API __attribute__((visibility("default")))
#else
#define GEMM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t is 'struct CUstream_st *'; declaring the tag keeps this header
 * free of CUDA includes while staying the same type. */
struct CUstream_st;

typedef enum {
    GEMM_FP32 = 0, /* A, B float; exact FP32 products and sums on the CUDA cores  */
    GEMM_TF32 = 1, /* A, B float; tensor cores read them as TF32 (10-bit mantissa)
                      and accumulate in FP32 in Tensor Memory                      */
    GEMM_BF16 = 2, /* A, B bfloat16 (raw uint16 storage); exact products,
                      FP32 accumulation in Tensor Memory                           */
    GEMM_FP16 = 3, /* A, B IEEE half (raw uint16 storage); exact products,
                      FP32 accumulation in Tensor Memory                           */
    GEMM_E4M3 = 4, /* A, B OCP FP8 E4M3 bytes (bias 7, no infinities); exact
                      products, FP32 accumulation in Tensor Memory                 */
    GEMM_E5M2 = 5  /* A, B OCP FP8 E5M2 bytes (bias 15); exact products, FP32
                      accumulation in Tensor Memory                                */
} gemm_dtype_t;

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = 1, /* bad size, leading dimension, pointer or overlap */
    GEMM_ERR_UNSUPPORTED = 2, /* valid request this build/device cannot serve     */
    GEMM_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed                 */
    GEMM_ERR_TIMEOUT = 4,     /* a kernel's bounded wait expired (see status)      */
    GEMM_ERR_NO_MEMORY = 5    /* workspace allocation failed                       */
} gemm_status_t;

/*
 * gemm_run -- C = A . B  (C is overwritten; gemm_run_ex adds alpha, beta, a
 * bias, an activation and a 16-bit output).
 *
 *   M, N, K     sizes, each >= 0.  M == 0 or N == 0: no-op.  K == 0: C is
 *               filled with zeros (the empty sum).
 *   dtype       gemm_dtype_t.  A and B are 'const float *' for GEMM_FP32 and
 *               GEMM_TF32, 'const uint16_t *' holding bfloat16 bits for
 *               GEMM_BF16 and IEEE half bits for GEMM_FP16, 'const uint8_t *'
 *               holding FP8 bytes for GEMM_E4M3 and GEMM_E5M2 ("Learn
 *               CuTeDSL" section 4: the tcgen05 MMA reads 8-bit inputs with
 *               twice the K per instruction of 16-bit ones).
 *   A, lda      device pointer to A[0][0], leading dimension in elements.
 *   B, ldb      device pointer to B[0][0], leading dimension in elements.
 *   C, ldc      device pointer to C[0][0] (float), leading dimension in elements.
 *   stream      the CUDA stream to enqueue on.
 *
 * Paths: GEMM_FP32 runs the tiled SIMT kernel; every other dtype runs the
 * persistent TMA + tcgen05 kernel.  When its tiles are too few to give every
 * SM about six blocks, the SIMT path cuts K into up to 8 ranges: their partial
 * sums go to a stream-ordered workspace of (ranges x M x N) floats, and a
 * second kernel adds them in range order (results are deterministic). That
 * workspace is allocated and freed on the stream like the ones below, and is
 * reported as GEMM_ERR_NO_MEMORY if unavailable.  Operands whose layout the
 * TMA engine cannot address (base not 16-byte aligned, or a row pitch that is
 * not a multiple of 16 bytes) are first copied into a stream-ordered workspace
 * with a padded pitch; that workspace is allocated and freed on the stream
 * (cudaMallocAsync/cudaFreeAsync) and reported as GEMM_ERR_NO_MEMORY if
 * unavailable.  For FP8 tiles narrower than 128 columns (and on request,
 * option "tc_b_major"), B is first transposed into the same kind of
 * workspace, because the MMA then reads its B operand K-major; otherwise B is
 * read as stored.  When there are too few output tiles to occupy every SM
 * and K is long, the tensor-core path splits K.  Two K ranges of a tile that
 * fit one round of 2-CTA clusters run on the two CTAs of a cluster and are
 * summed in distributed shared memory (no workspace, no second kernel); the
 * planner takes 128-column tiles in two such ranges where they keep as many
 * CTAs busy as 256-column tiles would (and, for TF32 and 8-bit inputs, in
 * place of 64-column tiles).  Otherwise partial tiles go to a workspace and a
 * second kernel sums them into C in a fixed order.  Either way the ranges are
 * added in order (results are deterministic, and the same both ways).  With
 * 16-bit inputs, at most 256 rows and a B of 64 MiB or more (B streaming
 * from HBM), split tiles are 128 columns wide.  When the tiles of the last,
 * partly idle round of the persistent
 * schedule would fill at most half of the machine, 16-bit inputs on short
 * schedules run them as two column halves each (every half over all of
 * K, straight to C: no workspace, and the same sums as a whole tile; the
 * launch ends sooner because each half's epilogue drains half the
 * accumulator); on request ("tc_tail_splits") they are split in K instead,
 * like split-K. C leaves through TMA stores when its base, pitch and row
 * length (N elements) are all multiples of 16 bytes, else through ordinary
 * stores.
 *
 * Errors: GEMM_ERR_INVALID_ARG for negative sizes, lda < K, ldb < N, ldc < N,
 * a NULL pointer with a non-empty extent, an unknown dtype, a pointer not
 * aligned to its element, or C overlapping A or B in memory.  A kernel whose
 * bounded wait expires records GEMM_ERR_TIMEOUT in a device status word that
 * gemm_get_status() reads.
 */
GEMM_API int gemm_run(int64_t M, int64_t N, int64_t K, int dtype,
             const void *A, int64_t lda, const void *B, int64_t ldb,
             float *C, int64_t ldc, struct CUstream_st *stream);

/*
 * gemm_run_ex -- C = act(alpha * (A . B) + beta * C + bias), stored as
 * out_dtype: the GEMM with its epilogue fused into the kernel that writes C.
 * "Shared memory and tensor cores" (ml-compiler-from-scratch ch. 13) section
 * 13.10 lists epilogue fusion among what production kernels add; "Learn
 * CuTeDSL" (section 6) fuses work on the accumulator before C is written.
 *
 *   M..ldb      as gemm_run.
 *   C, ldc      device pointer to C[0][0] of element type epi->out_dtype
 *               (float, or bfloat16 / IEEE half bits), leading dimension in
 *               elements.  Read first when epi->beta != 0.
 *   epi         NULL means alpha = 1, beta = 0, no bias, no activation, FP32
 *               output (exactly gemm_run).  Otherwise:
 *     alpha     scale of A . B
 *     beta      scale of the C already in memory (0: C is not read)
 *     bias      device pointer to N floats added to every row, or NULL
 *     activation  GEMM_ACT_NONE, GEMM_ACT_RELU (max(x, 0)) or GEMM_ACT_GELU
 *               (x * Phi(x) with the normal CDF written through erf)
 *     out_dtype GEMM_OUT_F32, GEMM_OUT_BF16 or GEMM_OUT_F16; the value is
 *               computed in FP32 and rounded to nearest even once
 * The epilogue is applied after all of K is summed (with split-K, by the
 * kernel that sums the K ranges).  Errors as gemm_run, plus
 * GEMM_ERR_INVALID_ARG for an unknown activation or output type, or a bias
 * pointer that is not device memory covering N floats.
 */
typedef enum { GEMM_ACT_NONE = 0, GEMM_ACT_RELU = 1, GEMM_ACT_GELU = 2 } gemm_activation_t;
typedef enum { GEMM_OUT_F32 = 0, GEMM_OUT_BF16 = 1, GEMM_OUT_F16 = 2 } gemm_out_t;

typedef struct {
    float alpha;
    float beta;
    const float *bias;
    int32_t activation;
    int32_t out_dtype;
} gemm_epilogue_t;

GEMM_API int gemm_run_ex(int64_t M, int64_t N, int64_t K, int dtype,
                         const void *A, int64_t lda, const void *B, int64_t ldb,
                         void *C, int64_t ldc, const gemm_epilogue_t *epi,
                         struct CUstream_st *stream);

/*
 * gemm_run_grouped -- a batch of independent GEMMs in one persistent launch,
 * C_g = act(alpha * A_g . B_g + beta * C_g + bias_g) for g < group_count
 * ("Learn CuTeDSL" section 8.4, grouped tile scheduler: the tiles of every
 * group flattened into one list of work units that the persistent CTAs share).
 *
 *   dtype        one gemm_dtype_t for every group.  Tensor-core dtypes run as
 *                one launch; GEMM_FP32 runs one SIMT launch per group.
 *   group_count  number of groups, 0 .. 2^20 (0: no-op).
 *   groups       HOST array of group_count gemm_group_t, read during the call
 *                only.  Each group's M..ldc follow gemm_run_ex (C in the
 *                epilogue's output type); bias is the group's own N floats
 *                (device memory) or NULL.
 *   epi          shared alpha, beta, activation and output type, or NULL (as
 *                gemm_run); its bias must be NULL.
 *   stream       the CUDA stream to enqueue on.
 * Groups with M == 0 or N == 0 are skipped; groups with K == 0 get the
 * epilogue of an empty sum.  All groups share one tile shape and CTA pairing,
 * chosen from their total tile count; there is no split-K.  Operands TMA cannot
 * address are packed (and TF32 B transposed) into a stream-ordered workspace,
 * which also holds the groups' descriptors.
 * Errors: as gemm_run_ex for any group's arguments, plus GEMM_ERR_INVALID_ARG
 * for group_count out of range, a NULL groups array, a non-NULL epi->bias, or
 * a group's C overlapping another group's A, B, C or bias.
 */
typedef struct {
    int64_t M, N, K;
    const void *A;
    int64_t lda;
    const void *B;
    int64_t ldb;
    void *C;
    int64_t ldc;
    const float *bias;
} gemm_group_t;

GEMM_API int gemm_run_grouped(int dtype, int64_t group_count, const gemm_group_t *groups,
                              const gemm_epilogue_t *epi, struct CUstream_st *stream);

/* Message for the calling thread's most recent failed call ("" if none).
 * The string is owned by the library and valid until the thread's next call. */
GEMM_API const char *gemm_last_error(void);

/*
 * gemm_get_status -- synchronise `stream`, then read and clear the device
 * status word that kernels set when a bounded wait expires.  Returns GEMM_OK,
 * GEMM_ERR_TIMEOUT (with the role and tile in gemm_last_error()), or
 * GEMM_ERR_CUDA if the synchronisation itself failed.
 */
GEMM_API int gemm_get_status(struct CUstream_st *stream);

/*
 * gemm_set_option / gemm_get_option -- process-wide tuning overrides, for
 * sweeps and tests.  Keys (value 0 = automatic unless stated):
 *   "tc_bn"          force the tensor-core tile width BN (64, 128, 256; CTA
 *                    pairs use 256)
 *   "tc_cta_group"   force 1- or 2-CTA tiles (1, 2)
 *   "tc_group_m"     raster group height in tiles (>= 1)
 *   "tc_max_ctas"    cap on persistent CTAs (>= 1; static schedule only)
 *   "tc_sched"       tensor-core work schedule: 1 static persistent (each
 *                    CTA or pair strides over the work units), 2 dynamic
 *                    ("Learn CuTeDSL" section 8.2, Cluster Launch Control:
 *                    one cluster per unit is launched and the running ones
 *                    steal the units of clusters that have not started);
 *                    0 auto: static, except grouped launches whose groups'
 *                    K differ by 2x or more (units of unequal cost)
 *   "tc_splits"      force split-K: K ranges for every output tile (1..32);
 *                    the partial tiles go to a workspace and are summed into
 *                    C in a fixed order by a second kernel
 *   "simt_splits"    FP32 (SIMT): 0 auto -- when the tiles cannot give every
 *                    SM about six blocks, K is cut into up to 8 ranges of
 *                    at least 32, their partial sums kept in a stream-ordered
 *                    workspace and added in order by a second kernel (the
 *                    result does not depend on timing); 1 off; n force n
 *   "tc_tail_splits" 0 auto (2 for TF32 when the column halves below do not
 *                    apply, off otherwise), 1 off, n >= 2: split the tiles
 *                    of the last, partly idle round of the persistent
 *                    schedule into n K ranges (same workspace and reduction)
 *   "tc_split_reduce" how the K ranges of split-K tiles are summed: 0 auto
 *                    (in cluster shared memory when every tile is split
 *                    into 2 ranges on single-CTA tiles and the tiles fit one
 *                    round of clusters, else the workspace and second
 *                    kernel), 1 always the workspace and second kernel,
 *                    2 in cluster shared memory where legal (every tile
 *                    split into 2 or 4 ranges, one CTA per range)
 *   "tc_split_lead"  with every tile split into 2 K ranges summed in
 *                    cluster shared memory (or the same shape forced
 *                    through the workspace), 128 columns or fewer and C
 *                    stored by TMA: the percent of k-blocks in the first
 *                    range (the plan's kb_split).  0 auto and 50: an even
 *                    split with the lane quarters shared out (measured
 *                    faster); 51..95 that share, the first range's CTA
 *                    owning the whole tile
 *   "tc_tail_halves" run the last round's tiles as column halves when the
 *                    halves fit in one round and the tile allows it (BN >=
 *                    128; B read as stored in whole 128-byte chunks per
 *                    CTA, or the K-major copy): 0 auto (16-bit inputs on
 *                    schedules of at most 4 rounds), 1 off, 2 wherever the
 *                    tile allows it
 *   "pdl"            0 (default) launch every kernel of the library as a
 *                    programmatic dependent of the previous kernel on the
 *                    stream: its set-up overlaps that kernel's end, and it
 *                    waits for that kernel to finish before touching global
 *                    memory; 1 off
 *   "tc_tma_store"   0 auto, 1 force TMA-store epilogue where legal, 2 force
 *                    ordinary-store epilogue
 *   "simt_variant"   force a SIMT variant: 1 = 128x128 tile, K step 8, 8x8
 *                    outputs per thread; 2 = same with K step 16; 3 = 128x256,
 *                    8x16 per thread; 4 = 256x128, 16x8 per thread; 5 = 64x64;
 *                    6 = 128x256 with K step 16; 7 = 64x64 with K step 16;
 *                    8 = 128x64 and 9 = 64x128 with K step 16, 8x8 per
 *                    thread in 128-thread blocks (9 is the default)
 *   "tc_b_major"     0 auto (BF16, FP16, FP8: B read as stored, N-major, except
 *                    FP8 tiles of 64 columns per CTA; TF32: B read from a
 *                    K-major transposed copy), 1 force the transposed copy,
 *                    2 force reading B as stored (a TF32 call, or an FP8 call
 *                    with 64 columns per CTA, then fails with
 *                    GEMM_ERR_UNSUPPORTED)
 *   "trace_addr"     device address of a trace buffer, 0 = off (see
 *                    gemm_trace_record_t below); "trace_records" its
 *                    capacity in records
 *   "wait_timeout_ms" bound on every in-kernel wait (default 2000)
 *   "debug_stall_mma" test hook: 1 makes the tensor-core kernel's MMA thread
 *                    first wait on a barrier nothing arrives at, so the wait
 *                    expires and gemm_get_status() reports GEMM_ERR_TIMEOUT
 * Returns GEMM_ERR_INVALID_ARG for an unknown key or an out-of-range value.
 */
GEMM_API int gemm_set_option(const char *key, int64_t value);
GEMM_API int64_t gemm_get_option(const char *key);

/* Plan the library would use for a call, computed on the host only (no GPU
 * work, no CUDA calls); pointer addresses matter only for alignment.  The
 * SM count is taken from `num_sms` (pass 0 to query the current device). */
typedef struct {
    int32_t path;        /* 0 SIMT FP32, 1 tensor cores                     */
    int32_t bm, bn, bk;  /* CTA tile (bk in elements)                      */
    int32_t stages;      /* shared-memory ring depth (tensor-core path)    */
    int32_t cta_group;   /* 1 or 2 CTAs per MMA tile                       */
    int32_t group_m;     /* raster group height in tiles                   */
    int32_t grid;        /* CTAs launched                                  */
    int32_t tiles;       /* output tiles                                   */
    int32_t pack_a;      /* A copied to a padded workspace first           */
    int32_t pack_b;      /* B copied to a padded workspace first           */
    int32_t tma_store;   /* epilogue writes C with TMA stores              */
    int32_t vec;         /* SIMT: 16-byte vector loads/stores legal        */
    int32_t smem_bytes;  /* dynamic shared memory per CTA                  */
    int32_t b_kmajor;    /* B staged K-major from a transposed copy (TF32)  */
    int32_t splits;      /* K ranges per split tile (tensor cores) or per
                            SIMT block (FP32); 1 = no split                */
    int32_t tail_tiles;  /* tiles split into K ranges (the last ones in the
                            schedule; all tiles under full split-K)       */
    int32_t sched;       /* 0: static persistent stride over work units;
                            1: Cluster Launch Control (one cluster per unit
                            launched, running CTAs steal the rest)         */
    int32_t half_tiles;  /* tiles run as two column halves (the last ones in
                            the schedule), each half over all of K         */
    int32_t cluster_split; /* 0, or the K ranges (2; 4 on request) of every
                            split tile, run by the CTAs of one cluster and
                            summed in cluster shared memory: no workspace
                            and no second kernel                            */
    int32_t kb_split;    /* 0: K ranges of equal length; else, with 2 ranges,
                            the k-blocks (bk deep) of the first.  Summed in
                            cluster shared memory, the first range's CTA
                            then owns the whole tile and the other sends
                            its partial to it (plain FP32 C stored by TMA;
                            with a fused epilogue each CTA owns half)     */
} gemm_plan_t;

GEMM_API int gemm_plan(int64_t M, int64_t N, int64_t K, int dtype,
              uint64_t a_addr, int64_t lda, uint64_t b_addr, int64_t ldb,
              uint64_t c_addr, int64_t ldc, int32_t num_sms, gemm_plan_t *out);

/*
 * gemm_run_tf32_static -- C = A . B with GEMM_TF32 arithmetic, allocating
 * nothing.  The pages describe no counterpart; this is a service entry point.
 *
 * Who needs it: gemm_run's TF32 path allocates a workspace on the stream for a
 * transposed copy of B.  Callers that cannot allocate device memory while they
 * run -- processes that give all free device memory to their own allocator at
 * start-up, or services that forbid device allocation after start-up because
 * an allocation can block on the device or fragment memory -- use this entry
 * point instead.  Its scratch is one fixed array of
 * GEMM_TF32_STATIC_SCRATCH_BYTES that the library reserves on every GPU it is
 * loaded on and keeps until the process exits.
 *
 * Arguments, layouts, ownership and results are those of gemm_run with
 * dtype = GEMM_TF32 (A, B, C float device pointers, leading dimensions in
 * elements, the caller's stream).  Extra limits, each reported as an error
 * with a message in gemm_last_error():
 *   - N * roundup(K, 4) must not exceed GEMM_TF32_STATIC_SCRATCH_BYTES / 4
 *     floats (GEMM_ERR_INVALID_ARG);
 *   - A must start on a 16-byte boundary with lda a multiple of 4
 *     (GEMM_ERR_UNSUPPORTED): there is no scratch for a copy of A.  So a
 *     contiguous A (lda == K) with K not a multiple of 4 is rejected; pad lda
 *     to a multiple of 4, or call gemm_run.
 * The first call on each device looks up the scratch array's device address
 * (cudaGetSymbolAddress) with that device current, and a call looks it up
 * again when the device's context has changed since (after cudaDeviceReset);
 * make such a call before any stream capture.  All calls share the array and it keeps the last call's
 * contents (no call needs it zeroed); calls whose GPU work overlaps -- e.g. on
 * two unordered streams -- race on it, so order them.
 */
#define GEMM_TF32_STATIC_SCRATCH_BYTES (16 * 1024 * 1024)
GEMM_API int gemm_run_tf32_static(int64_t M, int64_t N, int64_t K,
                                  const float *A, int64_t lda, const float *B, int64_t ldb,
                                  float *C, int64_t ldc, struct CUstream_st *stream);

/*
 * Timeline trace of the tensor-core kernel ("Learn CuTeDSL" section 7: the
 * kernel stamps %globaltimer at points of interest into a global buffer,
 * which the host turns into a timeline).  Off unless the option "trace_addr"
 * holds the device address of a caller-owned buffer of 32 + 32 *
 * "trace_records" bytes (8-byte aligned, device memory of the calling
 * device).  Its first 32 bytes are a header whose first uint32 counts the
 * record slots the kernel has reserved: each recording thread reserves 16 at
 * a time and fills them in turn, so a record costs no atomic of its own.
 * Records follow the header, in no particular order; slots at or beyond
 * "trace_records" are dropped but still counted, and reserved slots a
 * thread did not fill keep the caller's zeros (role 0: skip them).  Zero the
 * whole buffer before a traced call.  The buffer is read only after the
 * stream is synchronised; concurrent traced calls share the buffer.
 */
typedef struct {
    uint64_t t_begin_ns;  /* %globaltimer at the start of the span           */
    uint64_t t_end_ns;    /* %globaltimer at its end                          */
    int32_t unit;         /* work unit (-1: the CTA's whole life)             */
    int16_t role;         /* 1 TMA producer: the unit's loads issued;
                             2 MMA issuer: accumulator free -> last commit;
                             3 epilogue warp: accumulator full -> stored;
                             4 CTA: start -> teardown;
                             5 CTA set-up: sub 0 start -> barriers, Tensor
                               Memory and CTA/cluster barrier done, sub 1
                               -> the previous grid's wait done;
                             6 epilogue detail: sub 0-2 an owning warp of a
                               cluster split (accumulator full -> first
                               partial chunk in -> last chunk in -> last
                               store issued), sub 3 last store issued ->
                               its shared-memory reads done                */
    int16_t sm;           /* %smid                                            */
    int32_t cta;          /* blockIdx.x                                       */
    int32_t sub;          /* roles 1-2: k-blocks of the unit; role 3: lane
                             quarter (+4 when it sends its partial to a
                             cluster peer instead of storing)                 */
} gemm_trace_record_t;

/* Library ABI version (major * 10000 + minor * 100 + patch). */
GEMM_API int gemm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TCGEMM_GEMM_H */
