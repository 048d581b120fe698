// Internal interfaces between the library's translation units (not installed).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gemm.h"

namespace tcgemm {

// ---------------------------------------------------------------- options ---
struct Options {
    int tc_bn = 0;             // 0 auto, else 64/128/256
    int tc_cta_group = 0;      // 0 auto, else 1/2
    int tc_group_m = 0;        // 0 auto
    int tc_max_ctas = 0;       // 0 auto
    int tc_splits = 0;         // 0 auto, else K ranges for every tile (split-K)
    int tc_tail_splits = 0;    // 0 auto (2 for TF32), 1 off, else K ranges for the last round's tiles
    int pdl = 0;               // 0 on, 1 off: programmatic dependent launch of every kernel
    int simt_splits = 0;       // 0 auto, 1 off, n: K ranges for the SIMT kernel
    int tc_tail_halves = 0;    // 0 auto (16-bit inputs, <= 4 rounds), 1 off, 2 wherever the tile allows
    int tc_sched = 0;          // 0 auto, 1 static persistent, 2 Cluster Launch Control
    int tc_tma_store = 0;      // 0 auto, 1 force TMA store, 2 force plain stores
    int simt_variant = 0;      // 0 auto, else a compiled SIMT variant id (1..6)
    int tc_b_major = 0;        // 0 auto (as stored; FP8 narrow tiles transposed), 1 K-major copy, 2 as stored
    int tc_split_reduce = 0;   // 0 auto, 1 workspace + reduce kernel, 2 cluster shared memory
    int tc_split_lead = 0;     // two K ranges: percent of k-blocks in the first (0 auto, 50 even)
    int wait_timeout_ms = 2000;
    int64_t trace_addr = 0;    // device address of a trace buffer (0: off)
    int trace_records = 0;     // its capacity in records
    int debug_stall_mma = 0;   // test hook: make the MMA thread's first wait expire
};
Options options_snapshot();

// Programmatic dependent launch, used by every kernel of the library: a
// launch may start while the previous kernel on the stream finishes; each
// kernel waits for that kernel (griddepcontrol.wait) before its first
// global-memory access, and then lets the next launch start its own set-up.
// The host side: cudaLaunchKernelEx with programmatic stream serialisation
// (unless the "pdl" option turns it off).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (options_snapshot().pdl != 1) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

#ifdef __CUDACC__
// The device side, at the top of a kernel that needs nothing from before it
// but its arguments: wait for the previous grid, then release the next one.
__device__ __forceinline__ void pdl_enter() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
#endif

// --------------------------------------------------------------- epilogue ---
// Fused epilogue of one call (gemm_run_ex).  active == 0: C is FP32 and gets
// the accumulator as is (gemm_run); the other fields are then ignored.
struct EpiParams {
    float alpha = 1.f;
    float beta = 0.f;
    const float *bias = nullptr;   // N floats or nullptr
    int act = GEMM_ACT_NONE;
    int out = GEMM_OUT_F32;
    int active = 0;
};

// ------------------------------------------------------------ grouped GEMM ---
// One GEMM of a grouped launch as the tensor-core kernel reads it from device
// memory ("Learn CuTeDSL" section 8.4: the tiles of every group flattened into
// one list of work units, unit_start being the group's first).  The TMA
// descriptors come first: they must be 64-byte aligned.
struct alignas(128) GroupDesc {
    CUtensorMap tmA, tmB, tmC;
    int32_t M, N, num_kb, tiles_m, tiles_n, unit_start, tma_store, reserved;
    void *C;
    int64_t ldc;
    const float *bias;
};

// ------------------------------------------------------------------- plan ---
struct Plan {
    gemm_plan_t pub;           // what gemm_plan() reports
    int64_t lda_eff, ldb_eff;  // leading dimensions the kernel sees (after packing)
};

// Picks path, tile, ring depth, CTA group and grid for one call.  Host only.
int make_plan(int64_t M, int64_t N, int64_t K, int dtype,
              uint64_t a_addr, int64_t lda, uint64_t b_addr, int64_t ldb,
              uint64_t c_addr, int64_t ldc, int num_sms, int max_clusters_2cta,
              const Options &opt, Plan *out);

// ------------------------------------------------------------------- SIMT ---
// C = A.B in exact FP32 with the tile the plan chose, written through `epi`
// (C's element type is epi.out when epi.active, else FP32).  With
// plan.splits > 1, K is cut into that many ranges whose partial sums go to W
// (plan.splits x M x N floats) and a second kernel adds them in order.
cudaError_t simt_fp32_launch(const gemm_plan_t &plan, int M, int N, int K,
                             const float *A, int64_t lda, const float *B, int64_t ldb,
                             void *C, int64_t ldc, const EpiParams &epi, float *W, cudaStream_t stream);

// Tile of SIMT variant `id` (bm, bn, bk, dynamic shared bytes); 0 if unknown.
int simt_variant_tile(int id, int *bm, int *bn, int *bk, int *smem);

// ----------------------------------------------------------- tensor cores ---
// Fills plan-dependent shared-memory size (bytes) for a tensor-core variant,
// or returns 0 if the variant is not compiled in.
// b_kmajor: 1 = B from a K-major transposed copy, 0 = B as stored.
int tc_smem_bytes(int dtype, int cta_group, int bn, int b_kmajor);
int tc_stages(int dtype, int cta_group, int bn, int b_kmajor);
// 1 if the variant can run a tile as two column halves (plan.half_tiles).
int tc_halves_ok(int dtype, int cta_group, int bn, int b_kmajor);

// Encodes the tensor maps and launches the persistent kernel.  A/B are the
// (possibly packed) operands with the leading dimensions the plan reports;
// with plan.b_kmajor, B is the transposed copy (N x K, leading dimension ldb).
// W: the slabs for the split tiles' partial sums (plan.tail_tiles * plan.splits
// tiles of (128 * cta_group) x bn floats), or nullptr if no tile is split.
// Whole tiles are written through `epi` (C's element type is epi.out when the
// epilogue is active; plan.tma_store then refers to that type).  Returns a
// gemm_status_t.
int tc_launch(const gemm_plan_t &plan, int dtype, int M, int N, int K,
              const void *A, int64_t lda, const void *B, int64_t ldb,
              void *C, int64_t ldc, float *W, const EpiParams &epi, uint32_t timeout_ms, cudaStream_t stream,
              char *err, size_t errlen);

// Grouped launch: encodes one group's tensor maps into `d` (A and B as the
// plan stages them, C in the output type when d->tma_store); returns a
// gemm_status_t.
int tc_encode_group(const gemm_plan_t &plan, int dtype, GroupDesc *d, const void *A, int64_t lda, const void *B,
                    int64_t ldb, void *C, int64_t ldc, int out, int M, int N, int K, char *err, size_t errlen);

// Launches the persistent kernel over `group_count` groups whose descriptors
// are in device memory (unit_start ascending, every group non-empty with
// K > 0) and `num_units` units in all.
int tc_launch_grouped(const gemm_plan_t &plan, int dtype, const GroupDesc *groups, int group_count, int num_units,
                      const EpiParams &epi, uint32_t timeout_ms, cudaStream_t stream, char *err, size_t errlen);

// Reads and clears the device status word of the tensor-core kernel.
// words[0] = error code (0 none), [1] = role, [2] = tile, [3] = block.
cudaError_t tc_read_and_clear_status(uint32_t words[4]);

// Max co-resident 2-CTA clusters of the widest 2-CTA variant (0 if unknown).
int tc_max_active_clusters(int device);

// ------------------------------------------------------------------- pack ---
// dst[r * ld_dst + c] = src[r * ld_src + c] for r < rows, c < cols (elem bytes
// each); dst columns [cols, ld_dst) are zeroed.  [src_lo, src_hi) is memory
// the kernel may read (the source allocation; at least the footprint).
cudaError_t pack_rows_launch(const void *src, int64_t ld_src, void *dst, int64_t ld_dst,
                             int64_t rows, int64_t cols, int elem_bytes, uint64_t src_lo, uint64_t src_hi,
                             cudaStream_t stream);

// For each split tile i (tile index full_tiles + i in the raster order), sums
// its `splits` slabs W[(s * tail_tiles + i) * tile_rows * tile_cols ...] in
// split order into C (clipped to M x N), through `epi`.
cudaError_t split_reduce_launch(const float *W, int tail_tiles, int splits, int tile_rows, int tile_cols,
                                int full_tiles, int tiles_m, int tiles_n, int group_m, void *C, int64_t ldc,
                                int64_t M, int64_t N, const EpiParams &epi, cudaStream_t stream);

// C = epilogue of a zero accumulator (the K = 0 product) over M x N.
cudaError_t epilogue_fill_launch(void *C, int64_t ldc, int64_t M, int64_t N, const EpiParams &epi,
                                 cudaStream_t stream);

// dst[c * ld_dst + r] = src[r * ld_src + c] for r < rows, c < cols.
cudaError_t transpose_launch(const void *src, int64_t ld_src, void *dst, int64_t ld_dst,
                             int64_t rows, int64_t cols, int elem_bytes, cudaStream_t stream);

// ------------------------------------------- helpers shared by entry points ---
// Defined in gemm_api.cu.  api_error records a message for gemm_last_error()
// and returns `code`; the others are the argument, pointer and device checks
// gemm_run applies.
int api_error(int code, const char *message);
void api_clear_error();
int api_validate(int64_t M, int64_t N, int64_t K, int dtype, const void *A, int64_t lda, const void *B,
                 int64_t ldb, const void *C, int64_t ldc);
int api_check_device_span(const char *name, const void *p, uint64_t bytes, int dev);
// The trace buffer named by the options, if any, is device memory of `dev` with room for its records.
int api_check_trace(const Options &opt, int dev);
// The same, also reporting the allocation [*lo, *hi) that holds the span.
int api_check_device_span_range(const char *name, const void *p, uint64_t bytes, int dev, uint64_t *lo,
                                uint64_t *hi);
// gemm_epilogue_t -> EpiParams (NULL: inactive); checks the enumerations.
int api_epilogue(const gemm_epilogue_t *in, EpiParams *out);
// Element size in bytes of a gemm_dtype_t's operands.
int api_elem_bytes(int dtype);
int api_device_info(int dev, int *sms, int *cc_major, int *cc_minor, int *max_clusters);

}  // namespace tcgemm
