// gemm_run_tf32_static: the TF32 GEMM without any device allocation.
//
// Why it exists: gemm_run's TF32 path transposes B into a workspace it
// allocates on the stream (cudaMallocAsync / cudaFreeAsync).  Some callers
// cannot allow that: processes that hand all free device memory to their own
// allocator at start-up (a later allocation would fail or push out their
// pool), and services that forbid device allocation once running because an
// allocation can block on the device or fragment memory.  This entry point
// does the same work with its scratch in a fixed array that the library
// reserves on every GPU it is loaded on, and allocates nothing per call.
//
// The scratch: a file-scope __device__ array of GEMM_TF32_STATIC_SCRATCH_BYTES
// (16 MiB), holding the transposed copy of B (N rows of roundup(K, 4) floats).
// Host code cannot use the array's name as a device address, so on the first
// call on each device (with that device current) the entry point asks the
// runtime for the array's device address with cudaGetSymbolAddress and keeps
// it for that device, tagged with the unique id of the context it was looked
// up in.  When the device's current context is another one (after
// cudaDeviceReset, the module -- and with it the array -- is loaded anew), the
// address is looked up again.  A call that does this look-up should come
// before any stream capture.
//
// Every call shares the one array, and it keeps the previous call's contents.
// Nothing in it needs to start at zero: each call's transpose writes every
// element the GEMM then reads.  Calls whose work overlaps on the GPU (for
// example, issued on two streams without ordering between them) race on the
// array; order them on one stream or synchronise between them.
//
// Beyond the scratch it runs exactly what gemm_run runs for GEMM_TF32: the
// same argument checks, planner, transpose kernel and tensor-core kernel.
#include <cudaTypedefs.h>

#include <cstdio>
#include <mutex>

#include "internal.h"

namespace tcgemm {
namespace {

constexpr int64_t kScratchElems = GEMM_TF32_STATIC_SCRATCH_BYTES / 4;

static __device__ __align__(256) float g_tf32_bt_scratch[kScratchElems];

std::mutex g_scratch_mu;
struct ScratchSlot {
    unsigned long long ctx_id = 0;   // unique id of the context the address belongs to
    void *ptr = nullptr;
};
ScratchSlot g_scratch[64];

// Unique id of the calling thread's current context; false if none is current
// or the driver entry points are unavailable.
bool current_context_id(unsigned long long *id) {
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    });
    CUcontext ctx = nullptr;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
    return get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the scratch array on device `dev` (which must be current),
// looked up once per context.
int scratch_address(int dev, void **out) {
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    ScratchSlot &slot = g_scratch[dev];
    unsigned long long id = 0;
    bool have_id = current_context_id(&id);
    if (!slot.ptr || !have_id || slot.ctx_id != id) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_tf32_bt_scratch);   // also makes the context current
        if (e != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            char msg[256];
            std::snprintf(msg, sizeof msg, "cudaGetSymbolAddress of the static scratch failed: %s",
                          cudaGetErrorString(e));
            return api_error(GEMM_ERR_CUDA, msg);
        }
        if (!have_id) have_id = current_context_id(&id);
        if (!have_id) return api_error(GEMM_ERR_CUDA, "no current CUDA context after the scratch look-up");
        slot.ptr = p;
        slot.ctx_id = id;
    }
    *out = slot.ptr;
    return GEMM_OK;
}

}  // namespace
}  // namespace tcgemm

using namespace tcgemm;

extern "C" int gemm_run_tf32_static(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda, const float *B,
                                    int64_t ldb, float *C, int64_t ldc, struct CUstream_st *stream_) {
    api_clear_error();
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    int rc = api_validate(M, N, K, GEMM_TF32, A, lda, B, ldb, C, ldc);
    if (rc) return rc;
    if (M == 0 || N == 0) return GEMM_OK;
    const int64_t ldbt = (K + 3) / 4 * 4;
    if (K > 0 && N * ldbt > kScratchElems) {
        char msg[256];
        std::snprintf(msg, sizeof msg,
                      "N x roundup(K, 4) = %lld floats exceeds the static scratch of %lld floats (%d bytes)",
                      (long long)(N * ldbt), (long long)kScratchElems, (int)GEMM_TF32_STATIC_SCRATCH_BYTES);
        return api_error(GEMM_ERR_INVALID_ARG, msg);
    }
    const uint64_t c0 = (uint64_t)(uintptr_t)C, c1 = c0 + (uint64_t)((M - 1) * ldc + N) * 4u;
    if (K > 0) {
        const uint64_t a0 = (uint64_t)(uintptr_t)A, a1 = a0 + (uint64_t)((M - 1) * lda + K) * 4u;
        const uint64_t b0 = (uint64_t)(uintptr_t)B, b1 = b0 + (uint64_t)((K - 1) * ldb + N) * 4u;
        if ((a0 < c1 && c0 < a1) || (b0 < c1 && c0 < b1)) return api_error(GEMM_ERR_INVALID_ARG, "C overlaps A or B");
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return api_error(GEMM_ERR_CUDA, cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return api_error(GEMM_ERR_UNSUPPORTED, "device ordinal out of range");
    int sms = 0, ccmaj = 0, ccmin = 0, clusters = 0;
    if ((rc = api_device_info(dev, &sms, &ccmaj, &ccmin, &clusters))) return rc;
    if (!(ccmaj == 10 && ccmin == 3)) return api_error(GEMM_ERR_UNSUPPORTED, "this library is built for sm_103a only");
    if ((rc = api_check_device_span("C", C, c1 - c0, dev))) return rc;
    if (K == 0) {
        e = cudaMemset2DAsync(C, (size_t)ldc * 4, 0, (size_t)N * 4, (size_t)M, stream);
        return e == cudaSuccess ? GEMM_OK : api_error(GEMM_ERR_CUDA, cudaGetErrorString(e));
    }
    if ((rc = api_check_device_span("A", A, (uint64_t)((M - 1) * lda + K) * 4u, dev))) return rc;
    if ((rc = api_check_device_span("B", B, (uint64_t)((K - 1) * ldb + N) * 4u, dev))) return rc;

    Options opt = options_snapshot();
    if ((rc = api_check_trace(opt, dev))) return rc;
    opt.tc_b_major = 1;   // B always goes through the transposed copy in the scratch
    opt.tc_splits = 1;    // no workspace for partial sums of split tiles
    opt.tc_tail_splits = 1;
    Plan plan;
    rc = make_plan(M, N, K, GEMM_TF32, (uint64_t)(uintptr_t)A, lda, (uint64_t)(uintptr_t)B, ldb, c0, ldc, sms,
                   clusters, opt, &plan);
    if (rc) return rc;
    if (plan.pub.pack_a)
        return api_error(GEMM_ERR_UNSUPPORTED,
                         "A must start on a 16-byte boundary with lda a multiple of 4 (no scratch for a copy of A)");
    void *bt = nullptr;
    if ((rc = scratch_address(dev, &bt))) return rc;
    e = transpose_launch(B, ldb, bt, ldbt, K, N, 4, stream);
    if (e != cudaSuccess) return api_error(GEMM_ERR_CUDA, cudaGetErrorString(e));
    char err[256] = {0};
    rc = tc_launch(plan.pub, GEMM_TF32, (int)M, (int)N, (int)K, A, lda, bt, ldbt, C, ldc, nullptr, EpiParams(),
                   (uint32_t)opt.wait_timeout_ms, stream, err, sizeof err);
    if (rc != GEMM_OK) return api_error(rc, err);
    return GEMM_OK;
}
