// Exact-FP32 GEMM on the CUDA cores: shared-memory block tiling with register
// micro-tiles.
//
// Design, after "Shared memory and tensor cores" (ml-compiler-from-scratch
// ch. 13):
//  * section 13.1: a BM x BN block tile reads each A/B element from DRAM once
//    per tile, giving BM*BN/(2(BM+BN)) flop/byte (32 for 128 x 128);
//  * sections 13.3-13.4: tiles staged in shared memory, with the read-after-
//    write and write-after-read hazards each closed by a block barrier; here
//    the tiles are double-buffered, so one barrier per K step closes both
//    (section 13.4, last paragraph);
//  * section 13.6: A is stored transposed (k-major) so the inner loop reads
//    contiguous rows; its row pitch is padded by 4 floats, which makes the
//    transposed stores conflict-free under the 32-bank model while keeping
//    16-byte alignment for vector reads (checked in tests/test_simt_layout.py);
//  * section 13.7: each thread owns a register micro-tile of 4 x 4 quads (8 x 8
//    or 8 x 16 outputs), i.e. 64 FMAs per 4 vector loads (8 x 8) or 128 per 6
//    (8 x 16), so shared memory feeds the FMA pipe.
// From "GPU architecture and mapping kernels" (ch. 12) section 12.5: thread x
// runs along the contiguous axis of every global access (coalescing).
//
// Numerics: FP32 fused multiply-adds, one rounding each, k ascending per
// output; no fast-math, no TF32.  The FMAs go two at a time (sm_100's paired
// FP32 FMA on a float2: outputs j and j+1 of a row share a[i]), which halves
// the FMA instructions the issue slots must carry and leaves every result
// bit-identical to fmaf.  Every size >= 1 is legal: out-of-range loads read 0
// and out-of-range stores are skipped.
#include <type_traits>

#include "epilogue.cuh"
#include "internal.h"

namespace tcgemm {
namespace {

// Block tile BM x BN, K step BK; each thread owns RM x RN quads of 4 x 4
// outputs (TM = 4 RM rows, TN = 4 RN columns), its quads BM/RM rows and BN/RN
// columns apart so that every shared read is a 16-byte vector and the lanes of
// a warp read one contiguous run of B.
template <int BM_, int BN_, int BK_, int RM_, int RN_>
struct SimtCfg {
    static constexpr int BM = BM_, BN = BN_, BK = BK_, RM = RM_, RN = RN_;
    static constexpr int TM = 4 * RM, TN = 4 * RN;
    static constexpr int TY = BM / TM, TX = BN / TN;
    static constexpr int THREADS = TY * TX;
    static constexpr int LDS_A = BM + 4;   // padded pitch of the transposed A tile
    static constexpr int LDS_B = BN;
    static constexpr int A_VEC = BM * BK / 4 / THREADS;  // float4 loads per thread
    static constexpr int B_VEC = BK * BN / 4 / THREADS;
    static constexpr int SMEM_BYTES = 2 * BK * (LDS_A + LDS_B) * 4;   // double-buffered
    static_assert(A_VEC >= 1 && B_VEC >= 1, "tile too small for the thread count");
    static_assert(BM * BK / 4 % THREADS == 0 && BK * BN / 4 % THREADS == 0, "uneven tile loads");
    static_assert(TX % 2 == 0 && THREADS % 32 == 0, "warp layout");
};

template <bool VEC>
__device__ __forceinline__ float4 load_row4(const float *__restrict__ p, int64_t row, int64_t col,
                                            int64_t ld, int64_t rows, int64_t cols) {
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (row >= rows) return v;
    const float *q = p + row * ld + col;
    if (VEC && col + 3 < cols) return __ldg(reinterpret_cast<const float4 *>(q));
    if (col + 0 < cols) v.x = __ldg(q + 0);
    if (col + 1 < cols) v.y = __ldg(q + 1);
    if (col + 2 < cols) v.z = __ldg(q + 2);
    if (col + 3 < cols) v.w = __ldg(q + 3);
    return v;
}

template <bool VEC>
__device__ __forceinline__ void store_row4(float *__restrict__ p, int64_t row, int64_t col, int64_t ld,
                                           int64_t rows, int64_t cols, float a, float b, float c, float d) {
    if (row >= rows) return;
    float *q = p + row * ld + col;
    if (VEC && col + 3 < cols) {
        *reinterpret_cast<float4 *>(q) = make_float4(a, b, c, d);
        return;
    }
    if (col + 0 < cols) q[0] = a;
    if (col + 1 < cols) q[1] = b;
    if (col + 2 < cols) q[2] = c;
    if (col + 3 < cols) q[3] = d;
}

template <class Cfg, int MIN_BLOCKS, bool VEC, bool SPLIT>
__global__ void __launch_bounds__(Cfg::THREADS, MIN_BLOCKS)
sgemm_tiled(int M, int N, int K, const float *__restrict__ A, int64_t lda,
            const float *__restrict__ B, int64_t ldb, void *__restrict__ Cv, int64_t ldc, const EpiParams epi,
            int kps, float *__restrict__ W) {
    constexpr int BM = Cfg::BM, BN = Cfg::BN, BK = Cfg::BK, RM = Cfg::RM, RN = Cfg::RN;
    pdl_enter();
    extern __shared__ float4 smem_f4[];
    float *smem = reinterpret_cast<float *>(smem_f4);
    // sA[buf][k][m] (transposed, padded pitch), then sB[buf][k][n].
    auto sA = [&](int buf, int k) { return smem + (buf * BK + k) * Cfg::LDS_A; };
    auto sB = [&](int buf, int k) { return smem + 2 * BK * Cfg::LDS_A + (buf * BK + k) * Cfg::LDS_B; };

    const int tid = threadIdx.x;
    const int tx = tid % Cfg::TX, ty = tid / Cfg::TX;
    const int64_t m0 = (int64_t)blockIdx.y * BM;
    const int64_t n0 = (int64_t)blockIdx.x * BN;
    // Split K (a separate instance, so the whole-K kernel carries none of
    // it): block z sums k in [kb, ke) (kps a multiple of BK, so vector loads
    // stay aligned) and leaves its partial in W[z].
    const int kb = SPLIT ? (int)blockIdx.z * kps : 0;
    const int ke = SPLIT ? min(K, kb + kps) : K;

    float4 ra[Cfg::A_VEC], rb[Cfg::B_VEC];

    // Global -> registers: A rows of BK floats (BK/4 vectors each), B rows of BN floats.
    auto fetch = [&](int k0) {
#pragma unroll
        for (int i = 0; i < Cfg::A_VEC; ++i) {
            const int f = tid + i * Cfg::THREADS;
            const int r = f / (BK / 4), kq = f % (BK / 4);
            ra[i] = load_row4<VEC>(A, m0 + r, (int64_t)kb + k0 + 4 * kq, lda, M, ke);
        }
#pragma unroll
        for (int i = 0; i < Cfg::B_VEC; ++i) {
            const int f = tid + i * Cfg::THREADS;
            const int kr = f / (BN / 4), c4 = f % (BN / 4);
            rb[i] = load_row4<VEC>(B, (int64_t)kb + k0 + kr, n0 + 4 * c4, ldb, ke, N);
        }
    };
    // Registers -> shared buffer `buf`: A transposed to [k][m], B as is.
    auto deposit = [&](int buf) {
#pragma unroll
        for (int i = 0; i < Cfg::A_VEC; ++i) {
            const int f = tid + i * Cfg::THREADS;
            const int r = f / (BK / 4), kq = f % (BK / 4);
            sA(buf, 4 * kq + 0)[r] = ra[i].x;
            sA(buf, 4 * kq + 1)[r] = ra[i].y;
            sA(buf, 4 * kq + 2)[r] = ra[i].z;
            sA(buf, 4 * kq + 3)[r] = ra[i].w;
        }
#pragma unroll
        for (int i = 0; i < Cfg::B_VEC; ++i) {
            const int f = tid + i * Cfg::THREADS;
            const int kr = f / (BN / 4), c4 = f % (BN / 4);
            *reinterpret_cast<float4 *>(sB(buf, kr) + 4 * c4) = rb[i];
        }
    };

    // acc2[i][j] holds outputs (i, 2j) and (i, 2j + 1) of the micro-tile.
    float2 acc2[4 * RM][2 * RN];
#pragma unroll
    for (int i = 0; i < 4 * RM; ++i)
#pragma unroll
        for (int j = 0; j < 2 * RN; ++j) acc2[i][j] = make_float2(0.f, 0.f);
    auto acc = [&](int i, int j) -> float { return (j & 1) ? acc2[i][j >> 1].y : acc2[i][j >> 1].x; };

    const int ktiles = ke > kb ? (ke - kb + BK - 1) / BK : 0;
    // One K step on buffer BUF (a compile-time constant, so every shared
    // address below is a fixed offset from one base register).
    auto step = [&](auto buf_c, int kt) {
        constexpr int buf = decltype(buf_c)::value;
        const bool more = kt + 1 < ktiles;   // uniform across the block
        if (more) fetch((kt + 1) * BK);      // in flight while we compute
#pragma unroll
        for (int k = 0; k < BK; ++k) {
            float a[4 * RM], b[4 * RN];
#pragma unroll
            for (int q = 0; q < RM; ++q) {
                const float4 v = *reinterpret_cast<const float4 *>(sA(buf, k) + q * (BM / RM) + ty * 4);
                a[4 * q + 0] = v.x; a[4 * q + 1] = v.y; a[4 * q + 2] = v.z; a[4 * q + 3] = v.w;
            }
#pragma unroll
            for (int q = 0; q < RN; ++q) {
                const float4 v = *reinterpret_cast<const float4 *>(sB(buf, k) + q * (BN / RN) + tx * 4);
                b[4 * q + 0] = v.x; b[4 * q + 1] = v.y; b[4 * q + 2] = v.z; b[4 * q + 3] = v.w;
            }
#pragma unroll
            for (int i = 0; i < 4 * RM; ++i) {
                const float2 ai = make_float2(a[i], a[i]);
#pragma unroll
                for (int j = 0; j < 2 * RN; ++j)
                    acc2[i][j] = __ffma2_rn(ai, make_float2(b[2 * j], b[2 * j + 1]), acc2[i][j]);
            }
        }
        // The other buffer was last read before the previous barrier, so it can
        // be refilled now; the barrier below publishes it and also keeps this
        // buffer intact until every warp has finished reading it.
        if (more) deposit(buf ^ 1);
        __syncthreads();
    };
    fetch(0);
    deposit(0);
    __syncthreads();
    for (int kt = 0; kt < ktiles; kt += 2) {
        step(std::integral_constant<int, 0>{}, kt);
        if (kt + 1 < ktiles) step(std::integral_constant<int, 1>{}, kt + 1);
    }

    if constexpr (SPLIT) {
        // A K range's partial sums, raw: W[z] is M x N, row-major.
        float *w = W + (int64_t)blockIdx.z * M * N;
        const bool wvec = VEC && (N % 4 == 0);
#pragma unroll
        for (int i = 0; i < 4 * RM; ++i) {
            const int64_t row = m0 + (i / 4) * (BM / RM) + ty * 4 + (i % 4);
#pragma unroll
            for (int q = 0; q < RN; ++q) {
                const int64_t col = n0 + q * (BN / RN) + tx * 4;
                if (wvec)
                    store_row4<true>(w, row, col, N, M, N, acc(i, 4 * q + 0), acc(i, 4 * q + 1), acc(i, 4 * q + 2),
                                     acc(i, 4 * q + 3));
                else
                    store_row4<false>(w, row, col, N, M, N, acc(i, 4 * q + 0), acc(i, 4 * q + 1), acc(i, 4 * q + 2),
                                      acc(i, 4 * q + 3));
            }
        }
        return;
    }
    if (epi.active) {
        // Fused epilogue: element by element, each column's bias read once.
        float bias[4 * RN];
#pragma unroll
        for (int j = 0; j < 4 * RN; ++j) bias[j] = epi_bias(epi, n0 + (j / 4) * (BN / RN) + tx * 4 + (j % 4), N);
#pragma unroll
        for (int i = 0; i < 4 * RM; ++i) {
            const int64_t row = m0 + (i / 4) * (BM / RM) + ty * 4 + (i % 4);
            if (row >= M) continue;
#pragma unroll
            for (int j = 0; j < 4 * RN; ++j) {
                const int64_t col = n0 + (j / 4) * (BN / RN) + tx * 4 + (j % 4);
                if (col < N) epi_write(epi, Cv, row * ldc + col, acc(i, j), bias[j]);
            }
        }
        return;
    }
    float *C = static_cast<float *>(Cv);
#pragma unroll
    for (int i = 0; i < 4 * RM; ++i) {
        const int64_t row = m0 + (i / 4) * (BM / RM) + ty * 4 + (i % 4);
#pragma unroll
        for (int q = 0; q < RN; ++q)
            store_row4<VEC>(C, row, n0 + q * (BN / RN) + tx * 4, ldc, M, N, acc(i, 4 * q + 0), acc(i, 4 * q + 1),
                            acc(i, 4 * q + 2), acc(i, 4 * q + 3));
    }
}

// Sums the K ranges' partials W[0..splits) in order (so the result does not
// depend on which block finished first) and writes C through the epilogue.
__global__ void __launch_bounds__(256) simt_split_reduce(const float *__restrict__ W, int splits, int64_t M,
                                                         int64_t N, void *__restrict__ C, int64_t ldc,
                                                         const EpiParams epi) {
    pdl_enter();
    const int64_t total = M * N;
    for (int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; x < total; x += (int64_t)gridDim.x * blockDim.x) {
        float v = W[x];
        for (int z = 1; z < splits; ++z) v += W[(int64_t)z * total + x];
        const int64_t r = x / N, c = x - r * N;
        if (epi.active) epi_write(epi, C, r * ldc + c, v, epi_bias(epi, c, N));
        else static_cast<float *>(C)[r * ldc + c] = v;
    }
}

template <class Cfg, int MIN_BLOCKS>
cudaError_t launch_tile(bool vec, int M, int N, int K, const float *A, int64_t lda, const float *B,
                        int64_t ldb, void *C, int64_t ldc, const EpiParams &epi, int splits, float *W,
                        cudaStream_t s) {
    const int kps = splits > 1 ? (((K + splits - 1) / splits + Cfg::BK - 1) / Cfg::BK) * Cfg::BK : 0;
    const dim3 grid((unsigned)((N + Cfg::BN - 1) / Cfg::BN), (unsigned)((M + Cfg::BM - 1) / Cfg::BM),
                    (unsigned)(splits > 1 ? splits : 1));
    if (grid.y > 65535u || (splits > 1 && !W)) return cudaErrorInvalidConfiguration;
    auto kern = splits > 1 ? (vec ? sgemm_tiled<Cfg, MIN_BLOCKS, true, true> : sgemm_tiled<Cfg, MIN_BLOCKS, false, true>)
                           : (vec ? sgemm_tiled<Cfg, MIN_BLOCKS, true, false> : sgemm_tiled<Cfg, MIN_BLOCKS, false, false>);
    if (Cfg::SMEM_BYTES > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
        if (e != cudaSuccess) return e;
    }
    return launch_pdl(kern, grid, dim3(Cfg::THREADS), Cfg::SMEM_BYTES, s, M, N, K, A, lda, B, ldb, C, ldc, epi, kps,
                      splits > 1 ? W : nullptr);
}

// The compiled variants: id, tile, K step, quads per thread, min resident blocks.
#define SIMT_VARIANTS(X)          \
    X(1, 128, 128, 8, 2, 2, 2)    \
    X(2, 128, 128, 16, 2, 2, 1)   \
    X(3, 128, 256, 8, 2, 4, 1)    \
    X(4, 256, 128, 8, 4, 2, 1)    \
    X(5, 64, 64, 8, 2, 2, 4)      \
    X(6, 128, 256, 16, 2, 4, 1)   \
    X(7, 64, 64, 16, 2, 2, 4)     \
    X(8, 128, 64, 16, 2, 2, 3)    \
    X(9, 64, 128, 16, 2, 2, 3)

}  // namespace

cudaError_t simt_fp32_launch(const gemm_plan_t &plan, int M, int N, int K, const float *A, int64_t lda,
                             const float *B, int64_t ldb, void *C, int64_t ldc, const EpiParams &epi, float *W,
                             cudaStream_t stream) {
    const int splits = plan.splits > 1 ? plan.splits : 1;
    cudaError_t e = cudaErrorInvalidValue;
    // if (variant 1) e = ...; else if (variant 2) e = ...; ... else return (no such tile)
#define X(id_, bm_, bn_, bk_, rm_, rn_, minb_)                                                        \
    if (plan.bm == bm_ && plan.bn == bn_ && plan.bk == bk_)                                             \
        e = launch_tile<SimtCfg<bm_, bn_, bk_, rm_, rn_>, minb_>(plan.vec != 0, M, N, K, A, lda, B, ldb, C, \
                                                                 ldc, epi, splits, W, stream);          \
    else
    SIMT_VARIANTS(X)
#undef X
    return cudaErrorInvalidValue;
    if (e != cudaSuccess || splits == 1) return e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const int64_t want = ((int64_t)M * N + 255) / 256;
    const dim3 grid((unsigned)(want < (int64_t)sms * 8 ? (want > 0 ? want : 1) : (int64_t)sms * 8));
    return launch_pdl(simt_split_reduce, grid, dim3(256), 0, stream, W, splits, (int64_t)M, (int64_t)N, C, ldc, epi);
}

int simt_variant_tile(int id, int *bm, int *bn, int *bk, int *smem) {
#define X(id_, bm_, bn_, bk_, rm, rn, minb)                   \
    if (id == id_) {                                           \
        *bm = bm_;                                             \
        *bn = bn_;                                             \
        *bk = bk_;                                             \
        *smem = SimtCfg<bm_, bn_, bk_, rm, rn>::SMEM_BYTES;    \
        return 1;                                              \
    }
    SIMT_VARIANTS(X)
#undef X
    return 0;
}

}  // namespace tcgemm
