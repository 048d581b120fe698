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
//  * section 13.7: each thread owns an 8 x 8 micro-tile (two 4 x 4 quads per
//    axis, half a tile apart, so every shared load is a 16-byte vector and a
//    warp's B reads are contiguous), i.e. 64 FMAs per 4 vector loads.
// From "GPU architecture and mapping kernels" (ch. 12) section 12.5: thread x
// runs along the contiguous axis of every global access (coalescing).
//
// Numerics: plain FP32 fmaf with k ascending per output; no fast-math, no
// TF32.  Every size >= 1 is legal: out-of-range loads read 0 and out-of-range
// stores are skipped.
#include "internal.h"

namespace tcgemm {
namespace {

template <int BM_, int BN_, int BK_>
struct SimtCfg {
    static constexpr int BM = BM_, BN = BN_, BK = BK_;
    static constexpr int TM = 8, TN = 8;
    static constexpr int TY = BM / TM, TX = BN / TN;
    static constexpr int THREADS = TY * TX;
    static constexpr int LDS_A = BM + 4;   // padded pitch of the transposed A tile
    static constexpr int LDS_B = BN;
    static constexpr int A_VEC = BM * BK / 4 / THREADS;  // float4 loads per thread
    static constexpr int B_VEC = BK * BN / 4 / THREADS;
    static_assert(A_VEC >= 1 && B_VEC >= 1, "tile too small for the thread count");
    static_assert(BM * BK / 4 % THREADS == 0 && BK * BN / 4 % THREADS == 0, "uneven tile loads");
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

template <int BM, int BN, int BK, bool VEC>
__global__ void __launch_bounds__(SimtCfg<BM, BN, BK>::THREADS, (BM == 128 ? 2 : 4))
sgemm_tiled(int M, int N, int K, const float *__restrict__ A, int64_t lda,
            const float *__restrict__ B, int64_t ldb, float *__restrict__ C, int64_t ldc) {
    using Cfg = SimtCfg<BM, BN, BK>;
    __shared__ __align__(16) float sA[2][BK][Cfg::LDS_A];
    __shared__ __align__(16) float sB[2][BK][Cfg::LDS_B];

    const int tid = threadIdx.x;
    const int tx = tid % Cfg::TX, ty = tid / Cfg::TX;
    const int64_t m0 = (int64_t)blockIdx.y * BM;
    const int64_t n0 = (int64_t)blockIdx.x * BN;

    float4 ra[Cfg::A_VEC], rb[Cfg::B_VEC];

    // Global -> registers: A rows of BK floats (BK/4 vectors each), B rows of BN floats.
    auto fetch = [&](int k0) {
#pragma unroll
        for (int i = 0; i < Cfg::A_VEC; ++i) {
            const int f = tid + i * Cfg::THREADS;
            const int r = f / (BK / 4), kq = f % (BK / 4);
            ra[i] = load_row4<VEC>(A, m0 + r, (int64_t)k0 + 4 * kq, lda, M, K);
        }
#pragma unroll
        for (int i = 0; i < Cfg::B_VEC; ++i) {
            const int f = tid + i * Cfg::THREADS;
            const int kr = f / (BN / 4), c4 = f % (BN / 4);
            rb[i] = load_row4<VEC>(B, (int64_t)k0 + kr, n0 + 4 * c4, ldb, K, N);
        }
    };
    // Registers -> shared buffer `buf`: A transposed to [k][m], B as is.
    auto deposit = [&](int buf) {
#pragma unroll
        for (int i = 0; i < Cfg::A_VEC; ++i) {
            const int f = tid + i * Cfg::THREADS;
            const int r = f / (BK / 4), kq = f % (BK / 4);
            sA[buf][4 * kq + 0][r] = ra[i].x;
            sA[buf][4 * kq + 1][r] = ra[i].y;
            sA[buf][4 * kq + 2][r] = ra[i].z;
            sA[buf][4 * kq + 3][r] = ra[i].w;
        }
#pragma unroll
        for (int i = 0; i < Cfg::B_VEC; ++i) {
            const int f = tid + i * Cfg::THREADS;
            const int kr = f / (BN / 4), c4 = f % (BN / 4);
            *reinterpret_cast<float4 *>(&sB[buf][kr][4 * c4]) = rb[i];
        }
    };

    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

    const int ktiles = (K + BK - 1) / BK;
    fetch(0);
    deposit(0);
    __syncthreads();
    for (int kt = 0; kt < ktiles; ++kt) {
        const int buf = kt & 1;
        const bool more = kt + 1 < ktiles;   // uniform across the block
        if (more) fetch((kt + 1) * BK);      // in flight while we compute
#pragma unroll
        for (int k = 0; k < BK; ++k) {
            const float4 a0 = *reinterpret_cast<const float4 *>(&sA[buf][k][ty * 4]);
            const float4 a1 = *reinterpret_cast<const float4 *>(&sA[buf][k][BM / 2 + ty * 4]);
            const float4 b0 = *reinterpret_cast<const float4 *>(&sB[buf][k][tx * 4]);
            const float4 b1 = *reinterpret_cast<const float4 *>(&sB[buf][k][BN / 2 + tx * 4]);
            const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        // The other buffer was last read before the previous barrier, so it can
        // be refilled now; the barrier below publishes it and also keeps this
        // buffer intact until every warp has finished reading it.
        if (more) deposit(buf ^ 1);
        __syncthreads();
    }

#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t row = m0 + (i < 4 ? ty * 4 + i : BM / 2 + ty * 4 + (i - 4));
        store_row4<VEC>(C, row, n0 + tx * 4, ldc, M, N, acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
        store_row4<VEC>(C, row, n0 + BN / 2 + tx * 4, ldc, M, N, acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
    }
}

template <int BM, int BN, int BK>
cudaError_t launch_tile(bool vec, int M, int N, int K, const float *A, int64_t lda, const float *B,
                        int64_t ldb, float *C, int64_t ldc, cudaStream_t s) {
    using Cfg = SimtCfg<BM, BN, BK>;
    const dim3 grid((unsigned)((N + BN - 1) / BN), (unsigned)((M + BM - 1) / BM));
    if (grid.y > 65535u) return cudaErrorInvalidConfiguration;
    if (vec)
        sgemm_tiled<BM, BN, BK, true><<<grid, Cfg::THREADS, 0, s>>>(M, N, K, A, lda, B, ldb, C, ldc);
    else
        sgemm_tiled<BM, BN, BK, false><<<grid, Cfg::THREADS, 0, s>>>(M, N, K, A, lda, B, ldb, C, ldc);
    return cudaGetLastError();
}

}  // namespace

cudaError_t simt_fp32_launch(const gemm_plan_t &plan, int M, int N, int K, const float *A, int64_t lda,
                             const float *B, int64_t ldb, float *C, int64_t ldc, cudaStream_t stream) {
    if (plan.bm == 128) return launch_tile<128, 128, 8>(plan.vec != 0, M, N, K, A, lda, B, ldb, C, ldc, stream);
    if (plan.bm == 64) return launch_tile<64, 64, 8>(plan.vec != 0, M, N, K, A, lda, B, ldb, C, ldc, stream);
    return cudaErrorInvalidValue;
}

}  // namespace tcgemm
