// Operand pack and transpose.
//
// Pack: copy a row-major matrix into a buffer whose row pitch the TMA
// engine can address.  "Learn CuTeDSL" section 3.4: every stride of a TMA
// tensor other than the contiguous one must be a multiple of 16 bytes (and the
// base 16-byte aligned); a K x N BF16 matrix with N = 4095 has an 8190-byte
// pitch and cannot be described.  The copy rounds the pitch up to a multiple of
// 16 bytes and zero-fills the extra columns.
//
// Transpose: B (K x N, N contiguous) -> B^T (N x K, K contiguous) for the
// paths whose MMA reads B K-major (TF32; FP8 tiles narrower than 128 columns).
//
// Split reduce: sum the partial tiles of split tiles into C, through the
// fused epilogue.  Epilogue fill: the epilogue of a zero product (K = 0).
//
// Both are HBM-bound: one read and one write of the operand.  The grid is a multiple of
// the SM count; each warp walks whole rows so both sides stay coalesced even
// though the source rows start at arbitrary 2- or 4-byte offsets.
#include <cstring>

#include "epilogue.cuh"
#include "internal.h"
#include "tile_order.cuh"

namespace tcgemm {
namespace {

template <typename T>
__global__ void __launch_bounds__(256) pack_rows(const T *__restrict__ src, int64_t ld_src, T *__restrict__ dst,
                                                 int64_t ld_dst, int64_t rows, int64_t cols) {
    pdl_enter();
    const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x / 32);
    const int64_t warp = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    for (int64_t r = warp; r < rows; r += warps_total) {
        const T *s = src + r * ld_src;
        T *d = dst + r * ld_dst;
        for (int64_t c = lane; c < ld_dst; c += 32) d[c] = c < cols ? s[c] : T(0);
    }
}

// Vector pack: one thread per destination 16-byte chunk (consecutive threads
// along a row, so loads and stores coalesce).  A source row starts at an arbitrary ELEM-aligned
// address s; chunk j's bytes [s + 16j, s + 16j + 16) straddle the aligned
// words w0 = (s & ~15) + 16j and w0 + 16, so the thread loads both and
// funnel-shifts them by s & 15 bytes.  A word is read
// only if it lies inside [lo, hi), the source allocation; otherwise that
// chunk is copied element by element from inside the row.  Destination bytes
// past the row's end (the pitch padding) are written as zero.
__device__ __forceinline__ uint4 shift_words(const uint32_t (&v)[8], int ws, int hs) {
    auto f = [&](int k) { return __funnelshift_r(v[k], v[k + 1], hs); };
    switch (ws) {
        case 0: return make_uint4(f(0), f(1), f(2), f(3));
        case 1: return make_uint4(f(1), f(2), f(3), f(4));
        case 2: return make_uint4(f(2), f(3), f(4), f(5));
        default: return make_uint4(f(3), f(4), f(5), f(6));
    }
}

__device__ __forceinline__ uint32_t keep_bytes(uint32_t w, int nbytes) {
    return nbytes >= 4 ? w : nbytes <= 0 ? 0u : (w & ((1u << (8 * nbytes)) - 1u));
}

template <int ELEM>
__global__ void __launch_bounds__(256) pack_rows_vec(const uint8_t *__restrict__ src, int64_t ld_src_bytes,
                                                     uint8_t *__restrict__ dst, int64_t ld_dst_bytes, int64_t rows,
                                                     int64_t row_bytes, uintptr_t lo, uintptr_t hi) {
    pdl_enter();
    // one thread per destination 16-byte chunk, consecutive threads along a row
    const int64_t chunks = ld_dst_bytes / 16;
    const int64_t total = rows * chunks;
    for (int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; x < total; x += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = x / chunks, c = x - r * chunks;
        const uintptr_t s = reinterpret_cast<uintptr_t>(src) + (uintptr_t)(r * ld_src_bytes);
        const uintptr_t a = s & ~(uintptr_t)15;
        const int off = (int)(s - a);
        const int ws = off >> 2, hs = (off & 3) * 8;
        const int64_t b0 = 16 * c;   // first byte of this chunk within the row
        uint4 out = make_uint4(0u, 0u, 0u, 0u);
        if (b0 < row_bytes) {
            const uintptr_t w0 = a + (uintptr_t)b0;
            const uintptr_t need = off ? 32 : 16;
            if (w0 >= lo && w0 + need <= hi) {
                const uint4 xw = *reinterpret_cast<const uint4 *>(w0);
                const uint4 yw = off ? *reinterpret_cast<const uint4 *>(w0 + 16) : make_uint4(0u, 0u, 0u, 0u);
                const uint32_t v[8] = {xw.x, xw.y, xw.z, xw.w, yw.x, yw.y, yw.z, yw.w};
                out = shift_words(v, ws, hs);
            } else {
                uint32_t wds[4] = {0u, 0u, 0u, 0u};
                for (int e = 0; e < 16 / ELEM && b0 + e * ELEM < row_bytes; ++e) {
                    const uint32_t val = ELEM == 1   ? (uint32_t)*reinterpret_cast<const uint8_t *>(s + b0 + e)
                                         : ELEM == 2 ? (uint32_t)*reinterpret_cast<const uint16_t *>(s + b0 + e * 2)
                                                     : *reinterpret_cast<const uint32_t *>(s + b0 + e * 4);
                    const int bit = e * ELEM * 8;
                    wds[bit / 32] |= val << (bit % 32);
                }
                out = make_uint4(wds[0], wds[1], wds[2], wds[3]);
            }
            const int keep = (int)(row_bytes - b0);   // bytes of this chunk inside the row
            if (keep < 16) {
                out.x = keep_bytes(out.x, keep);
                out.y = keep_bytes(out.y, keep - 4);
                out.z = keep_bytes(out.z, keep - 8);
                out.w = keep_bytes(out.w, keep - 12);
            }
        }
        *reinterpret_cast<uint4 *>(dst + r * ld_dst_bytes + b0) = out;
    }
}

// 32 x 32 tiles through shared memory so both the read of `src` rows and the
// write of `dst` rows are coalesced; the +1 column breaks bank conflicts on the
// transposed read.
template <typename T>
__global__ void __launch_bounds__(256) transpose_tiles(const T *__restrict__ src, int64_t ld_src, T *__restrict__ dst,
                                                       int64_t ld_dst, int64_t rows, int64_t cols) {
    __shared__ T tile[32][33];
    pdl_enter();
    const int64_t tiles_c = (cols + 31) / 32;
    const int64_t tiles = ((rows + 31) / 32) * tiles_c;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
        const int64_t r0 = (t / tiles_c) * 32, c0 = (t % tiles_c) * 32;
        for (int i = ty; i < 32; i += 8) {
            const int64_t r = r0 + i, c = c0 + tx;
            tile[i][tx] = (r < rows && c < cols) ? src[r * ld_src + c] : T(0);
        }
        __syncthreads();
        for (int i = ty; i < 32; i += 8) {
            const int64_t c = c0 + i, r = r0 + tx;
            if (c < cols && r < rows) dst[c * ld_dst + r] = tile[tx][i];
        }
        __syncthreads();
    }
}

// 64 x 64 tiles of 4-byte elements moved with 16-byte global loads and stores
// (four per thread each way), for sources whose rows are 16-byte addressable.
// Tiles at the right and bottom edges fall back to element accesses.
__global__ void __launch_bounds__(256) transpose64_vec(const uint32_t *__restrict__ src, int64_t ld_src,
                                                       uint32_t *__restrict__ dst, int64_t ld_dst, int64_t rows,
                                                       int64_t cols) {
    __shared__ uint32_t tile[64][65];
    pdl_enter();
    const int64_t tiles_c = (cols + 63) / 64;
    const int64_t tiles = ((rows + 63) / 64) * tiles_c;
    const int q = threadIdx.x & 15;    // 16-byte group within a 64-wide row
    const int r_in = threadIdx.x >> 4; // 0..15
    for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
        const int64_t r0 = (t / tiles_c) * 64, c0 = (t % tiles_c) * 64;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = r_in + 16 * i;
            const int64_t gr = r0 + r, gc = c0 + 4 * q;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (gr < rows) {
                const uint32_t *p = src + gr * ld_src + gc;
                if (gc + 3 < cols) {
                    v = *reinterpret_cast<const uint4 *>(p);
                } else {
                    if (gc + 0 < cols) v.x = p[0];
                    if (gc + 1 < cols) v.y = p[1];
                    if (gc + 2 < cols) v.z = p[2];
                }
            }
            tile[r][4 * q + 0] = v.x;
            tile[r][4 * q + 1] = v.y;
            tile[r][4 * q + 2] = v.z;
            tile[r][4 * q + 3] = v.w;
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int c = r_in + 16 * i;              // source column = destination row
            const int64_t drow = c0 + c, dcol = r0 + 4 * q;
            if (drow < cols) {
                const uint4 v = make_uint4(tile[4 * q + 0][c], tile[4 * q + 1][c], tile[4 * q + 2][c], tile[4 * q + 3][c]);
                uint32_t *p = dst + drow * ld_dst + dcol;
                if (dcol + 3 < rows) {
                    *reinterpret_cast<uint4 *>(p) = v;
                } else {
                    if (dcol + 0 < rows) p[0] = v.x;
                    if (dcol + 1 < rows) p[1] = v.y;
                    if (dcol + 2 < rows) p[2] = v.z;
                }
            }
        }
        __syncthreads();
    }
}

// Split reduction: each thread owns four consecutive columns of one row of one
// split tile and adds that tile's slabs in split order, so the result does not
// depend on scheduling.  Slabs are dense tiles (16-byte aligned rows); C gets
// vector stores when its pitch and base allow them.
template <bool VEC>
__global__ void __launch_bounds__(256) split_reduce(const float *__restrict__ W, int tail_tiles, int splits,
                                                    int tile_rows, int tile_cols, int full_tiles, int tiles_m,
                                                    int tiles_n, int group_m, void *__restrict__ Cv, int64_t ldc,
                                                    int64_t M, int64_t N, const EpiParams epi) {
    // Launched as a programmatic dependent of the GEMM: wait until the GEMM's
    // slab writes are complete and visible.
    pdl_enter();
    const int64_t quads_per_row = tile_cols / 4;
    const int64_t per_tile = (int64_t)tile_rows * quads_per_row;
    const int64_t total = (int64_t)tail_tiles * per_tile;
    const int64_t slab = (int64_t)tile_rows * tile_cols;
    for (int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; x < total; x += (int64_t)gridDim.x * blockDim.x) {
        const int i = (int)(x / per_tile);
        const int64_t rem = x - (int64_t)i * per_tile;
        const int r = (int)(rem / quads_per_row);
        const int c = (int)(rem - (int64_t)r * quads_per_row) * 4;
        int tm, tn;
        tile_coords(full_tiles + i, tiles_m, tiles_n, group_m, tm, tn);
        const int64_t m = (int64_t)tm * tile_rows + r, n = (int64_t)tn * tile_cols + c;
        if (m >= M || n >= N) continue;
        const float *w = W + (int64_t)i * slab + (int64_t)r * tile_cols + c;
        const int64_t stride = (int64_t)tail_tiles * slab;   // from one split's slab to the next
        auto ld = [&](int sp) { return __ldcs(reinterpret_cast<const float4 *>(w + sp * stride)); };
        auto add = [](float4 &a, const float4 &v) {
            a.x += v.x;
            a.y += v.y;
            a.z += v.z;
            a.w += v.w;
        };
        // Four slabs' loads in flight at a time; the sums still run in split order.
        float4 acc = ld(0);
        int sp = 1;
        for (; sp + 3 < splits; sp += 4) {
            const float4 v1 = ld(sp), v2 = ld(sp + 1), v3 = ld(sp + 2), v4 = ld(sp + 3);
            add(acc, v1);
            add(acc, v2);
            add(acc, v3);
            add(acc, v4);
        }
        for (; sp < splits; ++sp) add(acc, ld(sp));
        if (epi.active) {
            const float v[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (n + q < N) epi_write(epi, Cv, m * ldc + n + q, v[q], epi_bias(epi, n + q, N));
            continue;
        }
        float *out = static_cast<float *>(Cv) + m * ldc + n;
        if (VEC && n + 3 < N) {
            *reinterpret_cast<float4 *>(out) = acc;
        } else {
            out[0] = acc.x;
            if (n + 1 < N) out[1] = acc.y;
            if (n + 2 < N) out[2] = acc.z;
            if (n + 3 < N) out[3] = acc.w;
        }
    }
}

__global__ void __launch_bounds__(256) epilogue_fill(void *__restrict__ C, int64_t ldc, int64_t M, int64_t N,
                                                     const EpiParams epi) {
    pdl_enter();
    const int64_t total = M * N;
    for (int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; x < total; x += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = x / N, c = x - r * N;
        epi_write(epi, C, r * ldc + c, 0.f, epi_bias(epi, c, N));
    }
}

int sm_count(cudaError_t *err) {
    int dev = 0, sms = 0;
    *err = cudaGetDevice(&dev);
    if (*err == cudaSuccess) *err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms;
}

}  // namespace

cudaError_t transpose_launch(const void *src, int64_t ld_src, void *dst, int64_t ld_dst, int64_t rows, int64_t cols,
                             int elem_bytes, cudaStream_t stream) {
    cudaError_t e;
    const int sms = sm_count(&e);
    if (e != cudaSuccess) return e;
    const bool vec = elem_bytes == 4 && (uintptr_t)src % 16 == 0 && ld_src % 4 == 0 && (uintptr_t)dst % 16 == 0 &&
                     ld_dst % 4 == 0;
    if (vec) {
        const int64_t tiles64 = ((rows + 63) / 64) * ((cols + 63) / 64);
        const int blocks64 = (int)(tiles64 < (int64_t)sms * 8 ? (tiles64 > 0 ? tiles64 : 1) : (int64_t)sms * 8);
        return launch_pdl(transpose64_vec, dim3(blocks64), dim3(256), 0, stream, static_cast<const uint32_t *>(src),
                          ld_src, static_cast<uint32_t *>(dst), ld_dst, rows, cols);
    }
    const int64_t tiles = ((rows + 31) / 32) * ((cols + 31) / 32);
    const dim3 grid((unsigned)(tiles < (int64_t)sms * 8 ? (tiles > 0 ? tiles : 1) : (int64_t)sms * 8));
    if (elem_bytes == 1)
        return launch_pdl(transpose_tiles<uint8_t>, grid, dim3(256), 0, stream, static_cast<const uint8_t *>(src),
                          ld_src, static_cast<uint8_t *>(dst), ld_dst, rows, cols);
    if (elem_bytes == 2)
        return launch_pdl(transpose_tiles<uint16_t>, grid, dim3(256), 0, stream, static_cast<const uint16_t *>(src),
                          ld_src, static_cast<uint16_t *>(dst), ld_dst, rows, cols);
    if (elem_bytes == 4)
        return launch_pdl(transpose_tiles<uint32_t>, grid, dim3(256), 0, stream, static_cast<const uint32_t *>(src),
                          ld_src, static_cast<uint32_t *>(dst), ld_dst, rows, cols);
    return cudaErrorInvalidValue;
}

cudaError_t split_reduce_launch(const float *W, int tail_tiles, int splits, int tile_rows, int tile_cols,
                                int full_tiles, int tiles_m, int tiles_n, int group_m, void *C, int64_t ldc,
                                int64_t M, int64_t N, const EpiParams &epi, cudaStream_t stream) {
    cudaError_t e;
    const int sms = sm_count(&e);
    if (e != cudaSuccess) return e;
    if (tile_cols % 4 != 0 || (uintptr_t)W % 16 != 0) return cudaErrorInvalidValue;
    const int64_t quads = (int64_t)tail_tiles * tile_rows * (tile_cols / 4);
    const int64_t want = (quads + 255) / 256;
    const int blocks = (int)(want < (int64_t)sms * 8 ? (want > 0 ? want : 1) : (int64_t)sms * 8);
    const bool vec = (ldc % 4 == 0) && ((uintptr_t)C % 16 == 0);
    // The launch may overlap the GEMM's tail (which releases it at its
    // teardown); the kernel's wait keeps the reads after the GEMM's writes.
    return launch_pdl(vec ? split_reduce<true> : split_reduce<false>, dim3((unsigned)blocks), dim3(256), 0, stream, W,
                      tail_tiles, splits, tile_rows, tile_cols, full_tiles, tiles_m, tiles_n, group_m, C, ldc, M, N,
                      epi);
}

cudaError_t epilogue_fill_launch(void *C, int64_t ldc, int64_t M, int64_t N, const EpiParams &epi,
                                 cudaStream_t stream) {
    cudaError_t e;
    const int sms = sm_count(&e);
    if (e != cudaSuccess) return e;
    const int64_t want = (M * N + 255) / 256;
    const int blocks = (int)(want < (int64_t)sms * 8 ? (want > 0 ? want : 1) : (int64_t)sms * 8);
    return launch_pdl(epilogue_fill, dim3(blocks), dim3(256), 0, stream, C, ldc, M, N, epi);
}

cudaError_t pack_rows_launch(const void *src, int64_t ld_src, void *dst, int64_t ld_dst, int64_t rows, int64_t cols,
                             int elem_bytes, uint64_t src_lo, uint64_t src_hi, cudaStream_t stream) {
    cudaError_t e;
    const int sms = sm_count(&e);
    if (e != cudaSuccess) return e;
    const int64_t want = (rows + 7) / 8;   // 8 warps per block, one row per warp per pass
    const dim3 grid((unsigned)(want < (int64_t)sms * 8 ? (want > 0 ? want : 1) : (int64_t)sms * 8));
    // The vector form needs a 16-byte aligned destination with 16-byte rows.
    if ((uintptr_t)dst % 16 == 0 && (ld_dst * elem_bytes) % 16 == 0 && src_hi > src_lo) {
        const int64_t chunks = rows * (ld_dst * elem_bytes / 16);
        const int64_t vwant = (chunks + 255) / 256;
        const dim3 vgrid((unsigned)(vwant < (int64_t)sms * 16 ? (vwant > 0 ? vwant : 1) : (int64_t)sms * 16));
        const uint8_t *s = static_cast<const uint8_t *>(src);
        uint8_t *d = static_cast<uint8_t *>(dst);
        const uintptr_t lo = (uintptr_t)src_lo, hi = (uintptr_t)src_hi;
        const int64_t eb = elem_bytes;
        if (elem_bytes == 1)
            return launch_pdl(pack_rows_vec<1>, vgrid, dim3(256), 0, stream, s, ld_src, d, ld_dst, rows, cols, lo, hi);
        if (elem_bytes == 2)
            return launch_pdl(pack_rows_vec<2>, vgrid, dim3(256), 0, stream, s, ld_src * eb, d, ld_dst * eb, rows,
                              cols * eb, lo, hi);
        if (elem_bytes == 4)
            return launch_pdl(pack_rows_vec<4>, vgrid, dim3(256), 0, stream, s, ld_src * eb, d, ld_dst * eb, rows,
                              cols * eb, lo, hi);
        return cudaErrorInvalidValue;
    }
    if (elem_bytes == 1)
        return launch_pdl(pack_rows<uint8_t>, grid, dim3(256), 0, stream, static_cast<const uint8_t *>(src), ld_src,
                          static_cast<uint8_t *>(dst), ld_dst, rows, cols);
    if (elem_bytes == 2)
        return launch_pdl(pack_rows<uint16_t>, grid, dim3(256), 0, stream, static_cast<const uint16_t *>(src), ld_src,
                          static_cast<uint16_t *>(dst), ld_dst, rows, cols);
    if (elem_bytes == 4)
        return launch_pdl(pack_rows<uint32_t>, grid, dim3(256), 0, stream, static_cast<const uint32_t *>(src), ld_src,
                          static_cast<uint32_t *>(dst), ld_dst, rows, cols);
    return cudaErrorInvalidValue;
}

}  // namespace tcgemm
