// Operand pack: copy a row-major matrix into a buffer whose row pitch the TMA
// engine can address.  "Learn CuTeDSL" section 3.4: every stride of a TMA
// tensor other than the contiguous one must be a multiple of 16 bytes (and the
// base 16-byte aligned); a K x N BF16 matrix with N = 4095 has an 8190-byte
// pitch and cannot be described.  The copy rounds the pitch up to a multiple of
// 16 bytes and zero-fills the extra columns.
//
// HBM-bound: one read and one write of the operand.  The grid is a multiple of
// the SM count; each warp walks whole rows so both sides stay coalesced even
// though the source rows start at arbitrary 2- or 4-byte offsets.
#include "internal.h"

namespace tcgemm {
namespace {

template <typename T>
__global__ void __launch_bounds__(256) pack_rows(const T *__restrict__ src, int64_t ld_src, T *__restrict__ dst,
                                                 int64_t ld_dst, int64_t rows, int64_t cols) {
    const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x / 32);
    const int64_t warp = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    for (int64_t r = warp; r < rows; r += warps_total) {
        const T *s = src + r * ld_src;
        T *d = dst + r * ld_dst;
        for (int64_t c = lane; c < ld_dst; c += 32) d[c] = c < cols ? s[c] : T(0);
    }
}

}  // namespace

cudaError_t pack_rows_launch(const void *src, int64_t ld_src, void *dst, int64_t ld_dst, int64_t rows, int64_t cols,
                             int elem_bytes, cudaStream_t stream) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int64_t want = (rows + 7) / 8;   // 8 warps per block, one row per warp per pass
    const int blocks = (int)(want < (int64_t)sms * 8 ? (want > 0 ? want : 1) : (int64_t)sms * 8);
    if (elem_bytes == 2)
        pack_rows<uint16_t><<<blocks, 256, 0, stream>>>(static_cast<const uint16_t *>(src), ld_src,
                                                        static_cast<uint16_t *>(dst), ld_dst, rows, cols);
    else if (elem_bytes == 4)
        pack_rows<uint32_t><<<blocks, 256, 0, stream>>>(static_cast<const uint32_t *>(src), ld_src,
                                                        static_cast<uint32_t *>(dst), ld_dst, rows, cols);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

}  // namespace tcgemm
