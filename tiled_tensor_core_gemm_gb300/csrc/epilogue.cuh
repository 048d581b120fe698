// The fused epilogue applied where C is written ("Shared memory and tensor
// cores" section 13.10: bias, activation, residual add or a type cast applied
// to the accumulator before the store):
//   y = act(alpha * acc + beta * C_old + bias[col]),  stored as the output type.
// Every kernel that writes C (the tensor-core epilogue warps, the split-K
// reduction, the SIMT kernel, the K = 0 fill) goes through epi_write, so the
// arithmetic is the same on every path: FP32 throughout, one
// round-to-nearest-even conversion at the store.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "internal.h"

namespace tcgemm {

__device__ __forceinline__ float epi_load_old(const void *C, int64_t idx, int out) {
    if (out == GEMM_OUT_BF16) return __bfloat162float(static_cast<const __nv_bfloat16 *>(C)[idx]);
    if (out == GEMM_OUT_F16) return __half2float(static_cast<const __half *>(C)[idx]);
    return static_cast<const float *>(C)[idx];
}

// bias[col], or 0 without a bias (or outside [0, N) -- such columns are never stored).
__device__ __forceinline__ float epi_bias(const EpiParams &e, int64_t col, int64_t N) {
    return (e.active && e.bias && col < N) ? __ldg(e.bias + col) : 0.f;
}

// Writes acc (the full sum over K) for C[idx] through the epilogue; bias is
// epi_bias() of the element's column.
__device__ __forceinline__ void epi_write(const EpiParams &e, void *C, int64_t idx, float acc, float bias) {
    if (!e.active) {
        static_cast<float *>(C)[idx] = acc;
        return;
    }
    float y = e.alpha * acc;
    if (e.beta != 0.f) y = fmaf(e.beta, epi_load_old(C, idx, e.out), y);
    y += bias;
    if (e.act == GEMM_ACT_RELU)
        y = fmaxf(y, 0.f);
    else if (e.act == GEMM_ACT_GELU)
        y = 0.5f * y * (1.f + erff(y * 0.70710678118654752f));   // x * Phi(x), Phi through erf
    if (e.out == GEMM_OUT_BF16)
        static_cast<__nv_bfloat16 *>(C)[idx] = __float2bfloat16_rn(y);
    else if (e.out == GEMM_OUT_F16)
        static_cast<__half *>(C)[idx] = __float2half_rn(y);
    else
        static_cast<float *>(C)[idx] = y;
}

}  // namespace tcgemm
