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

// y = act(alpha * acc + beta * old + bias) in FP32 (old is ignored when beta == 0).
__device__ __forceinline__ float epi_value(const EpiParams &e, float acc, float old, float bias) {
    float y = e.alpha * acc;
    if (e.beta != 0.f) y = fmaf(e.beta, old, y);
    y += bias;
    if (e.act == GEMM_ACT_RELU)
        y = fmaxf(y, 0.f);
    else if (e.act == GEMM_ACT_GELU)
        y = 0.5f * y * (1.f + erff(y * 0.70710678118654752f));   // x * Phi(x), Phi through erf
    return y;
}

// y rounded once (to nearest even) to the output type and stored at C[idx].
__device__ __forceinline__ void epi_store(void *C, int64_t idx, int out, float y) {
    if (out == GEMM_OUT_BF16)
        static_cast<__nv_bfloat16 *>(C)[idx] = __float2bfloat16_rn(y);
    else if (out == GEMM_OUT_F16)
        static_cast<__half *>(C)[idx] = __float2half_rn(y);
    else
        static_cast<float *>(C)[idx] = y;
}

// Two values rounded to the output type (16-bit outputs) and packed low-first
// into one 32-bit word, as they sit in memory.
__device__ __forceinline__ uint32_t epi_pack2(int out, float lo, float hi) {
    if (out == GEMM_OUT_F16) {
        const __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<const uint32_t *>(&h);
    }
    const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&b);
}

// The two 16-bit values of a packed word, widened (low half first).
__device__ __forceinline__ void epi_unpack2(int out, uint32_t w, float &lo, float &hi) {
    if (out == GEMM_OUT_F16) {
        const __half2 h = *reinterpret_cast<const __half2 *>(&w);
        lo = __low2float(h);
        hi = __high2float(h);
    } else {
        const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162 *>(&w);
        lo = __low2float(b);
        hi = __high2float(b);
    }
}

// Writes acc (the full sum over K) for C[idx] through the epilogue; bias is
// epi_bias() of the element's column.
__device__ __forceinline__ void epi_write(const EpiParams &e, void *C, int64_t idx, float acc, float bias) {
    if (!e.active) {
        static_cast<float *>(C)[idx] = acc;
        return;
    }
    const float old = e.beta != 0.f ? epi_load_old(C, idx, e.out) : 0.f;
    epi_store(C, idx, e.out, epi_value(e, acc, old, bias));
}

}  // namespace tcgemm
