// Operand-layout probes for the tensor-core path (test infrastructure: built
// and run by tests/test_gpu_operand_layout.py, not part of the library).
//
// umma: one tcgen05.mma (cta_group::1, M = 128, one MMA's K) whose A is
// one-hot in the K-major 128-byte-swizzled layout (row m has a 1 at
// k = m % UMMA_K), and whose B shared-memory region holds, at every element,
// one base-64 digit of that element's own index plus 1.  Then D[m][n] =
// B(k = m % UMMA_K, n): three runs give the index of the shared-memory element
// the MMA read for each (k, n) under a given descriptor.
//
// tma: a 32 x 32 FP32 box whose values are their own global index, loaded
// with a given swizzle mode into 1024-byte-aligned shared memory and dumped.
//
// Output: one line per case, "<name> <v0> <v1> ...": for the MMA cases the
// element index read for each (row m, column n) of D, row-major (k = m %
// UMMA_K); for the TMA cases the global index held by each shared-memory word.  Every access stays inside its buffer; every wait is
// bounded.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>
#include <vector>

#define CK(x)                                                                                   \
    do {                                                                                        \
        cudaError_t e_ = (x);                                                                   \
        if (e_ != cudaSuccess) {                                                                \
            printf("CUDA error %s at %s:%d\n", cudaGetErrorString(e_), __FILE__, __LINE__);     \
            return 1;                                                                           \
        }                                                                                       \
    } while (0)

constexpr int kABytes = 16384;
constexpr int kBBytes = 81920;
constexpr int kSmem = kABytes + kBBytes + 1024;   // + alignment slack

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ uint64_t gtimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ bool try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = gtimer();
    while (!try_wait(bar, parity))
        if (gtimer() - t0 > 1000000000ull) return false;
    return true;
}

__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t swz) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)(swz & 7u) << 61;
    return d;
}

struct UParams {
    int tf32;      // 0: bf16 kind::f16, 1: tf32
    int b_mn;      // 1: B MN-major, 0: K-major
    int swz;       // B descriptor layout type
    int lbo, sbo;  // B descriptor offsets (bytes)
    int N;         // MMA N (multiple of 32, <= 128)
    int pass;      // digit index
};

__global__ void __launch_bounds__(128, 1) umma_probe(UParams p, float *out, int *err) {
    extern __shared__ uint8_t raw[];
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t tslot;
    uint8_t *base = raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
    uint8_t *A = base, *B = base + kABytes;
    const int eb = p.tf32 ? 4 : 2;
    const int UK = 32 / eb;
    const int t = threadIdx.x;
    for (int i = t; i < kABytes / 4; i += 128) reinterpret_cast<uint32_t *>(A)[i] = 0u;
    const int nel = kBBytes / eb;
    for (int e = t; e < nel; e += 128) {
        const float v = (float)(((e >> (6 * p.pass)) & 63) + 1);
        if (p.tf32) reinterpret_cast<float *>(B)[e] = v;
        else reinterpret_cast<__nv_bfloat16 *>(B)[e] = __float2bfloat16_rn(v);
    }
    __syncthreads();
    {
        const int m = t, k = m % UK, kb = k * eb;
        const int off = (m / 8) * 1024 + (m % 8) * 128 + ((((kb >> 4) ^ (m % 8)) & 7) << 4) + (kb & 15);
        if (p.tf32) *reinterpret_cast<float *>(A + off) = 1.f;
        else *reinterpret_cast<__nv_bfloat16 *>(A + off) = __float2bfloat16_rn(1.f);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (t == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bar)) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (t < 32) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 128;" ::"r"(smem_u32(&tslot)) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = tslot;
    if (t == 0) {
        const uint64_t ad = sdesc(smem_u32(A), 16, 1024, 2);
        const uint64_t bd = p.b_mn ? sdesc(smem_u32(B), (uint32_t)p.lbo, (uint32_t)p.sbo, (uint32_t)p.swz)
                                   : sdesc(smem_u32(B), 16, 1024, 2);
        const uint32_t fmt = p.tf32 ? 2u : 1u;
        const uint32_t idesc = (1u << 4) | (fmt << 7) | (fmt << 10) | ((uint32_t)p.b_mn << 16) |
                               ((uint32_t)(p.N >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
        if (p.tf32)
            asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %4, 0;\n\t"
                         "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, q;\n\t}"
                         ::"r"(tmem), "l"(ad), "l"(bd), "r"(idesc), "r"(0) : "memory");
        else
            asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %4, 0;\n\t"
                         "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, q;\n\t}"
                         ::"r"(tmem), "l"(ad), "l"(bd), "r"(idesc), "r"(0) : "memory");
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(&bar))
                     : "memory");
    }
    const bool ok = wait_bounded(smem_u32(&bar), 0);
    if (!ok && t == 0) atomicExch(err, 1);
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const int w = t >> 5, lane = t & 31;
    if (__all_sync(0xffffffffu, ok)) {
        for (int c = 0; c < p.N / 32; ++c) {
            uint32_t r[32];
            const uint32_t ta = tmem + ((uint32_t)(32 * w) << 16) + (uint32_t)(32 * c);
            asm volatile(
                "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
                "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
                "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
                : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                  "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
                  "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
                  "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                : "r"(ta));
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            for (int j = 0; j < 32; ++j) out[(32 * w + lane) * p.N + 32 * c + j] = __uint_as_float(r[j]);
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (t < 32) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 128;" ::"r"(tmem) : "memory");
}

// ----------------------------------------------------------------- TMA probe
__global__ void __launch_bounds__(128, 1) tma_probe(const __grid_constant__ CUtensorMap map, float *out, int *err) {
    extern __shared__ uint8_t raw[];
    __shared__ __align__(8) uint64_t bar;
    uint8_t *base = raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
    const int t = threadIdx.x;
    for (int i = t; i < 2048; i += 128) reinterpret_cast<float *>(base)[i] = -1.f;
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    if (t == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bar)) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(&bar)), "r"(4096) : "memory");
        asm volatile(
            "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];"
            ::"r"(smem_u32(base)), "l"(reinterpret_cast<uint64_t>(&map)), "r"(smem_u32(&bar)), "r"(0), "r"(0)
            : "memory");
    }
    __syncthreads();
    const bool ok = wait_bounded(smem_u32(&bar), 0);
    if (!ok && t == 0) atomicExch(err, 1);
    __syncthreads();
    if (ok)
        for (int i = t; i < 1024; i += 128) out[i] = reinterpret_cast<const float *>(base)[i];
}

int main() {
    int *err;
    float *out;
    CK(cudaMalloc(&err, 4));
    CK(cudaMalloc(&out, 128 * 128 * 4));
    CK(cudaFuncSetAttribute(umma_probe, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem));
    struct Cfg { const char *name; UParams p; };
    // The forms the library uses: BF16 B as stored (128-byte swizzle of 16-byte
    // units), TF32 B as stored (128-byte swizzle of 32-byte units), and K-major B.
    const Cfg cfgs[] = {
        {"umma_bf16_mn_sw128_lbo2048_sbo1024_n128", {0, 1, 2, 2048, 1024, 128, 0}},
        {"umma_bf16_k_sw128_n64", {0, 0, 2, 16, 1024, 64, 0}},
        {"umma_tf32_k_sw128_n64", {1, 0, 2, 16, 1024, 64, 0}},
        {"umma_tf32_mn_sw128a32_lbo2048_sbo1024_n64", {1, 1, 1, 2048, 1024, 64, 0}},
        {"umma_tf32_mn_sw128a32_lbo4096_sbo512_n128", {1, 1, 1, 4096, 512, 128, 0}},
    };
    std::vector<float> h(128 * 128);
    for (const auto &c : cfgs) {
        std::vector<int> idx(128 * 128, 0);
        for (int pass = 0; pass < 3; ++pass) {
            UParams p = c.p;
            p.pass = pass;
            CK(cudaMemset(err, 0, 4));
            CK(cudaMemset(out, 0, 128 * 128 * 4));
            umma_probe<<<1, 128, kSmem>>>(p, out, err);
            CK(cudaGetLastError());
            CK(cudaDeviceSynchronize());
            int herr = 0;
            CK(cudaMemcpy(&herr, err, 4, cudaMemcpyDeviceToHost));
            if (herr) {
                printf("%s wait-expired\n", c.name);
                return 2;
            }
            CK(cudaMemcpy(h.data(), out, 128 * p.N * 4, cudaMemcpyDeviceToHost));
            for (int i = 0; i < 128 * p.N; ++i) {
                const float v = h[i];
                const int d = (int)v - 1;
                if (v != (float)(int)v || d < 0 || d > 63) idx[i] = -1000000;
                else idx[i] += d << (6 * pass);
            }
        }
        // every row m reads k = m % UK: print all 128 rows
        printf("%s", c.name);
        for (int i = 0; i < 128 * c.p.N; ++i) printf(" %d", idx[i]);
        printf("\n");
    }
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    CK(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q));
    auto enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    float *g;
    CK(cudaMalloc(&g, 64 * 64 * 4));
    std::vector<float> hg(64 * 64);
    for (int r = 0; r < 64; ++r)
        for (int cc = 0; cc < 64; ++cc) hg[r * 64 + cc] = (float)(r * 64 + cc);
    CK(cudaMemcpy(g, hg.data(), 64 * 64 * 4, cudaMemcpyHostToDevice));
    CK(cudaFuncSetAttribute(tma_probe, cudaFuncAttributeMaxDynamicSharedMemorySize, 8192 + 1024));
    struct TC { const char *name; CUtensorMapSwizzle s; };
    const TC tcs[] = {{"tma_sw128", CU_TENSOR_MAP_SWIZZLE_128B}, {"tma_sw128a32", CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B}};
    for (const auto &tc : tcs) {
        CUtensorMap map;
        cuuint64_t dims[2] = {64, 64};
        cuuint64_t strides[1] = {64 * 4};
        cuuint32_t box[2] = {32, 32};
        cuuint32_t es[2] = {1, 1};
        CUresult r = enc(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, g, dims, strides, box, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, tc.s, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) {
            printf("%s encode-failed %d\n", tc.name, (int)r);
            return 3;
        }
        CK(cudaMemset(err, 0, 4));
        tma_probe<<<1, 128, 8192 + 1024>>>(map, out, err);
        CK(cudaGetLastError());
        CK(cudaDeviceSynchronize());
        int herr = 0;
        CK(cudaMemcpy(&herr, err, 4, cudaMemcpyDeviceToHost));
        if (herr) {
            printf("%s wait-expired\n", tc.name);
            return 2;
        }
        CK(cudaMemcpy(h.data(), out, 1024 * 4, cudaMemcpyDeviceToHost));
        printf("%s", tc.name);
        for (int i = 0; i < 1024; ++i) printf(" %d", (int)h[i]);
        printf("\n");
    }
    return 0;
}
