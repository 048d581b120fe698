// Grouped GEMM: a batch of independent GEMMs of different shapes in one
// persistent tensor-core launch ("Learn CuTeDSL" section 8.4, grouped tile
// scheduler).  The host checks every group as gemm_run_ex does, picks one tile
// shape from the groups' total tile count, packs the operands TMA cannot
// address, encodes each group's tensor maps into a descriptor, copies the
// descriptors to device memory and launches the kernel, which flattens the
// groups' tiles into one list of work units (see unit_info in tc_gemm.cu).
#include <algorithm>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "internal.h"

namespace tcgemm {
namespace {

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t round_up(int64_t x, int64_t m) { return cdiv(x, m) * m; }

constexpr int64_t kMaxGroups = 1 << 20;

// ------------------------------------------------ pinned descriptor staging ---
// The descriptors reach device memory by cudaMemcpyAsync from pinned host
// memory, so the copy is asynchronous and the call never waits on the stream.
// Each device has a ring of slots; a slot is reused once the event recorded
// after its copy has completed.  Requests larger than a slot (or a failed
// pinned allocation) copy from ordinary host memory instead.
constexpr int kSlots = 8;
constexpr size_t kSlotBytes = 256 * 1024;

struct StageRing {
    std::mutex mu;
    uint8_t *host = nullptr;
    cudaEvent_t ev[kSlots] = {};
    bool recorded[kSlots] = {};
    bool busy[kSlots] = {};
    int next = 0;
    bool broken = false;
};
StageRing g_ring[64];

uint8_t *stage_acquire(int dev, size_t bytes, int *slot) {
    if (dev < 0 || dev >= 64 || bytes > kSlotBytes) return nullptr;
    StageRing &r = g_ring[dev];
    std::lock_guard<std::mutex> lk(r.mu);
    if (r.broken) return nullptr;
    if (!r.host) {
        void *h = nullptr;
        if (cudaHostAlloc(&h, kSlots * kSlotBytes, cudaHostAllocPortable) != cudaSuccess) {
            cudaGetLastError();
            r.broken = true;
            return nullptr;
        }
        for (int i = 0; i < kSlots; ++i) {
            if (cudaEventCreateWithFlags(&r.ev[i], cudaEventDisableTiming) != cudaSuccess) {
                cudaGetLastError();
                r.broken = true;
                return nullptr;
            }
        }
        r.host = static_cast<uint8_t *>(h);
    }
    for (int k = 0; k < kSlots; ++k) {
        const int s = (r.next + k) % kSlots;
        if (r.busy[s]) continue;                       // another thread is filling it
        if (r.recorded[s] && cudaEventSynchronize(r.ev[s]) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        r.busy[s] = true;
        r.next = (s + 1) % kSlots;
        *slot = s;
        return r.host + (size_t)s * kSlotBytes;
    }
    return nullptr;
}

void stage_release(int dev, int slot, cudaStream_t stream) {
    StageRing &r = g_ring[dev];
    std::lock_guard<std::mutex> lk(r.mu);
    r.recorded[slot] = cudaEventRecord(r.ev[slot], stream) == cudaSuccess;
    if (!r.recorded[slot]) cudaGetLastError();
    r.busy[slot] = false;
}

// ------------------------------------------------------------ arguments ---
struct Span {
    uint64_t lo, hi;
};

// Whether [lo, hi) meets any of the (sorted, disjoint) C spans.
bool any_overlap(const std::vector<Span> &sorted_c, uint64_t lo, uint64_t hi) {
    // the first C span whose end is past lo
    auto it = std::upper_bound(sorted_c.begin(), sorted_c.end(), lo,
                               [](uint64_t v, const Span &s) { return v < s.hi; });
    return it != sorted_c.end() && it->lo < hi;
}

struct Work {
    int64_t g;                 // index in the caller's array
    const void *A, *B;         // as the kernel reads them (maybe packed copies)
    int64_t lda, ldb;
    uint64_t a_off, b_off;     // workspace offsets of packed copies (0: none)
    bool pack_a, pack_b, trans_b;
    uint64_t a_lo, a_hi, b_lo, b_hi;
};

int run_grouped(int dtype, int64_t G, const gemm_group_t *groups, const EpiParams &epi_in, cudaStream_t stream) {
    if (G < 0 || G > kMaxGroups) return api_error(GEMM_ERR_INVALID_ARG, "group_count must be in [0, 2^20]");
    if (G == 0) return GEMM_OK;
    if (!groups) return api_error(GEMM_ERR_INVALID_ARG, "groups is NULL");
    if (epi_in.bias) return api_error(GEMM_ERR_INVALID_ARG, "the shared epilogue's bias must be NULL (each group has its own)");

    // ---- every group's arguments, before any CUDA call
    const int ob = (epi_in.active && epi_in.out != GEMM_OUT_F32) ? 2 : 4;
    std::vector<Span> c_spans;
    c_spans.reserve((size_t)G);
    bool any_bias = false;
    for (int64_t g = 0; g < G; ++g) {
        const gemm_group_t &q = groups[g];
        int rc = api_validate(q.M, q.N, q.K, dtype, q.A, q.lda, q.B, q.ldb, q.C, q.ldc);
        if (rc) return rc;
        if (q.M == 0 || q.N == 0) continue;
        const int eb = api_elem_bytes(dtype);
        const uint64_t c0 = (uint64_t)(uintptr_t)q.C, c1 = c0 + (uint64_t)((q.M - 1) * q.ldc + q.N) * ob;
        if (c0 % ob) return api_error(GEMM_ERR_INVALID_ARG, "a group's C is not aligned to its element");
        if (q.K > 0) {
            const uint64_t a0 = (uint64_t)(uintptr_t)q.A, b0 = (uint64_t)(uintptr_t)q.B;
            if (a0 % eb || b0 % eb) return api_error(GEMM_ERR_INVALID_ARG, "a group's A or B is not aligned to its element");
        }
        if (q.bias && (uint64_t)(uintptr_t)q.bias % 4)
            return api_error(GEMM_ERR_INVALID_ARG, "a group's bias is not 4-byte aligned");
        any_bias = any_bias || q.bias;
        c_spans.push_back({c0, c1});
    }
    // No group's C may overlap any group's A, B, C or bias (its own C too is
    // checked against its own A, B and bias).
    std::sort(c_spans.begin(), c_spans.end(), [](const Span &x, const Span &y) { return x.lo < y.lo; });
    for (size_t i = 1; i < c_spans.size(); ++i)
        if (c_spans[i].lo < c_spans[i - 1].hi) return api_error(GEMM_ERR_INVALID_ARG, "two groups' C overlap");
    for (int64_t g = 0; g < G; ++g) {
        const gemm_group_t &q = groups[g];
        if (q.M == 0 || q.N == 0) continue;
        const int eb = api_elem_bytes(dtype);
        if (q.K > 0) {
            const uint64_t a0 = (uint64_t)(uintptr_t)q.A, a1 = a0 + (uint64_t)((q.M - 1) * q.lda + q.K) * eb;
            const uint64_t b0 = (uint64_t)(uintptr_t)q.B, b1 = b0 + (uint64_t)((q.K - 1) * q.ldb + q.N) * eb;
            if (any_overlap(c_spans, a0, a1) || any_overlap(c_spans, b0, b1))
                return api_error(GEMM_ERR_INVALID_ARG, "a group's C overlaps a group's A or B");
        }
        if (q.bias) {
            const uint64_t s0 = (uint64_t)(uintptr_t)q.bias, s1 = s0 + (uint64_t)q.N * 4;
            if (any_overlap(c_spans, s0, s1)) return api_error(GEMM_ERR_INVALID_ARG, "a group's bias overlaps a C");
        }
    }

    if (c_spans.empty()) return GEMM_OK;   // every group has M == 0 or N == 0

    // ---- FP32: the SIMT kernel, one launch per group
    if (dtype == GEMM_FP32) {
        for (int64_t g = 0; g < G; ++g) {
            const gemm_group_t &q = groups[g];
            if (q.M == 0 || q.N == 0) continue;
            gemm_epilogue_t e{epi_in.alpha, epi_in.beta, q.bias, epi_in.act, epi_in.out};
            const int rc = gemm_run_ex(q.M, q.N, q.K, dtype, q.A, q.lda, q.B, q.ldb, q.C, q.ldc, &e,
                                       reinterpret_cast<struct CUstream_st *>(stream));
            if (rc) return rc;
        }
        return GEMM_OK;
    }

    // ---- device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return api_error(GEMM_ERR_CUDA, cudaGetErrorString(e));
    int sms = 0, ccmaj = 0, ccmin = 0, clusters = 0;
    int rc = api_device_info(dev, &sms, &ccmaj, &ccmin, &clusters);
    if (rc) return rc;
    if (!(ccmaj == 10 && ccmin == 3))
        return api_error(GEMM_ERR_UNSUPPORTED, "this library is built for sm_103a only");
    const int eb = api_elem_bytes(dtype);
    std::vector<Work> work;
    std::vector<int64_t> k_zero;
    for (int64_t g = 0; g < G; ++g) {
        const gemm_group_t &q = groups[g];
        if (q.M == 0 || q.N == 0) continue;
        if ((rc = api_check_device_span("C", q.C, (uint64_t)((q.M - 1) * q.ldc + q.N) * ob, dev))) return rc;
        if (q.bias && (rc = api_check_device_span("bias", q.bias, (uint64_t)q.N * 4, dev))) return rc;
        if (q.K == 0) {
            k_zero.push_back(g);
            continue;
        }
        Work w{};
        w.g = g;
        if ((rc = api_check_device_span_range("A", q.A, (uint64_t)((q.M - 1) * q.lda + q.K) * eb, dev, &w.a_lo, &w.a_hi)))
            return rc;
        if ((rc = api_check_device_span_range("B", q.B, (uint64_t)((q.K - 1) * q.ldb + q.N) * eb, dev, &w.b_lo, &w.b_hi)))
            return rc;
        work.push_back(w);
    }

    EpiParams epi = epi_in;
    if (any_bias) epi.active = 1;      // NULL-bias groups then add 0
    const Options opt = options_snapshot();
    if ((rc = api_check_trace(opt, dev))) return rc;

    // ---- one plan for every group, from the total tile count
    gemm_plan_t plan;
    std::memset(&plan, 0, sizeof plan);
    int64_t t2 = 0, t1_256 = 0;
    for (const Work &w : work) {
        const gemm_group_t &q = groups[w.g];
        t2 += cdiv(q.M, 256) * cdiv(q.N, 256);
        t1_256 += cdiv(q.M, 128) * cdiv(q.N, 256);
    }
    int cg = opt.tc_cta_group, bn = opt.tc_bn;
    if (cg == 0 && bn == 0) {
        if (clusters > 0 && t2 >= clusters) {
            cg = 2;
            bn = 256;
        } else {
            cg = 1;
            bn = t1_256 >= sms ? 256 : 128;
        }
    } else if (cg == 0) {
        cg = (bn == 256 && clusters > 0 && t2 >= clusters) ? 2 : 1;
    } else if (bn == 0) {
        bn = 256;
    }
    if (cg == 2 && clusters <= 0) return api_error(GEMM_ERR_UNSUPPORTED, "2-CTA tiles need cluster support");
    int b_kmajor = opt.tc_b_major == 1 ? 1 : 0;
    const bool fp8 = dtype == GEMM_E4M3 || dtype == GEMM_E5M2;
    if (fp8 && !b_kmajor && (bn / cg) % 128 != 0) {
        if (opt.tc_b_major == 2) return api_error(GEMM_ERR_UNSUPPORTED, "FP8 B as stored needs 128 columns per CTA");
        b_kmajor = 1;
    }
    if (tc_smem_bytes(dtype, cg, bn, b_kmajor) == 0)
        return api_error(GEMM_ERR_UNSUPPORTED, "no tensor-core variant for this tile");
    plan.path = 1;
    plan.bm = 128;
    plan.bn = bn;
    plan.bk = 128 / eb;
    plan.cta_group = cg;
    plan.b_kmajor = b_kmajor;
    plan.stages = tc_stages(dtype, cg, bn, b_kmajor);
    plan.smem_bytes = tc_smem_bytes(dtype, cg, bn, b_kmajor);
    plan.group_m = opt.tc_group_m > 0 ? opt.tc_group_m : (cg == 2 ? 8 : 16);
    plan.splits = 1;
    plan.tma_store = 0;                // decided per group

    // ---- workspace: descriptors, then packed / transposed operands
    const uint64_t desc_bytes = (uint64_t)work.size() * sizeof(GroupDesc);
    uint64_t off = round_up((int64_t)desc_bytes, 256);
    int64_t total_units = 0;
    for (Work &w : work) {
        const gemm_group_t &q = groups[w.g];
        const uint64_t a = (uint64_t)(uintptr_t)q.A, b = (uint64_t)(uintptr_t)q.B;
        w.pack_a = (a % 16) || ((q.lda * eb) % 16);
        w.lda = w.pack_a ? round_up(q.K, 16 / eb) : q.lda;
        if (w.pack_a) {
            w.a_off = off;
            off = round_up((int64_t)(off + (uint64_t)q.M * w.lda * eb), 256);
        }
        w.trans_b = b_kmajor;
        w.pack_b = !b_kmajor && ((b % 16) || ((q.ldb * eb) % 16));
        if (w.trans_b) {
            w.ldb = round_up(q.K, 16 / eb);
            w.b_off = off;
            off = round_up((int64_t)(off + (uint64_t)q.N * w.ldb * eb), 256);
        } else if (w.pack_b) {
            w.ldb = round_up(q.N, 16 / eb);
            w.b_off = off;
            off = round_up((int64_t)(off + (uint64_t)q.K * w.ldb * eb), 256);
        } else {
            w.ldb = q.ldb;
        }
        total_units += cdiv(q.M, 128 * cg) * cdiv(q.N, bn);
    }
    if (total_units > 0x7fffffff) return api_error(GEMM_ERR_INVALID_ARG, "too many tiles in one grouped launch");

    void *ws = nullptr;
    if (!work.empty()) {
        e = cudaMallocAsync(&ws, (size_t)off, stream);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return api_error(GEMM_ERR_NO_MEMORY, "grouped workspace allocation failed");
        }
    }
    uint8_t *wsb = static_cast<uint8_t *>(ws);
    auto fail_free = [&](int code, const char *msg) {
        if (ws) cudaFreeAsync(ws, stream);
        return api_error(code, msg);
    };

    // ---- packs, descriptors
    std::vector<GroupDesc> hd(work.size());
    std::memset(hd.data(), 0, hd.size() * sizeof(GroupDesc));
    int64_t unit_start = 0;
    char err[256] = {0};
    for (size_t i = 0; i < work.size(); ++i) {
        Work &w = work[i];
        const gemm_group_t &q = groups[w.g];
        w.A = q.A;
        w.B = q.B;
        if (w.pack_a) {
            e = pack_rows_launch(q.A, q.lda, wsb + w.a_off, w.lda, q.M, q.K, eb, w.a_lo, w.a_hi, stream);
            if (e != cudaSuccess) return fail_free(GEMM_ERR_CUDA, "operand pack failed");
            w.A = wsb + w.a_off;
        }
        if (w.trans_b) {
            e = transpose_launch(q.B, q.ldb, wsb + w.b_off, w.ldb, q.K, q.N, eb, stream);
            if (e != cudaSuccess) return fail_free(GEMM_ERR_CUDA, "B transpose failed");
            w.B = wsb + w.b_off;
        } else if (w.pack_b) {
            e = pack_rows_launch(q.B, q.ldb, wsb + w.b_off, w.ldb, q.K, q.N, eb, w.b_lo, w.b_hi, stream);
            if (e != cudaSuccess) return fail_free(GEMM_ERR_CUDA, "operand pack failed");
            w.B = wsb + w.b_off;
        }
        GroupDesc &d = hd[i];
        const uint64_t c0 = (uint64_t)(uintptr_t)q.C;
        d.tma_store = (opt.tc_tma_store != 2 && c0 % 16 == 0 && ((uint64_t)q.ldc * ob) % 16 == 0 &&
                       ((uint64_t)q.N * ob) % 16 == 0)
                          ? 1
                          : 0;
        d.C = q.C;
        d.ldc = q.ldc;
        d.bias = q.bias;
        d.unit_start = (int32_t)unit_start;
        rc = tc_encode_group(plan, dtype, &d, w.A, w.lda, w.B, w.ldb, q.C, q.ldc, epi.active ? epi.out : GEMM_OUT_F32,
                             (int)q.M, (int)q.N, (int)q.K, err, sizeof err);
        if (rc) return fail_free(rc, err);
        unit_start += (int64_t)d.tiles_m * d.tiles_n;
    }

    if (!work.empty()) {
        int slot = -1;
        uint8_t *stage = stage_acquire(dev, (size_t)desc_bytes, &slot);
        if (stage) {
            std::memcpy(stage, hd.data(), (size_t)desc_bytes);
            e = cudaMemcpyAsync(ws, stage, (size_t)desc_bytes, cudaMemcpyHostToDevice, stream);
            stage_release(dev, slot, stream);
        } else {
            e = cudaMemcpyAsync(ws, hd.data(), (size_t)desc_bytes, cudaMemcpyHostToDevice, stream);
        }
        if (e != cudaSuccess) return fail_free(GEMM_ERR_CUDA, "descriptor copy failed");
        int64_t units = cg == 2 ? clusters : sms;
        if (opt.tc_max_ctas > 0) units = std::min<int64_t>(units, std::max(1, opt.tc_max_ctas / cg));
        units = std::min<int64_t>(units, total_units);
        plan.tiles = (int32_t)total_units;
        // Units of unequal cost (groups' K differing by 2x or more) balance better
        // when running clusters steal work: 3% on a K-skewed 16-group workload,
        // no change on equal K (measured on GB300).
        int64_t kb_min = INT64_MAX, kb_max = 0;
        for (const Work &w : work) {
            const int64_t kb = cdiv(groups[w.g].K, 128 / eb);
            kb_min = std::min(kb_min, kb);
            kb_max = std::max(kb_max, kb);
        }
        plan.sched = opt.tc_sched == 2 ? 1 : opt.tc_sched == 1 ? 0 : (kb_max >= 2 * kb_min ? 1 : 0);
        plan.grid = (int32_t)((plan.sched ? total_units : units) * cg);
        rc = tc_launch_grouped(plan, dtype, reinterpret_cast<const GroupDesc *>(ws), (int)work.size(),
                               (int)total_units, epi, (uint32_t)opt.wait_timeout_ms, stream, err, sizeof err);
        if (rc) return fail_free(rc, err);
    }

    // ---- groups with K = 0: the epilogue of an empty sum
    for (int64_t g : k_zero) {
        const gemm_group_t &q = groups[g];
        EpiParams ez = epi;
        ez.bias = q.bias;
        if (ez.active) e = epilogue_fill_launch(q.C, q.ldc, q.M, q.N, ez, stream);
        else e = cudaMemset2DAsync(q.C, (size_t)q.ldc * 4, 0, (size_t)q.N * 4, (size_t)q.M, stream);
        if (e != cudaSuccess) return fail_free(GEMM_ERR_CUDA, "empty-sum fill failed");
    }
    if (ws) {
        e = cudaFreeAsync(ws, stream);
        if (e != cudaSuccess) return api_error(GEMM_ERR_CUDA, cudaGetErrorString(e));
    }
    return GEMM_OK;
}

}  // namespace
}  // namespace tcgemm

extern "C" int gemm_run_grouped(int dtype, int64_t group_count, const gemm_group_t *groups,
                                const gemm_epilogue_t *epi, struct CUstream_st *stream) {
    using namespace tcgemm;
    api_clear_error();
    EpiParams e;
    const int rc = api_epilogue(epi, &e);
    if (rc) return rc;
    return run_grouped(dtype, group_count, groups, e, reinterpret_cast<cudaStream_t>(stream));
}
