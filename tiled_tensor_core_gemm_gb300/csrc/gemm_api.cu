// C ABI of the GEMM library: argument checks, the host-side planner (path,
// tile shape, ring depth, CTA pairing, raster and grid), operand packing and
// dispatch.  See include/gemm.h for the contract of every entry point.
//
// The planner follows two rules from the pages: fill the machine ("GPU
// architecture and mapping kernels" ch. 12, exercise 12.8: prefer the largest
// tile that still gives every SM work, else shrink the tile), and run a
// persistent grid of one CTA (or CTA pair) per SM ("Learn CuTeDSL" section 8.1).
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "internal.h"

namespace tcgemm {
namespace {

thread_local char t_err[512];

int fail(int code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(t_err, sizeof t_err, fmt, ap);
    va_end(ap);
    return code;
}

std::mutex g_opt_mu;
Options g_opt;

struct DevInfo {
    bool valid = false;
    int sms = 0, cc_major = 0, cc_minor = 0, max_clusters = 0;
};
std::mutex g_dev_mu;
DevInfo g_dev[64];

int dev_info(int dev, DevInfo *out) {
    if (dev < 0 || dev >= 64) return fail(GEMM_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DevInfo &d = g_dev[dev];
    if (!d.valid) {
        cudaError_t e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (e != cudaSuccess) return fail(GEMM_ERR_CUDA, "device query: %s", cudaGetErrorString(e));
        d.max_clusters = (d.cc_major == 10 && d.cc_minor == 3) ? tc_max_active_clusters(dev) : 0;
        cudaGetLastError();
        d.valid = true;
    }
    *out = d;
    return GEMM_OK;
}

PFN_cuMemGetAddressRange_v3020 address_range_fn() {
    static PFN_cuMemGetAddressRange_v3020 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &p, 3020, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuMemGetAddressRange_v3020>(p);
    });
    return fn;
}

// The operand must be device memory of the current device, and its whole
// footprint [p, p + bytes) must lie inside one allocation.  On success,
// [*lo, *hi) is the allocation (or, if it cannot be queried, the footprint).
int check_device_span(const char *name, const void *p, uint64_t bytes, int dev, uint64_t *lo = nullptr,
                      uint64_t *hi = nullptr) {
    if (lo) *lo = (uint64_t)(uintptr_t)p;
    if (hi) *hi = (uint64_t)(uintptr_t)p + bytes;
    cudaPointerAttributes attr;
    cudaError_t e = cudaPointerGetAttributes(&attr, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(GEMM_ERR_INVALID_ARG, "%s: not a CUDA pointer (%s)", name, cudaGetErrorString(e));
    }
    if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged)
        return fail(GEMM_ERR_INVALID_ARG, "%s: not device memory (memory type %d)", name, (int)attr.type);
    if (attr.type == cudaMemoryTypeDevice && attr.device != dev)
        return fail(GEMM_ERR_INVALID_ARG, "%s: lives on device %d, current device is %d", name, attr.device, dev);
    if (auto fn = address_range_fn()) {
        CUdeviceptr base = 0;
        size_t size = 0;
        if (fn(&base, &size, (CUdeviceptr)(uintptr_t)p) == CUDA_SUCCESS) {
            const uint64_t start = (uint64_t)(uintptr_t)p;
            if (start + bytes > (uint64_t)base + size)
                return fail(GEMM_ERR_INVALID_ARG,
                            "%s: footprint of %llu bytes runs past the end of its allocation (%llu bytes left)", name,
                            (unsigned long long)bytes, (unsigned long long)((uint64_t)base + size - start));
            if (lo) *lo = (uint64_t)base;
            if (hi) *hi = (uint64_t)base + size;
        }
    }
    return GEMM_OK;
}

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }
int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

bool is_fp8(int dtype) { return dtype == GEMM_E4M3 || dtype == GEMM_E5M2; }

int elem_bytes(int dtype) { return (dtype == GEMM_BF16 || dtype == GEMM_FP16) ? 2 : is_fp8(dtype) ? 1 : 4; }

// Measured on GB300 (CUDA-event sweeps): with the paired FP32 FMAs the
// 64 x 128 tile with a K step of 16 (128 threads of 8 x 8 outputs, three
// blocks and 12 warps per SM) beats the 256-thread 128 x 128 tile (8 warps per
// SM) at 4096^3, 1024^3 and 256^3.
constexpr int kSimtDefault = 9;   // 64 x 128 x 16, 8 x 8 per thread
// SIMT split-K target: about two waves of the three resident 128-thread
// blocks per SM, K ranges of at least 32 (measured on GB300:
// 8 ranges at 1024^3 and 256^3, 2 at 2048^3, none at 4096^3).
constexpr int kSimtBlocksPerSm = 6;
constexpr int64_t kSimtMinKPerSplit = 32;
constexpr int kMinKbPerSplit = 8;   // k-blocks per K range, so each range fills the ring several times
// Split-K adds a second kernel and a workspace round trip (a few microseconds):
// only worth it from about 4 GFLOP up (measured on GB300).
constexpr int64_t kMinSplitWork = 1LL << 31;
// Column halves for the last round by default only on schedules this short.
constexpr int64_t kMaxRoundsForHalves = 4;
// Split-K shapes that stream B from HBM: at most this many rows of A (below the
// BF16 ridge point of about 280 flop per byte) against a 16-bit B of at least
// this many bytes (half of L2 and up) take 128-column tiles, twice as many
// tiles over shallower K ranges (measured on GB300: +5% to +10% at
// 64..256 x 8192 x 8192 and 128 x 4096 x 16384; B of 32 MB, or 512 rows and
// more, lose with them).
constexpr int64_t kStreamBMaxRows = 256;
constexpr int64_t kStreamBMinBytes = 64LL << 20;

}  // namespace

Options options_snapshot() {
    std::lock_guard<std::mutex> lk(g_opt_mu);
    return g_opt;
}

int make_plan(int64_t M, int64_t N, int64_t K, int dtype, uint64_t a_addr, int64_t lda, uint64_t b_addr, int64_t ldb,
              uint64_t c_addr, int64_t ldc, int num_sms, int max_clusters_2cta, const Options &opt, Plan *out) {
    gemm_plan_t &p = out->pub;
    std::memset(&p, 0, sizeof p);
    out->lda_eff = lda;
    out->ldb_eff = ldb;
    if (num_sms <= 0) num_sms = 1;
    if (dtype == GEMM_FP32) {
        int id = opt.simt_variant;
        if (id == 0) id = kSimtDefault;
        int bm = 0, bn = 0, bk = 0, smem = 0;
        if (!simt_variant_tile(id, &bm, &bn, &bk, &smem))
            return fail(GEMM_ERR_UNSUPPORTED, "no SIMT variant %d", id);
        p.path = 0;
        p.bm = bm;
        p.bn = bn;
        p.bk = bk;
        p.stages = 2;
        p.cta_group = 1;
        p.group_m = 1;
        p.tiles = (int32_t)(cdiv(M, bm) * cdiv(N, bn));
        // Too few tiles for about two waves of three blocks per SM (each
        // block's K loop is latency-bound): cut K into up to 8 ranges of at
        // least 32, summed in order by a second kernel.
        int64_t splits = opt.simt_splits > 0 ? opt.simt_splits : 1;
        if (opt.simt_splits == 0 && p.tiles < kSimtBlocksPerSm * num_sms && K >= 2 * kSimtMinKPerSplit)
            splits = std::min<int64_t>({cdiv(kSimtBlocksPerSm * num_sms, p.tiles), K / kSimtMinKPerSplit, 8});
        p.splits = (int32_t)std::max<int64_t>(1, std::min<int64_t>(splits, std::max<int64_t>(1, cdiv(K, bk))));
        p.grid = p.tiles * p.splits;
        p.vec = (lda % 4 == 0 && ldb % 4 == 0 && ldc % 4 == 0 && a_addr % 16 == 0 && b_addr % 16 == 0 &&
                 c_addr % 16 == 0);
        p.smem_bytes = smem;
        return GEMM_OK;
    }
    const int elem = elem_bytes(dtype);
    p.path = 1;
    p.bm = 128;
    p.bk = 128 / elem;
    p.pack_a = (a_addr % 16 != 0) || ((lda * elem) % 16 != 0);
    if (p.pack_a) out->lda_eff = round_up(K, 16 / elem);
    // B is read as stored (N-major) unless a K-major transposed copy is asked
    // for (or, below, an FP8 tile is too narrow for B's 128-byte chunks).
    p.b_kmajor = opt.tc_b_major == 1 ? 1 : 0;
    if (p.b_kmajor) {
        p.pack_b = 0;
        out->ldb_eff = round_up(K, 16 / elem);
    } else {
        p.pack_b = (b_addr % 16 != 0) || ((ldb * elem) % 16 != 0);
        if (p.pack_b) out->ldb_eff = round_up(N, 16 / elem);
    }
    // TMA stores need a 16-byte aligned base and pitch, and a row length of
    // whole 16-byte chunks: at a ragged right edge the store writes the whole
    // 16-byte chunk holding column N - 1 (measured on GB300), which would reach
    // into the ldc padding.
    const bool c_tma_ok = (c_addr % 16 == 0) && ((ldc * 4) % 16 == 0) && ((N * 4) % 16 == 0);
    p.tma_store = (opt.tc_tma_store == 2) ? 0 : (c_tma_ok ? 1 : 0);

    int cg = opt.tc_cta_group, bn = opt.tc_bn;
    int splits = opt.tc_splits;
    auto tiles_of = [&](int g, int b) { return cdiv(M, 128 * g) * cdiv(N, b); };
    const int64_t num_kb = cdiv(K, 128 / elem);
    // Two K ranges of 128-column tiles, summed in cluster shared memory, when
    // they fit one round of 2-CTA clusters: no workspace, no second kernel.
    const int64_t t128 = tiles_of(1, 128);
    const bool two_dsm_fit = splits != 1 && opt.tc_split_reduce != 1 && max_clusters_2cta > 0 &&
                             2 * t128 <= std::min<int64_t>(num_sms, 2LL * max_clusters_2cta) &&
                             num_kb >= 2 * kMinKbPerSplit / (elem == 1 ? 4 : 1);
    bool two_dsm = false;   // chose them: two K ranges below, whatever the work size
    if (cg == 0 && bn == 0) {
        if (max_clusters_2cta > 0 && tiles_of(2, 256) >= max_clusters_2cta) {
            cg = 2;
            bn = 256;
        } else if (tiles_of(1, 256) >= num_sms) {
            cg = 1;
            bn = 256;
        } else if (splits != 1 && M * N * K >= kMinSplitWork &&
                   std::min<int64_t>(num_sms / tiles_of(1, 256), num_kb / kMinKbPerSplit) >= 2) {
            // Too few 128x256 tiles for the SMs, but K is long: split K instead of
            // shrinking the tile (a narrow tile re-reads A once per column tile),
            // except where B streams from HBM past a few rows of A: there the
            // re-read A is small and more, narrower tiles keep more SMs reading B.
            cg = 1;
            bn = (elem == 2 && M <= kStreamBMaxRows && K * N * elem >= kStreamBMinBytes) ? 128 : 256;
            // 128-column tiles in two K ranges summed in cluster shared memory
            // beat 256-column tiles whose ranges go through the workspace (3 or
            // more of them), or that keep fewer CTAs busy.  Measured on GB300
            // (alternating blocks, µs per call, 256-column plan -> this one):
            // BF16 1024x1024x2048 15.1 -> 11.7, 512x2048x2048 15.1 -> 11.7,
            // 768x1536x3072 16.5 -> 14.0, 256x4096x4096 17.7 -> 16.1; FP16 and
            // TF32 alike; E4M3 512x2048x2048 11.3 -> 9.5 (twice the CTAs).  Not
            // where it keeps fewer CTAs busy (256x2048x8192: 18.6 -> 24.0).
            const int64_t t256 = tiles_of(1, 256);
            const int64_t s256 = std::min<int64_t>({num_sms / t256, num_kb / kMinKbPerSplit, 16});
            if (bn == 256 && two_dsm_fit && (s256 >= 3 ? 2 * t128 >= t256 * s256 : 2 * t128 > t256 * s256)) {
                bn = 128;
                two_dsm = true;
            }
        } else if (tiles_of(1, 128) >= num_sms) {
            cg = 1;
            bn = 128;
        } else if ((dtype == GEMM_TF32 || is_fp8(dtype)) && two_dsm_fit && 2 * t128 >= tiles_of(1, 64) &&
                   K >= 1024) {
            // TF32 and 8-bit inputs, too little work for the split above: two K
            // ranges of 128-column tiles in cluster shared memory rather than
            // 64-column tiles (for 8-bit inputs those also need B's K-major
            // copy).  Measured on GB300: TF32 1024^3 12.9 -> 12.1 µs, E4M3 /
            // E5M2 1024^3 10.3 -> 8.4; 16-bit inputs lose at that size.
            cg = 1;
            bn = 128;
            two_dsm = true;
        } else {
            cg = 1;
            bn = 64;
        }
    } else if (cg == 0) {
        cg = (bn == 256 && max_clusters_2cta > 0 && tiles_of(2, 256) >= max_clusters_2cta) ? 2 : 1;
    } else if (bn == 0) {
        bn = 256;
    }
    // FP8 B read as stored comes in 128-column chunks (128 bytes): a CTA's
    // share of a narrower tile reads the K-major copy instead.
    if (is_fp8(dtype) && !p.b_kmajor && (bn / cg) % 128 != 0) {
        if (opt.tc_b_major == 2)
            return fail(GEMM_ERR_UNSUPPORTED, "FP8 B as stored needs 128 columns per CTA (BN=%d, cta_group=%d)", bn,
                        cg);
        p.b_kmajor = 1;
        p.pack_b = 0;
        out->ldb_eff = round_up(K, 16 / elem);
    }
    if (tc_smem_bytes(dtype, cg, bn, p.b_kmajor) == 0)
        return fail(GEMM_ERR_UNSUPPORTED, "no tensor-core variant with cta_group=%d, BN=%d", cg, bn);
    if (cg == 2 && max_clusters_2cta <= 0)
        return fail(GEMM_ERR_UNSUPPORTED, "2-CTA tiles need cluster support on this device");
    p.cta_group = cg;
    p.bn = bn;
    p.stages = tc_stages(dtype, cg, bn, p.b_kmajor);
    p.smem_bytes = tc_smem_bytes(dtype, cg, bn, p.b_kmajor);
    p.group_m = opt.tc_group_m > 0 ? opt.tc_group_m : (cg == 2 ? 8 : 16);
    const int64_t tiles = tiles_of(cg, bn);
    p.tiles = (int32_t)tiles;
    int64_t units = cg == 2 ? max_clusters_2cta : num_sms;
    if (opt.tc_max_ctas > 0) units = std::min<int64_t>(units, std::max(1, opt.tc_max_ctas / cg));
    auto exact_splits = [&](int64_t want) {
        // every K range non-empty: splits = ceil(num_kb / ceil(num_kb / want))
        want = std::max<int64_t>(1, std::min<int64_t>(want, num_kb));
        return (int)cdiv(num_kb, cdiv(num_kb, want));
    };
    int64_t tail = 0, half = 0;
    if (splits == 0 && two_dsm)
        splits = 2;
    else if (splits == 0 && tiles * 2 <= units && M * N * K >= kMinSplitWork)
        splits = (int)std::max<int64_t>(1, std::min<int64_t>({units / tiles, num_kb / kMinKbPerSplit, 16}));
    const int64_t rem = tiles > units ? tiles % units : 0;   // tiles of the last, partly idle round
    if (splits > 1) {
        // split K for every tile
        splits = exact_splits(splits);
        if (splits > 1) tail = tiles;
    } else if (opt.tc_tail_splits < 2 && rem > 0 && 2 * rem <= units && tc_halves_ok(dtype, cg, bn, p.b_kmajor) &&
               (opt.tc_tail_halves == 2 ||
                (opt.tc_tail_halves == 0 && elem == 2 && tiles <= kMaxRoundsForHalves * units))) {
        // The last round's tiles as column halves: twice the units, each over
        // all of K, so no partial sums to combine.  A half's main loop takes
        // as many cycles as a whole tile's (the K-block cadence, about 545
        // cycles, not the MMA, sets its pace), but its epilogue drains half
        // the accumulator, which shortens the end of the launch.  Measured on
        // GB300: +2% on 16-bit inputs with 3-4 rounds
        // (4096^3, 16384 x 1024 x 4096), neutral at 8192^3 (14 power-capped
        // rounds), -3% on TF32 against its K split.
        half = rem;
    } else if ((opt.tc_tail_splits >= 2 || (opt.tc_tail_splits == 0 && dtype == GEMM_TF32)) && rem > 0) {
        // Split only the tiles of the last, partly idle round of the persistent
        // schedule, so that round's units each get a share of K.  Measured on
        // GB300: +4% for TF32 4096^3 (its half-rate MMA
        // makes each tile long against the reduction), 1-9% slower for 16- and
        // 8-bit inputs -- whose units in a partly idle last round already run
        // faster -- so it is on by default for TF32 only.
        const int want = opt.tc_tail_splits >= 2 ? opt.tc_tail_splits : 2;
        splits = exact_splits(want);
        if (splits > 1) tail = rem;
    }
    if (tail == 0) splits = 1;
    p.splits = splits;
    p.tail_tiles = (int32_t)tail;
    p.half_tiles = (int32_t)half;
    // Split K on every tile, two ranges, single-CTA tiles, one round of
    // clusters: the ranges of a tile run on the two CTAs of a cluster and are
    // summed in cluster shared memory (no workspace round trip, no second
    // kernel).  Measured on GB300: 128 x 8192 x 8192 (B streams from HBM).
    // On request, 4 ranges in clusters of 4 CTAs.
    const bool cs_shape = tail == tiles && cg == 1 && opt.tc_sched != 2 && (int64_t)splits * tiles <= units;
    if (opt.tc_split_reduce != 1 && cs_shape && splits == 2 && max_clusters_2cta > 0 && tiles <= max_clusters_2cta)
        p.cluster_split = 2;
    else if (opt.tc_split_reduce == 2 && cs_shape && splits == 4)
        p.cluster_split = 4;
    else if (opt.tc_split_reduce == 2 && tail > 0)
        return fail(GEMM_ERR_UNSUPPORTED,
                    "split-K in cluster shared memory needs every tile split in 2 (or 4) on single-CTA tiles, "
                    "ranges x tiles <= %lld CTAs and the static schedule (tiles=%lld splits=%d cta_group=%d)",
                    (long long)units, (long long)tiles, splits, cg);
    // On request, two K ranges of a tile on the CTAs of a cluster, 128
    // columns or fewer, C stored by TMA: CTA 0 takes the longer first range
    // and owns the whole tile, CTA 1 takes the shorter second range and sends
    // its partial while CTA 0 still streams (the kernel keeps a receive
    // region for it past a shorter ring).  The workspace path, when forced,
    // cuts K at the same k-block, so both give the same partial sums.
    // Measured on GB300 (128 x 8192 x 8192): 29.0 us with ranges of equal
    // length and the lane quarters shared out, 30.4 / 32.0 / 36.1 us with
    // 53 / 56 / 75% in the first range -- a CTA's stream rate is capped, so
    // the owners alone do not keep HBM busy -- hence off by default.
    if (cs_shape && splits == 2 && max_clusters_2cta > 0 && tiles <= max_clusters_2cta && bn <= 128 &&
        p.tma_store && opt.tc_split_lead > 50) {
        const int lead = opt.tc_split_lead;
        const int64_t even = cdiv(num_kb, 2);
        const int64_t kb = std::min<int64_t>(num_kb - 1, std::max<int64_t>(even, (num_kb * lead + 50) / 100));
        if (kb >= even && kb < num_kb) p.kb_split = (int32_t)kb;
    }
    const int64_t work_units = (tiles - tail - half) + tail * splits + 2 * half;
    units = std::min<int64_t>(units, work_units);
    // Static unless asked: measured on GB300 the dynamic schedule is within
    // 1% at 8192^3 and 2% slower on 4096-class shapes.
    p.sched = opt.tc_sched == 2 ? 1 : 0;
    // dynamic schedule: one cluster per work unit, the running ones steal the rest
    p.grid = (int32_t)((p.sched ? work_units : units) * cg);
    return GEMM_OK;
}

}  // namespace tcgemm

using namespace tcgemm;

extern "C" {

int gemm_version(void) { return 10000; }

const char *gemm_last_error(void) { return t_err; }

int gemm_set_option(const char *key, int64_t v) {
    t_err[0] = 0;
    if (!key) return fail(GEMM_ERR_INVALID_ARG, "option key is NULL");
    std::lock_guard<std::mutex> lk(g_opt_mu);
    if (!std::strcmp(key, "tc_bn")) {
        if (v != 0 && v != 64 && v != 128 && v != 256) return fail(GEMM_ERR_INVALID_ARG, "tc_bn must be 0/64/128/256");
        g_opt.tc_bn = (int)v;
    } else if (!std::strcmp(key, "tc_cta_group")) {
        if (v < 0 || v > 2) return fail(GEMM_ERR_INVALID_ARG, "tc_cta_group must be 0, 1 or 2");
        g_opt.tc_cta_group = (int)v;
    } else if (!std::strcmp(key, "tc_group_m")) {
        if (v < 0 || v > 4096) return fail(GEMM_ERR_INVALID_ARG, "tc_group_m must be in [0, 4096]");
        g_opt.tc_group_m = (int)v;
    } else if (!std::strcmp(key, "tc_max_ctas")) {
        if (v < 0 || v > (1 << 20)) return fail(GEMM_ERR_INVALID_ARG, "tc_max_ctas out of range");
        g_opt.tc_max_ctas = (int)v;
    } else if (!std::strcmp(key, "tc_splits")) {
        if (v < 0 || v > 32) return fail(GEMM_ERR_INVALID_ARG, "tc_splits must be in [0, 32]");
        g_opt.tc_splits = (int)v;
    } else if (!std::strcmp(key, "tc_tail_splits")) {
        if (v < 0 || v > 16) return fail(GEMM_ERR_INVALID_ARG, "tc_tail_splits must be in [0, 16]");
        g_opt.tc_tail_splits = (int)v;
    } else if (!std::strcmp(key, "pdl")) {
        if (v < 0 || v > 1) return fail(GEMM_ERR_INVALID_ARG, "pdl must be 0 or 1");
        g_opt.pdl = (int)v;
    } else if (!std::strcmp(key, "simt_splits")) {
        if (v < 0 || v > 8) return fail(GEMM_ERR_INVALID_ARG, "simt_splits must be in [0, 8]");
        g_opt.simt_splits = (int)v;
    } else if (!std::strcmp(key, "tc_split_reduce")) {
        if (v < 0 || v > 2) return fail(GEMM_ERR_INVALID_ARG, "tc_split_reduce must be 0, 1 or 2");
        g_opt.tc_split_reduce = (int)v;
    } else if (!std::strcmp(key, "tc_split_lead")) {
        if (v != 0 && (v < 50 || v > 95)) return fail(GEMM_ERR_INVALID_ARG, "tc_split_lead must be 0 or in [50, 95]");
        g_opt.tc_split_lead = (int)v;
    } else if (!std::strcmp(key, "tc_tail_halves")) {
        if (v < 0 || v > 2) return fail(GEMM_ERR_INVALID_ARG, "tc_tail_halves must be 0, 1 or 2");
        g_opt.tc_tail_halves = (int)v;
    } else if (!std::strcmp(key, "tc_sched")) {
        if (v < 0 || v > 2) return fail(GEMM_ERR_INVALID_ARG, "tc_sched must be 0 (auto), 1 (static) or 2 (dynamic)");
        g_opt.tc_sched = (int)v;
    } else if (!std::strcmp(key, "tc_tma_store")) {
        if (v < 0 || v > 2) return fail(GEMM_ERR_INVALID_ARG, "tc_tma_store must be 0, 1 or 2");
        g_opt.tc_tma_store = (int)v;
    } else if (!std::strcmp(key, "simt_variant")) {
        int bm, bn, bk, smem;
        if (v != 0 && !simt_variant_tile((int)v, &bm, &bn, &bk, &smem))
            return fail(GEMM_ERR_INVALID_ARG, "simt_variant must be 0 or a compiled variant id");
        g_opt.simt_variant = (int)v;
    } else if (!std::strcmp(key, "tc_b_major")) {
        if (v < 0 || v > 2) return fail(GEMM_ERR_INVALID_ARG, "tc_b_major must be 0, 1 or 2");
        g_opt.tc_b_major = (int)v;
    } else if (!std::strcmp(key, "debug_stall_mma")) {
        if (v < 0 || v > 1) return fail(GEMM_ERR_INVALID_ARG, "debug_stall_mma must be 0 or 1");
        g_opt.debug_stall_mma = (int)v;
    } else if (!std::strcmp(key, "trace_addr")) {
        if (v < 0 || v % 8 != 0) return fail(GEMM_ERR_INVALID_ARG, "trace_addr must be 0 or an 8-byte aligned address");
        g_opt.trace_addr = v;
    } else if (!std::strcmp(key, "trace_records")) {
        if (v < 0 || v > (1 << 24)) return fail(GEMM_ERR_INVALID_ARG, "trace_records must be in [0, 2^24]");
        g_opt.trace_records = (int)v;
    } else if (!std::strcmp(key, "wait_timeout_ms")) {
        if (v < 1 || v > 600000) return fail(GEMM_ERR_INVALID_ARG, "wait_timeout_ms must be in [1, 600000]");
        g_opt.wait_timeout_ms = (int)v;
    } else {
        return fail(GEMM_ERR_INVALID_ARG, "unknown option '%s'", key);
    }
    return GEMM_OK;
}

int64_t gemm_get_option(const char *key) {
    if (!key) return -1;
    Options o = options_snapshot();
    if (!std::strcmp(key, "tc_bn")) return o.tc_bn;
    if (!std::strcmp(key, "tc_cta_group")) return o.tc_cta_group;
    if (!std::strcmp(key, "tc_group_m")) return o.tc_group_m;
    if (!std::strcmp(key, "tc_max_ctas")) return o.tc_max_ctas;
    if (!std::strcmp(key, "tc_tma_store")) return o.tc_tma_store;
    if (!std::strcmp(key, "tc_splits")) return o.tc_splits;
    if (!std::strcmp(key, "tc_tail_splits")) return o.tc_tail_splits;
    if (!std::strcmp(key, "tc_tail_halves")) return o.tc_tail_halves;
    if (!std::strcmp(key, "tc_split_reduce")) return o.tc_split_reduce;
    if (!std::strcmp(key, "tc_split_lead")) return o.tc_split_lead;
    if (!std::strcmp(key, "simt_splits")) return o.simt_splits;
    if (!std::strcmp(key, "pdl")) return o.pdl;
    if (!std::strcmp(key, "tc_sched")) return o.tc_sched;
    if (!std::strcmp(key, "simt_variant")) return o.simt_variant;
    if (!std::strcmp(key, "tc_b_major")) return o.tc_b_major;
    if (!std::strcmp(key, "wait_timeout_ms")) return o.wait_timeout_ms;
    if (!std::strcmp(key, "trace_addr")) return o.trace_addr;
    if (!std::strcmp(key, "trace_records")) return o.trace_records;
    if (!std::strcmp(key, "debug_stall_mma")) return o.debug_stall_mma;
    return -1;
}

static int validate(int64_t M, int64_t N, int64_t K, int dtype, const void *A, int64_t lda, const void *B,
                    int64_t ldb, const void *C, int64_t ldc) {
    if (dtype != GEMM_FP32 && dtype != GEMM_TF32 && dtype != GEMM_BF16 && dtype != GEMM_FP16 && dtype != GEMM_E4M3 &&
        dtype != GEMM_E5M2)
        return fail(GEMM_ERR_INVALID_ARG, "unknown dtype %d", dtype);
    if (M < 0 || N < 0 || K < 0) return fail(GEMM_ERR_INVALID_ARG, "negative size (M=%lld N=%lld K=%lld)",
                                              (long long)M, (long long)N, (long long)K);
    const int64_t kMax = 0x7fffffffLL;
    if (M > kMax || N > kMax || K > kMax) return fail(GEMM_ERR_INVALID_ARG, "sizes must be below 2^31");
    if (lda < (K > 0 ? K : 1) || ldb < (N > 0 ? N : 1) || ldc < (N > 0 ? N : 1))
        return fail(GEMM_ERR_INVALID_ARG, "leading dimension too small (lda=%lld ldb=%lld ldc=%lld)", (long long)lda,
                    (long long)ldb, (long long)ldc);
    const int64_t kLdMax = 1LL << 36;
    if (lda > kLdMax || ldb > kLdMax || ldc > kLdMax)
        return fail(GEMM_ERR_INVALID_ARG, "leading dimension above 2^36 elements");
    if (M > 0 && N > 0) {
        if (!C) return fail(GEMM_ERR_INVALID_ARG, "C is NULL");
        if (K > 0 && (!A || !B)) return fail(GEMM_ERR_INVALID_ARG, "A or B is NULL");
    }
    return GEMM_OK;
}

static bool overlaps(uint64_t a0, uint64_t a1, uint64_t b0, uint64_t b1) { return a0 < b1 && b0 < a1; }

int gemm_plan(int64_t M, int64_t N, int64_t K, int dtype, uint64_t a_addr, int64_t lda, uint64_t b_addr, int64_t ldb,
              uint64_t c_addr, int64_t ldc, int32_t num_sms, gemm_plan_t *out) {
    t_err[0] = 0;
    if (!out) return fail(GEMM_ERR_INVALID_ARG, "out is NULL");
    int rc = validate(M, N, K, dtype, (const void *)1, lda, (const void *)1, ldb, (const void *)1, ldc);
    if (rc) return rc;
    int sms = num_sms, clusters = num_sms / 2;
    if (num_sms <= 0) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return fail(GEMM_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
        DevInfo d;
        if ((rc = dev_info(dev, &d))) return rc;
        sms = d.sms;
        clusters = d.max_clusters;
    }
    Plan plan;
    rc = make_plan(M, N, K, dtype, a_addr, lda, b_addr, ldb, c_addr, ldc, sms, clusters, options_snapshot(), &plan);
    if (rc == GEMM_OK) *out = plan.pub;
    return rc;
}

}  // extern "C"

namespace tcgemm {
namespace {

// One GEMM call: checks, plan, packs, kernels.  C's element type is epi.out
// when the epilogue is active, else FP32.
int run(int64_t M, int64_t N, int64_t K, int dtype, const void *A, int64_t lda, const void *B, int64_t ldb, void *C,
        int64_t ldc, const EpiParams &epi, cudaStream_t stream) {
    int rc = validate(M, N, K, dtype, A, lda, B, ldb, C, ldc);
    if (rc) return rc;
    if (M == 0 || N == 0) return GEMM_OK;

    const int eb = elem_bytes(dtype);
    const int ob = (epi.active && epi.out != GEMM_OUT_F32) ? 2 : 4;
    const uint64_t c0 = (uint64_t)(uintptr_t)C, c1 = c0 + (uint64_t)((M - 1) * ldc + N) * ob;
    if (c0 % ob != 0) return fail(GEMM_ERR_INVALID_ARG, "C is not aligned to its %d-byte element", ob);
    if (K > 0) {
        const uint64_t a0 = (uint64_t)(uintptr_t)A, a1 = a0 + (uint64_t)((M - 1) * lda + K) * eb;
        const uint64_t b0 = (uint64_t)(uintptr_t)B, b1 = b0 + (uint64_t)((K - 1) * ldb + N) * eb;
        if (a0 % eb != 0 || b0 % eb != 0)
            return fail(GEMM_ERR_INVALID_ARG, "A or B is not aligned to its %d-byte element", eb);
        if (overlaps(a0, a1, c0, c1) || overlaps(b0, b1, c0, c1))
            return fail(GEMM_ERR_INVALID_ARG, "C overlaps A or B");
    }
    const bool has_bias = epi.active && epi.bias;
    if (has_bias) {
        const uint64_t s0 = (uint64_t)(uintptr_t)epi.bias, s1 = s0 + (uint64_t)N * 4;
        if (s0 % 4 != 0) return fail(GEMM_ERR_INVALID_ARG, "bias is not 4-byte aligned");
        if (overlaps(s0, s1, c0, c1)) return fail(GEMM_ERR_INVALID_ARG, "bias overlaps C");
    }

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(GEMM_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    DevInfo d;
    if ((rc = dev_info(dev, &d))) return rc;
    if (!(d.cc_major == 10 && d.cc_minor == 3))
        return fail(GEMM_ERR_UNSUPPORTED, "this library is built for sm_103a only (device is sm_%d%d)", d.cc_major,
                    d.cc_minor);
    if ((rc = check_device_span("C", C, c1 - c0, dev))) return rc;
    if (has_bias && (rc = check_device_span("bias", epi.bias, (uint64_t)N * 4, dev))) return rc;
    if (K == 0) {
        if (epi.active) {
            e = epilogue_fill_launch(C, ldc, M, N, epi, stream);
            return e == cudaSuccess ? GEMM_OK : fail(GEMM_ERR_CUDA, "epilogue fill: %s", cudaGetErrorString(e));
        }
        e = cudaMemset2DAsync(C, (size_t)ldc * 4, 0, (size_t)N * 4, (size_t)M, stream);
        return e == cudaSuccess ? GEMM_OK : fail(GEMM_ERR_CUDA, "cudaMemset2DAsync: %s", cudaGetErrorString(e));
    }
    uint64_t a_lo = 0, a_hi = 0, b_lo = 0, b_hi = 0;
    if ((rc = check_device_span("A", A, (uint64_t)((M - 1) * lda + K) * eb, dev, &a_lo, &a_hi))) return rc;
    if ((rc = check_device_span("B", B, (uint64_t)((K - 1) * ldb + N) * eb, dev, &b_lo, &b_hi))) return rc;

    const Options opt = options_snapshot();
    if ((rc = api_check_trace(opt, dev))) return rc;
    Plan plan;
    rc = make_plan(M, N, K, dtype, (uint64_t)(uintptr_t)A, lda, (uint64_t)(uintptr_t)B, ldb, c0, ldc, d.sms,
                   d.max_clusters, opt, &plan);
    if (rc) return rc;
    // With the fused epilogue, C's element may be 2 bytes: the TMA store rules
    // of make_plan (aligned base, pitch and row length) in that element size.
    if (epi.active)
        plan.pub.tma_store = (opt.tc_tma_store != 2 && c0 % 16 == 0 && ((uint64_t)ldc * ob) % 16 == 0 &&
                              ((uint64_t)N * ob) % 16 == 0)
                                 ? 1
                                 : 0;
    const gemm_plan_t &p = plan.pub;

    if (p.path == 0) {
        // K ranges: their partial sums live in a stream-ordered workspace.
        void *sw = nullptr;
        if (p.splits > 1) {
            const size_t bytes = (size_t)p.splits * (size_t)M * (size_t)N * 4;
            e = cudaMallocAsync(&sw, bytes, stream);
            if (e != cudaSuccess) {
                cudaGetLastError();
                return fail(GEMM_ERR_NO_MEMORY, "workspace of %zu bytes: %s", bytes, cudaGetErrorString(e));
            }
        }
        e = simt_fp32_launch(p, (int)M, (int)N, (int)K, static_cast<const float *>(A), lda,
                             static_cast<const float *>(B), ldb, C, ldc, epi, static_cast<float *>(sw), stream);
        if (sw) {
            const cudaError_t f = cudaFreeAsync(sw, stream);
            if (e == cudaSuccess) e = f;
        }
        return e == cudaSuccess ? GEMM_OK : fail(GEMM_ERR_CUDA, "SIMT kernel launch: %s", cudaGetErrorString(e));
    }
    // Tensor-core path: pack operands TMA cannot address, then launch.
    const void *Ause = A, *Buse = B;
    void *ws = nullptr;
    const uint64_t a_bytes = p.pack_a ? (uint64_t)M * plan.lda_eff * eb : 0;
    const uint64_t b_bytes = p.b_kmajor ? (uint64_t)N * plan.ldb_eff * eb
                             : p.pack_b ? (uint64_t)K * plan.ldb_eff * eb : 0;
    const uint64_t a_off = 0, b_off = (a_bytes + 255) / 256 * 256;
    // Partial tiles of split tiles: tail_tiles x splits slabs of (128 * cta_group) x bn floats
    // (none when the K ranges are summed in cluster shared memory).
    const bool slabs = p.tail_tiles > 0 && !p.cluster_split;
    const uint64_t w_bytes = slabs ? (uint64_t)p.tail_tiles * p.splits * 128 * p.cta_group * p.bn * 4 : 0;
    const uint64_t w_off = (b_off + b_bytes + 255) / 256 * 256;
    if (p.pack_a || p.pack_b || p.b_kmajor || slabs) {
        e = cudaMallocAsync(&ws, (size_t)(w_off + w_bytes), stream);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return fail(GEMM_ERR_NO_MEMORY, "workspace of %llu bytes: %s", (unsigned long long)(w_off + w_bytes),
                        cudaGetErrorString(e));
        }
        uint8_t *w = static_cast<uint8_t *>(ws);
        // (one launch per operand: measured faster than one launch over both)
        if (p.pack_a) {
            e = pack_rows_launch(A, lda, w + a_off, plan.lda_eff, M, K, eb, a_lo, a_hi, stream);
            Ause = w + a_off;
        }
        if (e == cudaSuccess && p.b_kmajor) {
            e = transpose_launch(B, ldb, w + b_off, plan.ldb_eff, K, N, eb, stream);
            Buse = w + b_off;
        } else if (e == cudaSuccess && p.pack_b) {
            e = pack_rows_launch(B, ldb, w + b_off, plan.ldb_eff, K, N, eb, b_lo, b_hi, stream);
            Buse = w + b_off;
        }
        if (e != cudaSuccess) {
            cudaFreeAsync(ws, stream);
            return fail(GEMM_ERR_CUDA, "operand pack: %s", cudaGetErrorString(e));
        }
    }
    char err[256] = {0};
    float *Wp = slabs ? reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + w_off) : nullptr;
    rc = tc_launch(p, dtype, (int)M, (int)N, (int)K, Ause, plan.lda_eff, Buse, plan.ldb_eff, C, ldc, Wp, epi,
                   (uint32_t)opt.wait_timeout_ms, stream, err, sizeof err);
    if (rc == GEMM_OK && Wp) {
        const int tile_rows = 128 * p.cta_group;
        e = split_reduce_launch(Wp, p.tail_tiles, p.splits, tile_rows, p.bn, p.tiles - p.tail_tiles,
                                (int)cdiv(M, tile_rows), (int)cdiv(N, p.bn), p.group_m, C, ldc, M, N, epi,
                                stream);
        if (e != cudaSuccess) {
            std::snprintf(err, sizeof err, "split reduce: %s", cudaGetErrorString(e));
            rc = GEMM_ERR_CUDA;
        }
    }
    if (ws) {
        e = cudaFreeAsync(ws, stream);
        if (rc == GEMM_OK && e != cudaSuccess) return fail(GEMM_ERR_CUDA, "cudaFreeAsync: %s", cudaGetErrorString(e));
    }
    if (rc != GEMM_OK) return fail(rc, "%s", err);
    return GEMM_OK;
}

}  // namespace
}  // namespace tcgemm

extern "C" {

int gemm_run(int64_t M, int64_t N, int64_t K, int dtype, const void *A, int64_t lda, const void *B, int64_t ldb,
             float *C, int64_t ldc, struct CUstream_st *stream_) {
    t_err[0] = 0;
    return run(M, N, K, dtype, A, lda, B, ldb, C, ldc, EpiParams(), reinterpret_cast<cudaStream_t>(stream_));
}

int gemm_run_ex(int64_t M, int64_t N, int64_t K, int dtype, const void *A, int64_t lda, const void *B, int64_t ldb,
                void *C, int64_t ldc, const gemm_epilogue_t *epi, struct CUstream_st *stream_) {
    t_err[0] = 0;
    EpiParams e;
    const int rc = api_epilogue(epi, &e);
    if (rc) return rc;
    return run(M, N, K, dtype, A, lda, B, ldb, C, ldc, e, reinterpret_cast<cudaStream_t>(stream_));
}

int gemm_get_status(struct CUstream_st *stream_) {
    t_err[0] = 0;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return fail(GEMM_ERR_CUDA, "cudaStreamSynchronize: %s", cudaGetErrorString(e));
    uint32_t w[4] = {0, 0, 0, 0};
    e = tc_read_and_clear_status(w);
    if (e != cudaSuccess) return fail(GEMM_ERR_CUDA, "status read: %s", cudaGetErrorString(e));
    if (w[0] != 0) {
        static const char *roles[] = {"?", "producer", "mma", "epilogue", "drain"};
        return fail((int)w[0], "kernel wait expired: role=%s tile=%d block=%u", roles[w[1] < 5 ? w[1] : 0],
                    (int)w[2], w[3]);
    }
    return GEMM_OK;
}

}  // extern "C"

// ------------------------------------------------ shared with other entry points ---
namespace tcgemm {

int api_error(int code, const char *message) { return fail(code, "%s", message); }

void api_clear_error() { t_err[0] = 0; }

int api_validate(int64_t M, int64_t N, int64_t K, int dtype, const void *A, int64_t lda, const void *B, int64_t ldb,
                 const void *C, int64_t ldc) {
    return validate(M, N, K, dtype, A, lda, B, ldb, C, ldc);
}

int api_check_device_span(const char *name, const void *p, uint64_t bytes, int dev) {
    return check_device_span(name, p, bytes, dev);
}

int api_check_trace(const Options &opt, int dev) {
    if (!opt.trace_addr) return GEMM_OK;
    return check_device_span("trace buffer", reinterpret_cast<const void *>((uintptr_t)opt.trace_addr),
                             32ull + 32ull * (uint64_t)opt.trace_records, dev);
}

int api_check_device_span_range(const char *name, const void *p, uint64_t bytes, int dev, uint64_t *lo,
                                uint64_t *hi) {
    return check_device_span(name, p, bytes, dev, lo, hi);
}

int api_epilogue(const gemm_epilogue_t *in, EpiParams *out) {
    *out = EpiParams();
    if (!in) return GEMM_OK;
    if (in->activation != GEMM_ACT_NONE && in->activation != GEMM_ACT_RELU && in->activation != GEMM_ACT_GELU)
        return fail(GEMM_ERR_INVALID_ARG, "unknown activation %d", (int)in->activation);
    if (in->out_dtype != GEMM_OUT_F32 && in->out_dtype != GEMM_OUT_BF16 && in->out_dtype != GEMM_OUT_F16)
        return fail(GEMM_ERR_INVALID_ARG, "unknown output type %d", (int)in->out_dtype);
    out->alpha = in->alpha;
    out->beta = in->beta;
    out->bias = in->bias;
    out->act = in->activation;
    out->out = in->out_dtype;
    out->active =
        !(out->alpha == 1.f && out->beta == 0.f && !out->bias && out->act == GEMM_ACT_NONE && out->out == GEMM_OUT_F32);
    return GEMM_OK;
}

int api_elem_bytes(int dtype) { return elem_bytes(dtype); }

int api_device_info(int dev, int *sms, int *cc_major, int *cc_minor, int *max_clusters) {
    DevInfo d;
    int rc = dev_info(dev, &d);
    if (rc) return rc;
    *sms = d.sms;
    *cc_major = d.cc_major;
    *cc_minor = d.cc_minor;
    *max_clusters = d.max_clusters;
    return GEMM_OK;
}

}  // namespace tcgemm
