// Persistent tensor-core GEMM for BF16, FP16, TF32 and FP8 inputs with FP32 accumulation
// in Tensor Memory (tcgen05), fed by TMA, for sm_103a.
//
// Structure, after "Learn CuTeDSL":
//  * section 5.1 / 5.4: warp specialisation around a circular buffer of STAGES
//    shared-memory slots, each with a "full" mbarrier (TMA bytes landed) and an
//    "empty" mbarrier (the MMAs that read it have completed); the phase bit of
//    each barrier flips once per lap of the ring.
//      warp 0      TMA producer (one thread issues every copy),
//      warp 1      allocates Tensor Memory; one thread issues every MMA,
//      warps 2..5  epilogue: Tensor Memory -> registers -> shared -> global.
//  * section 4.3.1: the accumulator lives in Tensor Memory (128 lanes x 512
//    columns of 32 bits); it is allocated once by warp 1 for the CTA's life.
//  * section 4.3.4: every MMA batch follows mbarrier wait -> tcgen05 fence ->
//    MMA issue -> tcgen05.commit onto an mbarrier; the first MMA of each tile
//    runs with the accumulate flag off.
//  * the closing notes of the TFLOPS table: two accumulators (2 x BN columns)
//    so the epilogue of tile i overlaps the MMAs of tile i+1, and the output
//    leaves through swizzled shared memory and TMA stores (section 3.3)
//    instead of strided per-thread stores.
//  * section 8.1: a static persistent schedule -- one CTA (or CTA pair) per SM,
//    striding over output tiles, here in grouped raster order so that tiles
//    that run together share A row-panels and B column-panels in L2.
//  * section 4.3.5: the 2-CTA variant -- a CTA pair computes a 256-row tile
//    with one M=256 MMA issued by the even CTA; each CTA loads its own 128 rows
//    of A and its own half of the B columns with plain (non-multicast) TMA, and
//    signals the even CTA's "full" barrier.
//
// Operand layouts: A is row-major M x K, i.e. K-major; B is row-major K x N,
// i.e. N-major ("MN-major" for the MMA).  Both are staged with the 128-byte
// swizzle.  TMA zero-fills everything outside [0,K) x [0,M) and [0,N) x [0,K),
// so ragged tails add nothing to the sums; TMA stores clip to [0,N) x [0,M).
//
// Every wait is bounded (mbarrier try_wait plus a %globaltimer deadline); on
// expiry the thread records GEMM_ERR_TIMEOUT in a device status word, raises
// a CTA-wide abort flag that every other wait loop checks, and all roles fall
// through to the common teardown, which still frees Tensor Memory.
#include <cudaTypedefs.h>

#include <cstdio>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "epilogue.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "tile_order.cuh"

namespace tcgemm {

__device__ uint32_t g_tc_status[4];

namespace {

constexpr int kThreads = 192;
constexpr int kBM = 128;                       // rows per CTA = Tensor Memory lanes
constexpr int kEpiWarps = 4;
constexpr int kEpiBufBytes = 32 * 128;         // 32 rows x 32 fp32, 128-byte swizzled
constexpr int kEpiBytes = kEpiWarps * 2 * kEpiBufBytes;
constexpr int kSmemBudget = 232448;            // 227 KB opt-in dynamic shared memory
constexpr int kBarBytes = 1024;
constexpr int kUQ = 4;                         // unit-queue slots (dynamic schedule)

enum Role : uint32_t { kRoleProducer = 1, kRoleMma = 2, kRoleEpilogue = 3, kRoleDrain = 4 };

// How B is staged: as stored (N-major, "MN-major" for the MMA), or from a
// K-major transposed copy.  B as stored comes in 128-byte column chunks of BK
// K-rows.  For 16- and 8-bit operands each chunk uses the 128-byte swizzle of
// 16-byte units (atoms of 8 K-rows, 1024 bytes).  The TF32 MMA reads an
// MN-major operand only with the 128-byte swizzle of 32-byte units (measured
// on GB300 by reading back which shared-memory element each (k, n) of one MMA
// took: with 16-byte units it reads nothing valid): atoms of 4 K-rows, 512
// bytes apart, in which row r holds its four 32-byte units in the order
// u ^ (r % 4) -- the layout the TMA engine writes for that swizzle mode.
enum BMode : int { kBNMajor = 0, kBKMajor = 1 };

// Operand element type of a variant.
enum Dt : int { kDtBF16 = 0, kDtTF32 = 1, kDtFP16 = 2, kDtE4M3 = 3, kDtE5M2 = 4 };

constexpr int dt_elem(int dt) { return dt == kDtTF32 ? 4 : (dt == kDtE4M3 || dt == kDtE5M2) ? 1 : 2; }

template <int DT, int CG, int BN, int BMODE>
struct TcCfg {
    static constexpr bool TF32 = DT == kDtTF32;
    static constexpr bool F8 = DT == kDtE4M3 || DT == kDtE5M2;
    static constexpr int KIND = TF32 ? ptx::kKindTF32 : F8 ? ptx::kKindF8 : ptx::kKindF16;
    static constexpr bool BKM = BMODE == kBKMajor;
    static constexpr int ELEM = dt_elem(DT);
    static constexpr int BK = 128 / ELEM;           // one 128-byte swizzle row of K
    static constexpr int UMMA_K = 32 / ELEM;        // K of one MMA: 16 (16-bit) / 8 (tf32) / 32 (fp8)
    static constexpr int KSTEPS = BK / UMMA_K;      // 4 MMAs per stage
    static constexpr int BN_CTA = BN / CG;          // B columns this CTA loads
    static constexpr int CHUNK_COLS = 128 / ELEM;   // columns in one 128-byte row of B
    static constexpr int B_CHUNKS = BN_CTA / CHUNK_COLS;
    static constexpr int B_CHUNK_BYTES = BK * 128;  // one column chunk: BK rows x 128 B
    static constexpr int A_BYTES = kBM * 128;
    // B K-major (a transposed copy, N x K): one box of BN_CTA rows x 128 bytes.
    // B MN-major (as stored, K x N): B_CHUNKS boxes of BK rows x 128 bytes.
    static constexpr int B_BYTES = BKM ? BN_CTA * 128 : B_CHUNKS * B_CHUNK_BYTES;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int B_KSTEP_BYTES = (UMMA_K / 8) * 1024;  // one MMA's K-rows of a 128-byte chunk
    // B as stored: TF32 takes the 32-byte-unit swizzle (4-row atoms 512 B apart),
    // other types the 16-byte-unit one (8-row atoms 1024 B apart).
    static constexpr bool B_ATOM32 = TF32 && !BKM;
    static constexpr uint32_t B_SBO = B_ATOM32 ? 512u : 1024u;
    static constexpr uint32_t B_LAYOUT = B_ATOM32 ? ptx::kLayoutSw128Atom32 : ptx::kLayoutSw128;
    static constexpr int STAGES_FIT = (kSmemBudget - 1024 - kEpiBytes - kBarBytes) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
    static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + kEpiBytes + kBarBytes;
    static constexpr int TMEM_COLS = 2 * BN <= 32 ? 32 : 2 * BN <= 64 ? 64 : 2 * BN <= 128 ? 128 : 2 * BN <= 256 ? 256 : 512;
    // Instruction descriptor: D f32 (bits 4-5 = 1), A/B format (bits 7-9, 10-12:
    // f16 = 0 and bf16 = 1 for kind::f16, tf32 = 2 for kind::tf32, e4m3 = 0 and
    // e5m2 = 1 for kind::f8f6f4), A K-major (bit 15 = 0), B MN-major (bit 16 = 1)
    // or K-major (0), N >> 3 in bits 17-22, M >> 4 in bits 24-28.
    static constexpr uint32_t FMT = DT == kDtTF32 ? 2u : (DT == kDtFP16 || DT == kDtE4M3) ? 0u : 1u;
    static constexpr uint32_t IDESC = (1u << 4) | (FMT << 7) | (FMT << 10) | ((BKM ? 0u : 1u) << 16) |
                                      ((uint32_t)(BN >> 3) << 17) | ((uint32_t)((kBM * CG) >> 4) << 24);
    // The same MMA at half the tile width (a column-half unit).
    static constexpr uint32_t IDESC_HALF = (IDESC & ~(0x3Fu << 17)) | ((uint32_t)((BN / 2) >> 3) << 17);
    // A column half reads B as stored in whole 128-byte chunks; a K-major B box
    // is loaded whole and the MMA reads its first half.
    static constexpr bool HALVES = (BN / 2) % 16 == 0 && BN / 2 >= 64 && (BKM || B_CHUNKS % 2 == 0);
    static_assert(BN % 16 == 0 && BN >= 32 && BN <= 256, "MMA N out of range");
    static_assert(BKM || (BN_CTA % CHUNK_COLS == 0 && B_CHUNKS >= 1), "B tile must be whole 128-byte chunks");
    static_assert(BN_CTA <= 256, "TMA box rows");
    static_assert(STAGES >= 2, "shared memory too small for a ring");
    static_assert(2 * BN <= 512, "two accumulators must fit in Tensor Memory");
    static_assert(SMEM_BYTES <= kSmemBudget, "shared memory budget exceeded");
    static_assert((2 * STAGES + 65) * 8 <= kBarBytes, "barrier area too small");
    // Split K reduced across a cluster: the partials a CTA receives (one per
    // other K range, for its lane quarters) and the ones it stages to send
    // (its other lane quarters) fit in its idle ring: at most 6 quarter-tiles.
    static_assert(6 * 32 * BN * 4 <= STAGES * STAGE_BYTES, "ring too small for the cluster split-K partials");
    // (with 2 ranges: 2 received + 2 staged to send + 2 of the owner's own = 6 as well)
};

struct TcParams {
    int M, N, K;
    int tiles_m, tiles_n, num_tiles;   // tiles of (128*CG) x BN
    int num_kb;                        // ceil(K / BK)
    int full_tiles;                    // tiles [0, full_tiles) run over all of K and store to C
    int tail_tiles;                    // the remaining tiles run as `splits` K ranges each
    int splits;                        // K ranges per tail tile
    int half_tiles;                    // or: the last tiles run as two column halves each, over all of K, to C
    int kb_per_split;                  // k-blocks per K range
    int num_units;                     // full_tiles + tail_tiles * splits work units
    int group_m;                       // raster group height, in tile rows
    int tma_store;
    int debug_stall;                   // test hook: the MMA thread first waits on a barrier nothing arrives at
    void *C;                           // FP32, or epi.out when the epilogue is active
    int64_t ldc;
    EpiParams epi;                     // fused epilogue
    const GroupDesc *groups;           // grouped launch: per-group sizes, maps and C (nullptr: one GEMM)
    int group_count;
    int sched;                         // 0: static stride over units; 1: Cluster Launch Control
    int csplit;                        // 0, or the K ranges of each tile reduced across a cluster of that
                                       // many CTAs (one tile per cluster; cta_group 1)
    int csr_rx;                        // 0: each CTA of the cluster owns some lane quarters of the tile;
                                       // else (2 ranges) CTA 0 owns the whole tile and receives CTA 1's
                                       // partial at this byte offset of its shared memory, past the ring
    int ring;                          // ring stages in use (0: all STAGES); fewer leave csr_rx free
    unsigned long long timeout_ns;
    uint32_t *trace_count;             // timeline trace: record counter (nullptr: off)
    gemm_trace_record_t *trace;        // and the records after it
    int trace_cap;
};

// Work unit u -> output tile (tm, tn), its K range [kb0, kb1), the slab its
// partial sum goes to (-1: the unit covers all of K and stores to C) and the
// column half it covers (-1: the whole tile width).
//
// Units [0, full_tiles) are whole tiles.  The tiles that would leave part of
// the machine idle in the last round of the persistent schedule are either
// (a) run as two column halves each, over all of K and straight to C, when
//     the halves fit in one round (each half drains half the accumulator, so
//     the launch's last epilogue is shorter; the main loop of a half takes
//     as many cycles as a whole tile's: the K-block cadence, not the MMA,
//     sets it); or
// (b) split into K ranges, as is every tile when K is split throughout; the
//     ranges of one split index come together, so units that run at once read
//     the same slices of A and B.  Partial tiles go to slabs (one full tile
//     each) that a second kernel sums in split order.
__device__ __forceinline__ void unit_coords(int u, const TcParams &p, int &tm, int &tn, int &kb0, int &kb1,
                                            int &slab, int &half) {
    half = -1;
    if (u < p.full_tiles) {
        tile_coords(u, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
        kb0 = 0;
        kb1 = p.num_kb;
        slab = -1;
        return;
    }
    const int v = u - p.full_tiles;
    if (p.half_tiles > 0) {
        half = v / p.half_tiles;
        tile_coords(p.full_tiles + (v - half * p.half_tiles), p.tiles_m, p.tiles_n, p.group_m, tm, tn);
        kb0 = 0;
        kb1 = p.num_kb;
        slab = -1;
        return;
    }
    const int split = v / p.tail_tiles;
    const int i = v - split * p.tail_tiles;
    tile_coords(p.full_tiles + i, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
    kb0 = split * p.kb_per_split;
    kb1 = min(p.num_kb, kb0 + p.kb_per_split);
    slab = split * p.tail_tiles + i;
}

// Everything a role needs about one work unit: its tile, K range and slab
// (unit_coords), and the GEMM it belongs to -- the kernel's own parameters, or
// in a grouped launch the descriptor of the group whose units contain u (a
// binary search over the groups' first units).
struct Unit {
    int tm, tn, kb0, kb1, slab;
    int half;                          // -1: the whole tile width; 0 / 1: that column half
    int M, N;
    const CUtensorMap *mA, *mB, *mC;
    void *C;
    int64_t ldc;
    const float *bias;
    int tma_store;
    int group;                         // -1 outside a grouped launch
};

__device__ __forceinline__ Unit unit_info(int u, const TcParams &p, const CUtensorMap *tmA, const CUtensorMap *tmB,
                                          const CUtensorMap *tmC) {
    Unit U;
    if (p.groups == nullptr) {
        unit_coords(u, p, U.tm, U.tn, U.kb0, U.kb1, U.slab, U.half);
        U.M = p.M;
        U.N = p.N;
        U.mA = tmA;
        U.mB = tmB;
        U.mC = tmC;
        U.C = p.C;
        U.ldc = p.ldc;
        U.bias = p.epi.bias;
        U.tma_store = p.tma_store;
        U.group = -1;
        return U;
    }
    int lo = 0, hi = p.group_count - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.groups[mid].unit_start <= u) lo = mid;
        else hi = mid - 1;
    }
    const GroupDesc *g = p.groups + lo;
    tile_coords(u - g->unit_start, g->tiles_m, g->tiles_n, p.group_m, U.tm, U.tn);
    U.kb0 = 0;
    U.kb1 = g->num_kb;
    U.slab = -1;
    U.half = -1;
    U.M = g->M;
    U.N = g->N;
    U.mA = &g->tmA;
    U.mB = &g->tmB;
    U.mC = &g->tmC;
    U.C = g->C;
    U.ldc = g->ldc;
    U.bias = g->bias;
    U.tma_store = g->tma_store;
    U.group = lo;
    return U;
}

// One timeline record (when tracing is on): a span of `role` on `unit`.
// A recording thread reserves record slots kTraceBlock at a time with one
// atomic on the buffer's counter (slot.x = its next slot, slot.y = the end of
// its block; returned updated) and fills them with plain stores, so that a
// record costs no round trip to L2; slots it reserves but does not fill stay
// as the caller zeroed them (role 0).
constexpr uint32_t kTraceBlock = 16;
__device__ __noinline__ uint2 trace_put(const TcParams &p, uint2 slot, int role, int unit, int sub, uint64_t t0,
                                        uint64_t t1) {
    if (slot.x == slot.y) {
        slot.x = atomicAdd(p.trace_count, kTraceBlock);
        slot.y = slot.x + kTraceBlock;
    }
    const uint32_t i = slot.x++;
    if (i >= (uint32_t)p.trace_cap) return slot;
    gemm_trace_record_t r;
    r.t_begin_ns = t0;
    r.t_end_ns = t1;
    r.unit = unit;
    r.role = (int16_t)role;
    r.sm = (int16_t)ptx::smid();
    r.cta = (int32_t)blockIdx.x;
    r.sub = sub;
    p.trace[i] = r;
    return slot;
}

__device__ __noinline__ void record_failure(uint32_t role, int tile, volatile int *abort_flag) {
    *abort_flag = 1;
    if (atomicCAS(&g_tc_status[0], 0u, (uint32_t)GEMM_ERR_TIMEOUT) == 0u) {
        g_tc_status[1] = role;
        g_tc_status[2] = (uint32_t)tile;
        g_tc_status[3] = blockIdx.x;
        __threadfence();
    }
}

template <bool CLUSTER>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                         unsigned long long timeout_ns) {
    if (ptx::mbar_try_wait<CLUSTER>(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (ptx::mbar_try_wait<CLUSTER>(bar, parity)) return true;
        if (*abort_flag) return false;
        if (ptx::globaltimer_ns() - t0 > timeout_ns) return false;
    }
}

template <int DT, int CG, int BN, int BMODE>
__global__ void __launch_bounds__(kThreads, 1)
tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmW, const TcParams p) {
    using Cf = TcCfg<DT, CG, BN, BMODE>;
    constexpr bool kPair = CG == 2;
    constexpr bool BKM = Cf::BKM;
    const bool tracing = p.trace_count != nullptr;
    const uint64_t t_start = tracing ? ptx::globaltimer_ns() : 0;
    uint2 tslot = make_uint2(0u, 0u);   // this thread's reserved trace slots (trace_put)
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment (in the shared window) for the swizzle atoms.
    const uint32_t raw_addr = ptx::smem_addr(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    uint8_t *stages = smem;
    uint8_t *epi = smem + Cf::STAGES * Cf::STAGE_BYTES;
    // Barrier area, in 8-byte words: full[S], empty[S], acc_full[2], acc_empty[2],
    // never, old_c[8], unit queue full[4] / empty[4], clc_full, clc_used, pad,
    // CLC response (2 words), unit queue (2 words), TMEM slot + abort flag,
    // cluster split-K ready[4] / partials-in[4].
    uint64_t *bars = reinterpret_cast<uint64_t *>(epi + kEpiBytes);
    constexpr int kW = 2 * Cf::STAGES;
    uint8_t *clc_resp = reinterpret_cast<uint8_t *>(bars + kW + 24);          // 16-byte aligned
    volatile int *unit_q = reinterpret_cast<volatile int *>(bars + kW + 26);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + kW + 28);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const uint32_t bar0 = ptx::smem_addr(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * (uint32_t)s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (uint32_t)(Cf::STAGES + s); };
    auto accf_bar = [&](int a) { return bar0 + 8u * (uint32_t)(2 * Cf::STAGES + a); };
    auto acce_bar = [&](int a) { return bar0 + 8u * (uint32_t)(2 * Cf::STAGES + 2 + a); };
    const uint32_t never_bar = bar0 + 8u * (uint32_t)(2 * Cf::STAGES + 4);   // never arrived at
    // old-C loads of the residual epilogue: one barrier per staging buffer
    auto oldc_bar = [&](int i) { return bar0 + 8u * (uint32_t)(kW + 5 + i); };
    // dynamic schedule: unit queue slots (producer -> MMA, epilogue) and the CLC response
    auto uq_full = [&](int i) { return bar0 + 8u * (uint32_t)(kW + 13 + i); };
    auto uq_empty = [&](int i) { return bar0 + 8u * (uint32_t)(kW + 17 + i); };
    const uint32_t clc_full = bar0 + 8u * (uint32_t)(kW + 21);
    const uint32_t clc_used = bar0 + 8u * (uint32_t)(kW + 22);   // leader: both CTAs read the response
    // cluster split-K, per TMEM lane quarter: ready (the owning CTA's ring is
    // free to receive) and, per 32-column chunk, in (every other K range's
    // partial of that chunk has arrived)
    auto csr_ready = [&](uint32_t q) { return bar0 + 8u * (uint32_t)(kW + 29) + 8u * q; };
    auto csr_in = [&](uint32_t q, uint32_t c) { return bar0 + 8u * (uint32_t)(kW + 33) + 8u * (q * 8u + c); };
    const bool dyn = p.sched != 0;

    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = kPair ? ptx::cluster_ctarank() : 0u;
    // Cluster split-K: CTA crank of each cluster takes K range crank of the
    // cluster's one tile (work unit crank * tiles + tile); no further units.
    const uint32_t csplit = (uint32_t)p.csplit;
    const uint32_t crank = csplit ? ptx::cluster_ctarank() : 0u;
    const int unit = csplit ? (int)(crank * (uint32_t)p.tail_tiles + blockIdx.x / csplit) : (int)blockIdx.x / CG;
    const int nunits = csplit ? p.num_units : (int)gridDim.x / CG;
    const int ring = p.ring > 0 ? p.ring : Cf::STAGES;

    if (threadIdx.x == 0) {
        for (int s = 0; s < Cf::STAGES; ++s) {
            ptx::mbar_init(full_bar(s), 1);
            ptx::mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(accf_bar(a), 1);
            ptx::mbar_init(acce_bar(a), kEpiWarps * CG);
        }
        ptx::mbar_init(never_bar, 1);
        for (int i = 0; i < 2 * kEpiWarps; ++i) ptx::mbar_init(oldc_bar(i), 1);
        for (int i = 0; i < kUQ; ++i) {
            ptx::mbar_init(uq_full(i), 1);
            // consumers: the MMA thread (leader CTA only) and each epilogue warp
            ptx::mbar_init(uq_empty(i), (rank == 0 ? 1 : 0) + kEpiWarps);
        }
        ptx::mbar_init(clc_full, 1);
        ptx::mbar_init(clc_used, CG);
        for (uint32_t i = 0; i < 4; ++i) {
            ptx::mbar_init(csr_ready(i), 1);               // the owner's one arrival
            for (uint32_t c = 0; c < 8; ++c) ptx::mbar_init(csr_in(i, c), 1);   // the owner's, plus the bytes
        }
        *abort_flag = 0;
        ptx::fence_mbar_init();
        if (csplit == 2 && p.csr_rx && crank == 0)
            // one owner: the bytes of every chunk of the peer's partial, expected from the start
            for (uint32_t i = 0; i < 4; ++i)
                for (uint32_t c = 0; c < (uint32_t)(BN / 32); ++c) ptx::mbar_arrive_expect_tx(csr_in(i, c), 4096u);
    }
    if (warp == 0 && lane == 0 && p.groups == nullptr) {
        ptx::prefetch_tensormap(&tmA);
        ptx::prefetch_tensormap(&tmB);
        if (p.tma_store) ptx::prefetch_tensormap(&tmC);
        if (p.tail_tiles) ptx::prefetch_tensormap(&tmW);
    }
    if (warp == 1) {
        ptx::tmem_alloc<CG>(ptx::smem_addr(tmem_slot), Cf::TMEM_COLS);
        ptx::tmem_relinquish<CG>();
    }
    ptx::tc_fence_before();
    if (kPair || csplit) ptx::cluster_sync(); else __syncthreads();   // peers' barriers ready before any remote arrive
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // Launched as a programmatic dependent of the previous kernel on the
    // stream, this CTA may have started before that kernel ended: the set-up
    // above touched only its own shared and Tensor Memory.  Wait here, before
    // any global-memory access, for that kernel to finish and its writes to be
    // visible; then let the next launch start its own set-up (when no split-K
    // reduction, which reads this grid's slabs, comes next).
    const uint64_t t_synced = tracing ? ptx::globaltimer_ns() : 0;
    ptx::pdl_wait();
    if ((p.tail_tiles == 0 || csplit) && threadIdx.x == 0) ptx::pdl_launch_dependents();
    if (tracing && threadIdx.x == 0) {
        // set-up: barriers, Tensor Memory and the CTA (or cluster) barrier; then the wait for the previous grid
        tslot = trace_put(p, tslot, 5, -1, 0, t_start, t_synced);
        tslot = trace_put(p, tslot, 5, -1, 1, t_synced, ptx::globaltimer_ns());
    }

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int last_group = -1;
            // All k-blocks of unit t into the ring; false once a wait expired.
            auto load_unit = [&](int t) -> bool {
                const Unit U = unit_info(t, p, &tmA, &tmB, &tmC);
                if (U.group != last_group) {
                    // a group's maps were copied in before the launch: acquire them for TMA
                    ptx::fence_tensormap_acquire(U.mA);
                    ptx::fence_tensormap_acquire(U.mB);
                    ptx::prefetch_tensormap(U.mA);
                    ptx::prefetch_tensormap(U.mB);
                    last_group = U.group;
                }
                // A column-half unit: this CTA's share is half as wide; B as stored
                // then comes in half the chunks (a K-major box is loaded whole).
                const bool halfu = Cf::HALVES && U.half >= 0;
                const int cta_cols = halfu ? Cf::BN_CTA / 2 : Cf::BN_CTA;
                const int m0 = U.tm * (kBM * CG) + (int)rank * kBM;
                const int n0 = U.tn * BN + (halfu ? U.half * (BN / 2) : 0) + (int)rank * cta_cols;
                const int nchunks = BKM ? 0 : cta_cols / Cf::CHUNK_COLS;
                const uint32_t tx_bytes =
                    (uint32_t)((Cf::A_BYTES + (BKM ? Cf::B_BYTES : nchunks * Cf::B_CHUNK_BYTES)) * CG);
                const uint64_t t_unit = tracing ? ptx::globaltimer_ns() : 0;
                for (int kb = U.kb0; kb < U.kb1; ++kb) {
                    if (!wait_bar<kPair>(empty_bar(stage), phase ^ 1u, abort_flag, p.timeout_ns)) {
                        record_failure(kRoleProducer, t, abort_flag);
                        return false;
                    }
                    const uint32_t fb = full_bar(stage);
                    if (rank == 0) ptx::mbar_arrive_expect_tx(fb, tx_bytes);
                    const uint32_t sa = ptx::smem_addr(stages + stage * Cf::STAGE_BYTES);
                    const uint32_t sb = sa + Cf::A_BYTES;
                    const int k0 = kb * Cf::BK;
                    if (!kPair) {
                        ptx::tma_load_2d(sa, U.mA, fb, k0, m0);
                        if (BKM) {
                            ptx::tma_load_2d(sb, U.mB, fb, k0, n0);
                        } else {
#pragma unroll
                            for (int c = 0; c < Cf::B_CHUNKS; ++c)
                                if (c < nchunks)
                                    ptx::tma_load_2d(sb + c * Cf::B_CHUNK_BYTES, U.mB, fb, n0 + c * Cf::CHUNK_COLS, k0);
                        }
                    } else {
                        const uint32_t fb_even = ptx::mapa_shared(fb, 0);
                        ptx::tma_load_2d_pair(sa, U.mA, fb_even, k0, m0);
                        if (BKM) {
                            ptx::tma_load_2d_pair(sb, U.mB, fb_even, k0, n0);
                        } else {
#pragma unroll
                            for (int c = 0; c < Cf::B_CHUNKS; ++c)
                                if (c < nchunks)
                                    ptx::tma_load_2d_pair(sb + c * Cf::B_CHUNK_BYTES, U.mB, fb_even,
                                                          n0 + c * Cf::CHUNK_COLS, k0);
                        }
                    }
                    if (++stage == ring) { stage = 0; phase ^= 1u; }
                }
                if (tracing) tslot = trace_put(p, tslot, 1, t, U.kb1 - U.kb0, t_unit, ptx::globaltimer_ns());
                return true;
            };
            if (!dyn) {
                // static persistent schedule: every unit'th unit, striding by the grid
                for (int t = unit; ok && t < p.num_units; t += nunits) ok = load_unit(t);
            } else {
                // Cluster Launch Control: start on this cluster's own unit, then
                // steal the units of clusters that have not started yet.  Each
                // unit (and finally -1) is published to the MMA thread and the
                // epilogue warps through the unit queue.  In a CTA pair the
                // leader asks, the response reaches both CTAs, and the leader
                // asks again only once both have read the previous one.
                int t = unit;
                int qslot = 0;
                uint32_t qphase = 0, clc_phase = 0, used_phase = 0;
                bool more = true, asked_before = false;
                const uint32_t resp = ptx::smem_addr(clc_resp);
                while (ok) {
                    if (!wait_bar<false>(uq_empty(qslot), qphase ^ 1u, abort_flag, p.timeout_ns)) {
                        record_failure(kRoleProducer, t, abort_flag);
                        ok = false;
                        break;
                    }
                    unit_q[qslot] = t;
                    ptx::mbar_arrive(uq_full(qslot));
                    if (++qslot == kUQ) { qslot = 0; qphase ^= 1u; }
                    if (t < 0) break;
                    if (more) {
                        // ask for the next unit while this one loads
                        ptx::mbar_arrive_expect_tx(clc_full, 16u);
                        if (rank == 0) {
                            if (kPair && asked_before) {
                                if (!wait_bar<kPair>(clc_used, used_phase, abort_flag, p.timeout_ns)) {
                                    record_failure(kRoleProducer, t, abort_flag);
                                    ok = false;
                                    break;
                                }
                                used_phase ^= 1u;
                            }
                            ptx::fence_proxy_async_smem();   // our read of the last response before the next write
                            if (kPair) ptx::clc_try_cancel_multicast(resp, clc_full);
                            else ptx::clc_try_cancel(resp, clc_full);
                        }
                        asked_before = true;
                    }
                    ok = load_unit(t);
                    if (!ok) break;
                    if (!more) {
                        t = -1;
                        continue;
                    }
                    if (!wait_bar<kPair>(clc_full, clc_phase, abort_flag, p.timeout_ns)) {
                        record_failure(kRoleProducer, t, abort_flag);
                        ok = false;
                        break;
                    }
                    clc_phase ^= 1u;
                    uint32_t first_x = 0;
                    const bool got = ptx::clc_query(resp, first_x) != 0;
                    if (kPair) ptx::mbar_arrive_cluster(ptx::mapa_shared(clc_used, 0));
                    if (got && (int)(first_x / CG) < p.num_units) {
                        t = (int)(first_x / CG);
                    } else {
                        t = -1;                  // nothing left to steal: every unit has its cluster
                        more = false;
                    }
                }
            }
            // Drain: wait until the MMAs have released every slot, so that no
            // tensor-core read of this CTA's shared memory and no commit
            // arrival on its barriers is still outstanding at teardown.
            for (int i = 0; ok && i < ring; ++i) {
                if (!wait_bar<kPair>(empty_bar(stage), phase ^ 1u, abort_flag, p.timeout_ns)) {
                    record_failure(kRoleDrain, -1, abort_flag);
                    break;
                }
                if (++stage == ring) { stage = 0; phase ^= 1u; }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (rank == 0 && lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            // Test hook: wait on a barrier nothing arrives at, for half the bound, so
            // that this wait (and not the producer's, stalled behind it) expires first.
            if (p.debug_stall && !wait_bar<kPair>(never_bar, 0u, abort_flag, p.timeout_ns / 2)) {
                record_failure(kRoleMma, unit, abort_flag);
                ok = false;
            }
            // The unit sequence: the static stride, or the producer's unit queue.
            int qslot = 0;
            uint32_t qphase = 0;
            auto next_unit = [&](int t, int &out) -> bool {
                if (!dyn) {
                    out = (t < 0 ? unit : t + nunits);
                    if (out >= p.num_units) out = -1;
                    return true;
                }
                if (!wait_bar<false>(uq_full(qslot), qphase, abort_flag, p.timeout_ns)) return false;
                out = unit_q[qslot];
                ptx::mbar_arrive(uq_empty(qslot));
                if (++qslot == kUQ) { qslot = 0; qphase ^= 1u; }
                return true;
            };
            int t = -1;
            if (ok && !next_unit(-1, t)) {
                record_failure(kRoleMma, unit, abort_flag);
                ok = false;
            }
            while (ok && t >= 0) {
                const Unit U = unit_info(t, p, &tmA, &tmB, &tmC);
                const int kb0 = U.kb0, kb1 = U.kb1;
                const uint32_t idesc = (Cf::HALVES && U.half >= 0) ? Cf::IDESC_HALF : Cf::IDESC;
                if (!wait_bar<kPair>(acce_bar(acc), acc_phase ^ 1u, abort_flag, p.timeout_ns)) {
                    record_failure(kRoleMma, t, abort_flag);
                    break;
                }
                ptx::tc_fence_after();
                const uint64_t t_unit = tracing ? ptx::globaltimer_ns() : 0;
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!wait_bar<kPair>(full_bar(stage), phase, abort_flag, p.timeout_ns)) {
                        record_failure(kRoleMma, t, abort_flag);
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t sa = ptx::smem_addr(stages + stage * Cf::STAGE_BYTES);
                    const uint32_t sb = sa + Cf::A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < Cf::KSTEPS; ++kk) {
                        // A: K-major, 8-row groups 1024 B apart; K advances 32 B inside the swizzle row.
                        const uint64_t adesc = ptx::sdesc_sw128(sa + 32u * kk, 16u, 1024u);
                        // B K-major: laid out like A.  B MN-major: 128-byte column chunks
                        // B_CHUNK_BYTES apart (leading), swizzle atoms of K-rows B_SBO apart (stride).
                        const uint64_t bdesc =
                            BKM ? ptx::sdesc_sw128(sb + 32u * kk, 16u, 1024u)
                                : ptx::sdesc(sb + (uint32_t)(Cf::B_KSTEP_BYTES * kk), (uint32_t)Cf::B_CHUNK_BYTES,
                                             Cf::B_SBO, Cf::B_LAYOUT);
                        ptx::mma<CG, Cf::KIND>(d_tmem, adesc, bdesc, idesc, (kb != kb0 || kk != 0) ? 1u : 0u);
                    }
                    if (kPair) ptx::mma_commit_pair(empty_bar(stage), 0x3);
                    else ptx::mma_commit(empty_bar(stage));
                    if (++stage == ring) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                if (kPair) ptx::mma_commit_pair(accf_bar(acc), 0x3);
                else ptx::mma_commit(accf_bar(acc));
                if (tracing) tslot = trace_put(p, tslot, 2, t, kb1 - kb0, t_unit, ptx::globaltimer_ns());
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
                if (!next_unit(t, t)) {
                    record_failure(kRoleMma, t, abort_flag);
                    break;
                }
            }
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------- epilogue
        // Each warp owns 32 accumulator rows (its Tensor Memory lane quarter)
        // and stages boxes of 32 rows x 128 bytes -- 32 FP32 columns, or 64
        // columns of a 16-bit output -- in two buffers, so one box is filled
        // while the TMA store of the previous one drains.
        const uint32_t ew = warp - 2;        // staging-buffer owner index
        const uint32_t q = warp & 3;         // Tensor Memory lane quarter this warp may read
        uint8_t *bufs = epi + ew * 2 * kEpiBufBytes;
        const bool fused = p.epi.active != 0;
        const bool need_old = fused && p.epi.beta != 0.f;
        const int out = p.epi.out;
        int acc = 0;
        uint32_t acc_phase = 0;
        uint32_t nchunk = 0;                 // boxes staged so far (buffer nchunk & 1)
        uint32_t old_phase = 0;              // parity of each buffer's old-C barrier
        uint64_t t_last_issue = 0;           // (traced) when this warp issued its last TMA store
        bool ok = true;
        int last_group = -1;
        // The unit sequence: the static stride, or the producer's unit queue
        // (every lane waits, lane 0 frees the slot).
        int qslot = 0;
        uint32_t qphase = 0;
        auto next_unit = [&](int t, int &out) -> bool {
            if (!dyn) {
                out = (t < 0 ? unit : t + nunits);
                if (out >= p.num_units) out = -1;
                return true;
            }
            const bool got = wait_bar<false>(uq_full(qslot), qphase, abort_flag, p.timeout_ns);
            if (!__all_sync(0xffffffffu, got)) return false;
            out = unit_q[qslot];
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(uq_empty(qslot));
            if (++qslot == kUQ) { qslot = 0; qphase ^= 1u; }
            return true;
        };
        int t = -1;
        if (!next_unit(-1, t)) {
            if (lane == 0) record_failure(kRoleEpilogue, unit, abort_flag);
            ok = false;
        }
        while (ok && t >= 0) {
            const Unit U = unit_info(t, p, &tmA, &tmB, &tmC);
            const int slab = U.slab;
            const int m0 = U.tm * (kBM * CG) + (int)rank * kBM + 32 * (int)q;   // this warp's first row
            const bool halfu = Cf::HALVES && U.half >= 0;
            const int ucols = halfu ? BN / 2 : BN;                                // columns of this unit
            const int n0 = U.tn * BN + (halfu ? U.half * (BN / 2) : 0);
            const int srow = (int)rank * kBM + 32 * (int)q;                       // same row inside a slab
            const bool to_slab = slab >= 0 && !csplit;
            const bool use_tma = to_slab || U.tma_store;
            if (U.group != last_group) {
                if (lane == 0 && U.tma_store) {
                    ptx::fence_tensormap_acquire(U.mC);
                    ptx::prefetch_tensormap(U.mC);
                }
                last_group = U.group;
            }
            EpiParams e = p.epi;             // the group's own bias in a grouped launch
            e.bias = U.bias;
            // The epilogue runs in registers (thread = row) when the box leaves
            // through TMA; partial sums of a split tile go to their slab raw.
            const bool reg_epi = fused && U.tma_store && !to_slab;
            const bool pack16 = reg_epi && out != GEMM_OUT_F32;
            const int box_cols = pack16 ? 64 : 32;
            const bool lane_ok = wait_bar<kPair>(accf_bar(acc), acc_phase, abort_flag, p.timeout_ns);
            if (!__all_sync(0xffffffffu, lane_ok)) {
                if (lane == 0) record_failure(kRoleEpilogue, t, abort_flag);
                break;
            }
            ptx::tc_fence_after();
            const uint64_t t_unit = tracing ? ptx::globaltimer_ns() : 0;
            uint64_t t_first_in = 0, t_last_in = 0;     // cluster split-K owner: partials' arrival (traced)
            const uint32_t trow = tmem_base + ((32u * q) << 16) + (uint32_t)(acc * BN);
            // Split K reduced across the cluster ("Learn CuTeDSL" section 9:
            // distributed shared memory of a thread-block cluster).  Lane
            // quarter q of the tile belongs to CTA q / (4 / csplit).  Each
            // other CTA stages its partial of it, 32 rows x BN FP32, in its
            // own ring (idle now: each CTA has run its only unit) and moves
            // it to the owner's ring with one bulk copy per 32-column chunk,
            // whose bytes complete the owner's barrier of that chunk.  The
            // owner adds each chunk to its own, in K-range order, as soon as
            // it has arrived.  Ring layout: the received quarter-tiles first,
            // (csplit - 1) * 4 / csplit of them, then the ones staged to send.
            if (csplit == 2 && p.csr_rx) {
                // Two K ranges, one owner: CTA 0 of the cluster runs the longer
                // first range and sums and stores the whole tile; CTA 1 runs the
                // second and sends its partial the moment its MMAs end, while
                // CTA 0 still streams.  The partial lands past CTA 0's ring
                // (which runs `ring` stages deep for this), whose chunk barriers
                // CTA 0 armed at set-up, so the sender needs no go-ahead.  The
                // layout of a quarter's chunk: 32 rows of 128 bytes, 16-byte
                // units swizzled by row (the TMA store's box layout).
                const uint32_t part_bytes = 32u * (uint32_t)BN * 4u;
                const uint32_t rx = ptx::smem_addr(stages) + (uint32_t)p.csr_rx + q * part_bytes;
                if (crank != 0) {
                    uint8_t *local = stages + q * part_bytes;          // this CTA's ring, idle now
                    const uint32_t dst = ptx::mapa_shared(rx, 0);
#pragma unroll 1
                    for (int c = 0; c < BN / 32; ++c) {
                        uint32_t r[32];
                        ptx::tmem_ld_32x32b_x32(trow + (uint32_t)(32 * c), r);
                        ptx::tmem_wait_ld(r);
                        uint8_t *row = local + c * 4096 + lane * 128u;
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            *reinterpret_cast<uint4 *>(row + (((uint32_t)k ^ (lane & 7u)) * 16u)) =
                                make_uint4(r[4 * k], r[4 * k + 1], r[4 * k + 2], r[4 * k + 3]);
                        ptx::fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0)
                            ptx::bulk_copy_to_peer(dst + (uint32_t)c * 4096u, ptx::smem_addr(local + c * 4096), 4096u,
                                                   ptx::mapa_shared(csr_in(q, (uint32_t)c), 0));
                    }
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(acce_bar(acc));
                    if (tracing && lane == 0) tslot = trace_put(p, tslot, 3, t, (int)q + 4, t_unit, ptx::globaltimer_ns());
                } else {
                    uint8_t *slot = stages + p.csr_rx + q * part_bytes;
#pragma unroll 1
                    for (int c = 0; c < BN / 32; ++c) {
                        uint32_t r[32];
                        ptx::tmem_ld_32x32b_x32(trow + (uint32_t)(32 * c), r);
                        ptx::tmem_wait_ld(r);
                        if (c == BN / 32 - 1) {
                            // the accumulator is in registers: hand Tensor Memory back
                            ptx::tc_fence_before();
                            __syncwarp();
                            if (lane == 0) ptx::mbar_arrive(acce_bar(acc));
                        }
                        const bool got = wait_bar<true>(csr_in(q, (uint32_t)c), 0u, abort_flag, p.timeout_ns);
                        if (!__all_sync(0xffffffffu, got)) {
                            if (lane == 0) record_failure(kRoleEpilogue, t, abort_flag);
                            ok = false;
                            break;
                        }
                        if (tracing) {
                            t_last_in = ptx::globaltimer_ns();
                            if (c == 0) t_first_in = t_last_in;
                        }
                        uint8_t *srow = slot + c * 4096 + lane * 128u;
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const uint32_t off = ((uint32_t)k ^ (lane & 7u)) * 16u;
                            const float4 b = *reinterpret_cast<const float4 *>(srow + off);
                            // K-range order: this CTA's range 0, then the peer's range 1
                            *reinterpret_cast<float4 *>(srow + off) =
                                make_float4(__uint_as_float(r[4 * k]) + b.x, __uint_as_float(r[4 * k + 1]) + b.y,
                                            __uint_as_float(r[4 * k + 2]) + b.z, __uint_as_float(r[4 * k + 3]) + b.w);
                        }
                        ptx::fence_proxy_async_smem();
                        __syncwarp();
                        const int col0 = n0 + 32 * c;
                        if (lane == 0 && m0 < U.M && col0 < U.N) {
                            ptx::tma_store_2d(U.mC, rx + (uint32_t)c * 4096u, col0, m0);
                            ptx::bulk_commit_group();
                            if (tracing) t_last_issue = ptx::globaltimer_ns();
                        }
                    }
                    if (tracing && lane == 0) {
                        tslot = trace_put(p, tslot, 3, t, (int)q, t_unit, ptx::globaltimer_ns());
                        tslot = trace_put(p, tslot, 6, t, 0, t_unit, t_first_in);
                        tslot = trace_put(p, tslot, 6, t, 1, t_first_in, t_last_in);
                        tslot = trace_put(p, tslot, 6, t, 2, t_last_in, t_last_issue);
                    }
                }
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
                if (!ok) break;
                if (!next_unit(t, t)) {
                    if (lane == 0) record_failure(kRoleEpilogue, t, abort_flag);
                    break;
                }
                continue;
            }
            bool csr_owner = false;                    // this warp sums its quarter's K ranges
            uint32_t csr_base = 0;                     // where the other ranges' partials of it land
            if (csplit) {
                const uint32_t per = 4u / csplit, owner = q / per, qloc = q % per;
                const uint32_t part_bytes = 32u * (uint32_t)BN * 4u;
                if (owner != crank) {
                    const bool rdy = wait_bar<true>(csr_ready(q), 0u, abort_flag, p.timeout_ns);
                    if (!__all_sync(0xffffffffu, rdy)) {
                        if (lane == 0) record_failure(kRoleEpilogue, t, abort_flag);
                        break;
                    }
                    const uint32_t j = crank < owner ? crank : crank - 1;
                    const uint32_t dst = ptx::mapa_shared(ptx::smem_addr(stages) + (j * per + qloc) * part_bytes, owner);
                    // staged after the received quarter-tiles, one region per quarter this CTA sends
                    const uint32_t sent = q < crank * per ? q : q - per;
                    uint8_t *local = stages + ((csplit - 1) * per + sent) * part_bytes;
#pragma unroll 1
                    for (int c = 0; c < BN / 32; ++c) {
                        uint32_t r[32];
                        ptx::tmem_ld_32x32b_x32(trow + (uint32_t)(32 * c), r);
                        ptx::tmem_wait_ld(r);
                        uint8_t *row = local + c * 4096 + lane * 128u;
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            *reinterpret_cast<uint4 *>(row + (((uint32_t)k ^ (lane & 7u)) * 16u)) =
                                make_uint4(r[4 * k], r[4 * k + 1], r[4 * k + 2], r[4 * k + 3]);
                        ptx::fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0)
                            ptx::bulk_copy_to_peer(dst + (uint32_t)c * 4096u, ptx::smem_addr(local + c * 4096), 4096u,
                                                   ptx::mapa_shared(csr_in(q, (uint32_t)c), owner));
                    }
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(acce_bar(acc));
                    if (tracing && lane == 0) tslot = trace_put(p, tslot, 3, t, (int)q + 4, t_unit, ptx::globaltimer_ns());
                    acc ^= 1;
                    if (acc == 0) acc_phase ^= 1u;
                    if (ok && !next_unit(t, t)) {
                        if (lane == 0) record_failure(kRoleEpilogue, t, abort_flag);
                        break;
                    }
                    continue;
                }
                if (lane == 0) {
                    // the bytes each chunk will receive, then the go-ahead to the senders
                    for (uint32_t c = 0; c < (uint32_t)(BN / 32); ++c)
                        ptx::mbar_arrive_expect_tx(csr_in(q, c), 4096u * (csplit - 1));
                    for (uint32_t s = 0; s < csplit; ++s)
                        if (s != crank) ptx::mbar_arrive_cluster(ptx::mapa_shared(csr_ready(q), s));
                }
                csr_base = ptx::smem_addr(stages) + qloc * part_bytes;
                csr_owner = true;
            }
            // A plain FP32 C stored by TMA: the owner writes each summed chunk
            // back into the first received slot (already in the 128-byte
            // swizzled box layout) and stores it from there, no staging buffer.
            const bool csr_direct = csr_owner && !fused && U.tma_store && box_cols == 32;
            if (csr_direct && csplit == 2) {
                // Two ranges: copy this warp's own accumulator into the ring
                // right away (after the received and the sent quarter-tiles),
                // so that while the peer's chunks arrive the sums need only
                // shared memory; Tensor Memory is handed back at once.
                const uint32_t per = 2u, part_bytes = 32u * (uint32_t)BN * 4u;
                uint8_t *own = stages + (2u * per + (q % per)) * part_bytes;
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t r[32];
                    ptx::tmem_ld_32x32b_x32(trow + (uint32_t)(32 * c), r);
                    ptx::tmem_wait_ld(r);
                    uint8_t *row = own + c * 4096 + lane * 128u;
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        *reinterpret_cast<uint4 *>(row + (((uint32_t)k ^ (lane & 7u)) * 16u)) =
                            make_uint4(r[4 * k], r[4 * k + 1], r[4 * k + 2], r[4 * k + 3]);
                }
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(acce_bar(acc));
                uint8_t *slot = stages + (size_t)(csr_base - ptx::smem_addr(stages));   // the peer's partial
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    const bool got = wait_bar<true>(csr_in(q, (uint32_t)c), 0u, abort_flag, p.timeout_ns);
                    if (!__all_sync(0xffffffffu, got)) {
                        if (lane == 0) record_failure(kRoleEpilogue, t, abort_flag);
                        ok = false;
                        break;
                    }
                    if (tracing) {
                        t_last_in = ptx::globaltimer_ns();
                        if (c == 0) t_first_in = t_last_in;
                    }
                    uint8_t *srow = slot + c * 4096 + lane * 128u;
                    const uint8_t *orow = own + c * 4096 + lane * 128u;
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const uint32_t off = ((uint32_t)k ^ (lane & 7u)) * 16u;
                        const float4 a = *reinterpret_cast<const float4 *>(orow + off);
                        const float4 b = *reinterpret_cast<const float4 *>(srow + off);
                        // K-range order: range 0 + range 1, whichever CTA holds which
                        *reinterpret_cast<float4 *>(srow + off) =
                            crank == 0 ? make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w)
                                       : make_float4(b.x + a.x, b.y + a.y, b.z + a.z, b.w + a.w);
                    }
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    const int col0 = n0 + 32 * c;
                    if (lane == 0 && m0 < U.M && col0 < U.N) {
                        ptx::tma_store_2d(U.mC, csr_base + (uint32_t)c * 4096u, col0, m0);
                        ptx::bulk_commit_group();
                        if (tracing) t_last_issue = ptx::globaltimer_ns();
                    }
                }
                if (tracing && lane == 0) {
                    const uint64_t t_end = ptx::globaltimer_ns();
                    tslot = trace_put(p, tslot, 3, t, (int)q, t_unit, t_end);
                    tslot = trace_put(p, tslot, 6, t, 0, t_unit, t_first_in);
                    tslot = trace_put(p, tslot, 6, t, 1, t_first_in, t_last_in);
                    tslot = trace_put(p, tslot, 6, t, 2, t_last_in, t_last_issue);
                }
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
                if (ok && !next_unit(t, t)) {
                    if (lane == 0) record_failure(kRoleEpilogue, t, abort_flag);
                    break;
                }
                continue;
            }
#pragma unroll 1
            for (int jb = 0; jb < ucols / box_cols; ++jb, ++nchunk) {
                uint8_t *buf = bufs + (nchunk & 1u) * kEpiBufBytes;
                const int col0 = n0 + box_cols * jb;
                const bool box_live = m0 < U.M && col0 < U.N;
                // The TMA store that last read this buffer (two boxes ago) must be done.
                if (nchunk >= 2 && !csr_direct) {
                    if (lane == 0) ptx::bulk_wait_group_read<1>();
                    __syncwarp();
                }
                // Residual (beta != 0): the old C box arrives by TMA in this buffer
                // and each thread rewrites its own row in place.
                if (reg_epi && need_old && box_live) {
                    const uint32_t bi = nchunk & 1u;
                    const uint32_t ob = oldc_bar(2 * (int)ew + (int)bi);
                    if (lane == 0) {
                        ptx::mbar_arrive_expect_tx(ob, (uint32_t)kEpiBufBytes);
                        ptx::tma_load_2d(ptx::smem_addr(buf), U.mC, ob, col0, m0);
                    }
                    const bool got = wait_bar<false>(ob, (old_phase >> bi) & 1u, abort_flag, p.timeout_ns);
                    old_phase ^= 1u << bi;
                    if (!__all_sync(0xffffffffu, got)) {
                        if (lane == 0) record_failure(kRoleEpilogue, t, abort_flag);
                        ok = false;
                        break;
                    }
                }
                uint8_t *row_base = buf + lane * 128u;
#pragma unroll 1
                for (int h = 0; h < box_cols / 32; ++h) {
                    uint32_t r[32];
                    ptx::tmem_ld_32x32b_x32(trow + (uint32_t)(box_cols * jb + 32 * h), r);
                    ptx::tmem_wait_ld(r);
                    if (csr_owner) {
                        // this quarter's K ranges summed in range order, this CTA's own at crank
                        const uint32_t per = 4u / csplit, part_bytes = 32u * (uint32_t)BN * 4u;
                        const uint32_t chunk = (uint32_t)((box_cols * jb + 32 * h) / 32);
                        const bool got = wait_bar<true>(csr_in(q, chunk), 0u, abort_flag, p.timeout_ns);
                        if (!__all_sync(0xffffffffu, got)) {
                            if (lane == 0) record_failure(kRoleEpilogue, t, abort_flag);
                            ok = false;
                            break;
                        }
                        if (tracing) {
                            t_last_in = ptx::globaltimer_ns();
                            if (chunk == 0) t_first_in = t_last_in;
                        }
                        const uint32_t row = csr_base + chunk * 4096u + lane * 128u;
                        float sum[32];
#pragma unroll 1
                        for (uint32_t s = 0; s < csplit; ++s) {
#pragma unroll
                            for (int k = 0; k < 8; ++k) {
                                float4 v;
                                if (s == crank) {
                                    v = make_float4(__uint_as_float(r[4 * k]), __uint_as_float(r[4 * k + 1]),
                                                    __uint_as_float(r[4 * k + 2]), __uint_as_float(r[4 * k + 3]));
                                } else {
                                    const uint32_t j = s < crank ? s : s - 1;
                                    v = ptx::ld_shared_v4f(row + j * per * part_bytes + (((uint32_t)k ^ (lane & 7u)) * 16u));
                                }
                                if (s == 0) {
                                    sum[4 * k] = v.x; sum[4 * k + 1] = v.y; sum[4 * k + 2] = v.z; sum[4 * k + 3] = v.w;
                                } else {
                                    sum[4 * k] += v.x; sum[4 * k + 1] += v.y; sum[4 * k + 2] += v.z; sum[4 * k + 3] += v.w;
                                }
                            }
                        }
#pragma unroll
                        for (int c = 0; c < 32; ++c) r[c] = __float_as_uint(sum[c]);
                        if (csr_direct) {
                            // the sum, in place of the first received partial
#pragma unroll
                            for (int k = 0; k < 8; ++k)
                                *reinterpret_cast<uint4 *>(stages + (row - ptx::smem_addr(stages)) +
                                                           (((uint32_t)k ^ (lane & 7u)) * 16u)) =
                                    make_uint4(r[4 * k], r[4 * k + 1], r[4 * k + 2], r[4 * k + 3]);
                        }
                    }
                    if (jb == ucols / box_cols - 1 && h == box_cols / 32 - 1) {
                        // The accumulator is fully in registers/shared: hand it back to the MMA.
                        ptx::tc_fence_before();
                        __syncwarp();
                        if (lane == 0) {
                            if (kPair) ptx::mbar_arrive_cluster(ptx::mapa_shared(acce_bar(acc), 0));
                            else ptx::mbar_arrive(acce_bar(acc));
                        }
                    }
                    if (reg_epi) {
                        // Row m0 + lane, columns cb .. cb + 31: lane c holds bias[cb + c].
                        const int cb = col0 + 32 * h;
                        const float bias_lane = epi_bias(e, cb + (int)lane, U.N);
                        // The old C of these 32 columns, read in 16-byte chunks (one
                        // chunk per lane per quarter-warp phase: conflict-free).
                        float old[32];
#pragma unroll
                        for (int c = 0; c < 32; ++c) old[c] = 0.f;
                        if (need_old) {
                            if (pack16) {
#pragma unroll
                                for (int k = 0; k < 4; ++k) {
                                    const uint4 v = *reinterpret_cast<const uint4 *>(
                                        row_base + (((uint32_t)(4 * h + k) ^ (lane & 7u)) * 16u));
                                    epi_unpack2(out, v.x, old[8 * k + 0], old[8 * k + 1]);
                                    epi_unpack2(out, v.y, old[8 * k + 2], old[8 * k + 3]);
                                    epi_unpack2(out, v.z, old[8 * k + 4], old[8 * k + 5]);
                                    epi_unpack2(out, v.w, old[8 * k + 6], old[8 * k + 7]);
                                }
                            } else {
#pragma unroll
                                for (int k = 0; k < 8; ++k) {
                                    const float4 v = *reinterpret_cast<const float4 *>(
                                        row_base + (((uint32_t)k ^ (lane & 7u)) * 16u));
                                    old[4 * k + 0] = v.x;
                                    old[4 * k + 1] = v.y;
                                    old[4 * k + 2] = v.z;
                                    old[4 * k + 3] = v.w;
                                }
                            }
                        }
                        float y[32];
#pragma unroll
                        for (int c = 0; c < 32; ++c)
                            y[c] = epi_value(e, __uint_as_float(r[c]), old[c],
                                             __shfl_sync(0xffffffffu, bias_lane, c));
                        if (pack16) {
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                uint4 v;
                                v.x = epi_pack2(out, y[8 * k + 0], y[8 * k + 1]);
                                v.y = epi_pack2(out, y[8 * k + 2], y[8 * k + 3]);
                                v.z = epi_pack2(out, y[8 * k + 4], y[8 * k + 5]);
                                v.w = epi_pack2(out, y[8 * k + 6], y[8 * k + 7]);
                                *reinterpret_cast<uint4 *>(row_base + (((uint32_t)(4 * h + k) ^ (lane & 7u)) * 16u)) = v;
                            }
                        } else {
#pragma unroll
                            for (int c = 0; c < 8; ++c)
                                *reinterpret_cast<float4 *>(row_base + (((uint32_t)c ^ (lane & 7u)) * 16u)) =
                                    make_float4(y[4 * c + 0], y[4 * c + 1], y[4 * c + 2], y[4 * c + 3]);
                        }
                    } else if (!csr_direct) {
                        // Row `lane`, 16-byte chunk c stored at position c ^ (row % 8): the
                        // 128-byte swizzle the TMA store expects, and conflict-free here.
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            *reinterpret_cast<float4 *>(row_base + (((uint32_t)c ^ (lane & 7u)) * 16u)) =
                                make_float4(__uint_as_float(r[4 * c + 0]), __uint_as_float(r[4 * c + 1]),
                                            __uint_as_float(r[4 * c + 2]), __uint_as_float(r[4 * c + 3]));
                    }
                }
                if (!ok) break;   // a cluster peer's partial never arrived (recorded above)
                if (use_tma) {
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        const uint32_t src =
                            csr_direct ? csr_base + (uint32_t)jb * 4096u : ptx::smem_addr(buf);   // box = chunk jb
                        if (to_slab) ptx::tma_store_3d(&tmW, src, 32 * jb, srow, slab);
                        else if (box_live) ptx::tma_store_2d(U.mC, src, col0, m0);
                        ptx::bulk_commit_group();
                        if (tracing) t_last_issue = ptx::globaltimer_ns();
                    }
                } else {
                    // C not addressable by TMA: lane = column, each row of the box
                    // leaves as one coalesced store; the old C (beta != 0) is
                    // loaded eight rows at a time ahead of their stores.
                    __syncwarp();
                    const int col = col0 + (int)lane;
                    const uint32_t cchunk = lane >> 2, cword = lane & 3u;
                    if (!fused) {
                        // The box's 32 rows: every shared load first, then the
                        // stores, with the row and column tests and the address
                        // arithmetic done once (the last round's epilogue runs
                        // exposed at the end of the launch).
                        const int nrows = min(32, U.M - m0);
                        const bool col_ok = col < U.N;
                        float *dst = static_cast<float *>(U.C) + (int64_t)m0 * U.ldc + col;
                        const uint8_t *src = buf + cword * 4u;
                        float v[32];
#pragma unroll
                        for (int rr = 0; rr < 32; ++rr)
                            v[rr] = *reinterpret_cast<const float *>(src + rr * 128 + ((cchunk ^ (uint32_t)(rr & 7)) * 16u));
                        if (col_ok) {
#pragma unroll
                            for (int rr = 0; rr < 32; ++rr) {
                                if (rr < nrows) *dst = v[rr];
                                dst += U.ldc;
                            }
                        }
                        __syncwarp();
                        continue;
                    }
                    const float bias = epi_bias(e, col, U.N);
#pragma unroll 1
                    for (int r0 = 0; r0 < 32; r0 += 8) {
                        float old[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            old[i] = (need_old && m0 + r0 + i < U.M && col < U.N)
                                         ? epi_load_old(U.C, (int64_t)(m0 + r0 + i) * U.ldc + col, out)
                                         : 0.f;
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int rr = r0 + i, grow = m0 + rr;
                            const float v = *reinterpret_cast<const float *>(
                                buf + rr * 128 + ((cchunk ^ (uint32_t)(rr & 7)) * 16u) + cword * 4u);
                            if (grow < U.M && col < U.N) {
                                const int64_t idx = (int64_t)grow * U.ldc + col;
                                if (fused) epi_store(U.C, idx, out, epi_value(e, v, old[i], bias));
                                else static_cast<float *>(U.C)[idx] = v;
                            }
                        }
                    }
                    __syncwarp();
                }
            }
            if (tracing && lane == 0) {
                const uint64_t t_end = ptx::globaltimer_ns();
                tslot = trace_put(p, tslot, 3, t, (int)q, t_unit, t_end);
                if (t_first_in) {
                    // owner of a cluster split: to the first partial chunk, to the last, to the last store
                    tslot = trace_put(p, tslot, 6, t, 0, t_unit, t_first_in);
                    tslot = trace_put(p, tslot, 6, t, 1, t_first_in, t_last_in);
                    tslot = trace_put(p, tslot, 6, t, 2, t_last_in, t_last_issue);
                }
            }
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
            if (ok && !next_unit(t, t)) {
                if (lane == 0) record_failure(kRoleEpilogue, t, abort_flag);
                break;
            }
        }
        // Before the CTA's shared memory goes away, its TMA stores must have
        // read it; their global writes complete on their own and are
        // visible once the grid has completed (which the next kernel on
        // the stream waits for in griddepcontrol.wait).
        if (lane == 0) ptx::bulk_wait_group_read<0>();
        if (tracing && lane == 0 && t_last_issue) tslot = trace_put(p, tslot, 6, -1, 3, t_last_issue, ptx::globaltimer_ns());
        __syncwarp();
    }

    // ------------------------------------------------------------ teardown
    // The split-K reduction (launched next, when tiles were split) may be
    // scheduled now; it waits for this grid's slab writes before reading them.
    if (p.tail_tiles > 0 && !csplit && threadIdx.x == 0) ptx::pdl_launch_dependents();
    ptx::tc_fence_before();
    // (a cluster split's peers stay until no CTA of the cluster touches another's shared memory)
    if (kPair || csplit) ptx::cluster_sync(); else __syncthreads();
    ptx::tc_fence_after();
    if (warp == 1) ptx::tmem_dealloc<CG>(tmem_base, Cf::TMEM_COLS);
    if (tracing && threadIdx.x == 0) tslot = trace_put(p, tslot, 4, -1, 0, t_start, ptx::globaltimer_ns());
}

// ------------------------------------------------------------------ host ---
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// Row-major matrix of `rows` x `cols` elements with a pitch of `ld` elements,
// tiled in boxes of box_cols x box_rows with a 128-byte swizzle (of 16-byte
// units unless `swizzle` says otherwise).
CUresult encode_2d(CUtensorMap *map, CUtensorMapDataType dt, int elem, const void *base, int64_t cols, int64_t rows,
                   int64_t ld, int box_cols, int box_rows,
                   CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
    auto enc = tensor_map_encoder();
    if (!enc) return CUDA_ERROR_NOT_SUPPORTED;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(ld * elem)};
    cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// FP32 slabs [count][rows][cols], dense, stored in 32 x 32 x 1 boxes with
// the 128-byte swizzle.
CUresult encode_3d_slabs(CUtensorMap *map, const void *base, int64_t cols, int64_t rows, int64_t count) {
    auto enc = tensor_map_encoder();
    if (!enc) return CUDA_ERROR_NOT_SUPPORTED;
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)count};
    cuuint64_t strides[2] = {(cuuint64_t)(cols * 4), (cuuint64_t)(rows * cols * 4)};
    cuuint32_t box[3] = {32, 32, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// Tensor maps of one GEMM's operands as variant <DT, CG, BN, BMODE> stages
// them: A in BK x 128-row boxes, B as stored (128-byte column chunks) or as the
// K-major copy, C (when it leaves through TMA) in 32-row boxes of 128 bytes:
// 32 FP32 columns, or 64 of a 16-bit output.
template <int DT, int CG, int BN, int BMODE>
CUresult encode_operands(int M, int N, int K, const void *A, int64_t lda, const void *B, int64_t ldb, void *C,
                         int64_t ldc, int out, bool tma_store, CUtensorMap *ta, CUtensorMap *tb, CUtensorMap *tc) {
    using Cf = TcCfg<DT, CG, BN, BMODE>;
    const CUtensorMapDataType dt = DT == kDtTF32   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : DT == kDtFP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                   : Cf::F8        ? CU_TENSOR_MAP_DATA_TYPE_UINT8     // bytes, moved as is
                                                   : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    std::memset(tc, 0, sizeof *tc);
    CUresult r = encode_2d(ta, dt, Cf::ELEM, A, K, M, lda, Cf::BK, kBM);
    if (r == CUDA_SUCCESS)
        r = Cf::BKM ? encode_2d(tb, dt, Cf::ELEM, B, K, N, ldb, Cf::BK, Cf::BN_CTA)   // B^T: N x K
                    : encode_2d(tb, dt, Cf::ELEM, B, N, K, ldb, Cf::CHUNK_COLS, Cf::BK,
                                Cf::B_ATOM32 ? CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B : CU_TENSOR_MAP_SWIZZLE_128B);
    if (r == CUDA_SUCCESS && tma_store) {
        if (out == GEMM_OUT_F32)
            r = encode_2d(tc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, C, N, M, ldc, 32, 32);
        else
            r = encode_2d(tc, out == GEMM_OUT_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                          2, C, N, M, ldc, 64, 32);
    }
    return r;
}

// Launches the kernel with the plan's grid (CTA pairs as clusters of two).
template <int DT, int CG, int BN, int BMODE>
int launch_kernel(const gemm_plan_t &plan, const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &tc,
                  const CUtensorMap &tw, const TcParams &p, cudaStream_t stream, char *err, size_t errlen) {
    using Cf = TcCfg<DT, CG, BN, BMODE>;
    auto kern = tc_gemm_kernel<DT, CG, BN, BMODE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cf::SMEM_BYTES);
    if (e != cudaSuccess) {
        std::snprintf(err, errlen, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
        return GEMM_ERR_CUDA;
    }
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3((unsigned)plan.grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = Cf::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned n_attr = 0;
    if (CG == 2 || p.csplit) {
        // a CTA pair, or the CTAs of one tile's K ranges
        attr[n_attr].id = cudaLaunchAttributeClusterDimension;
        attr[n_attr].val.clusterDim.x = CG == 2 ? 2 : (unsigned)p.csplit;
        attr[n_attr].val.clusterDim.y = 1;
        attr[n_attr].val.clusterDim.z = 1;
        ++n_attr;
    }
    if (options_snapshot().pdl != 1) {
        // may start while the previous kernel on the stream finishes (the
        // kernel waits for it before touching global memory)
        attr[n_attr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n_attr].val.programmaticStreamSerializationAllowed = 1;
        ++n_attr;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n_attr;
    e = cudaLaunchKernelEx(&cfg, kern, ta, tb, tc, tw, p);
    if (e != cudaSuccess) {
        std::snprintf(err, errlen, "tensor-core kernel launch: %s", cudaGetErrorString(e));
        return GEMM_ERR_CUDA;
    }
    return GEMM_OK;
}

TcParams base_params(const gemm_plan_t &plan, const EpiParams &epi, uint32_t timeout_ms) {
    TcParams p;
    std::memset(&p, 0, sizeof p);
    p.splits = 1;
    p.group_m = plan.group_m > 0 ? plan.group_m : 1;
    p.tma_store = plan.tma_store;
    p.debug_stall = options_snapshot().debug_stall_mma;
    p.epi = epi;
    p.groups = nullptr;
    p.sched = plan.sched;
    p.timeout_ns = (unsigned long long)timeout_ms * 1000000ull;
    const Options o = options_snapshot();
    if (o.trace_addr) {
        p.trace_count = reinterpret_cast<uint32_t *>((uintptr_t)o.trace_addr);
        p.trace = reinterpret_cast<gemm_trace_record_t *>((uintptr_t)o.trace_addr + 32);
        p.trace_cap = o.trace_records;
    }
    return p;
}

template <int DT, int CG, int BN, int BMODE>
int launch_variant(const gemm_plan_t &plan, int M, int N, int K, const void *A, int64_t lda, const void *B,
                   int64_t ldb, void *C, int64_t ldc, float *W, const EpiParams &epi, uint32_t timeout_ms,
                   cudaStream_t stream, char *err, size_t errlen) {
    using Cf = TcCfg<DT, CG, BN, BMODE>;
    CUtensorMap ta, tb, tc, tw;
    std::memset(&tw, 0, sizeof tw);
    CUresult r = encode_operands<DT, CG, BN, BMODE>(M, N, K, A, lda, B, ldb, C, ldc,
                                                    epi.active ? epi.out : GEMM_OUT_F32, plan.tma_store != 0, &ta,
                                                    &tb, &tc);
    if (r == CUDA_SUCCESS && plan.tail_tiles > 0 && !plan.cluster_split) {
        if (!W) {
            std::snprintf(err, errlen, "split tail without a workspace");
            return GEMM_ERR_INVALID_ARG;
        }
        r = encode_3d_slabs(&tw, W, BN, kBM * CG, (int64_t)plan.tail_tiles * plan.splits);
    }
    if (r != CUDA_SUCCESS) {
        std::snprintf(err, errlen, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
        return GEMM_ERR_CUDA;
    }
    TcParams p = base_params(plan, epi, timeout_ms);
    p.M = M;
    p.N = N;
    p.K = K;
    p.tiles_m = (M + kBM * CG - 1) / (kBM * CG);
    p.tiles_n = (N + BN - 1) / BN;
    p.num_tiles = p.tiles_m * p.tiles_n;
    p.num_kb = (K + Cf::BK - 1) / Cf::BK;
    p.tail_tiles = plan.tail_tiles;
    p.half_tiles = plan.tail_tiles > 0 ? 0 : plan.half_tiles;
    p.full_tiles = p.num_tiles - p.tail_tiles - p.half_tiles;
    p.splits = p.tail_tiles > 0 ? plan.splits : 1;
    p.kb_per_split = (p.num_kb + p.splits - 1) / p.splits;
    if (p.splits == 2 && plan.kb_split > 0) {
        // an uneven pair of K ranges: the first has kb_split k-blocks
        if (plan.kb_split < p.kb_per_split || plan.kb_split >= p.num_kb) {
            std::snprintf(err, errlen, "kb_split %d out of range for %d k-blocks", plan.kb_split, p.num_kb);
            return GEMM_ERR_INVALID_ARG;
        }
        p.kb_per_split = plan.kb_split;
    }
    p.num_units = p.full_tiles + p.tail_tiles * p.splits + 2 * p.half_tiles;
    p.C = C;
    p.ldc = ldc;
    p.ring = Cf::STAGES;
    if (plan.cluster_split) {
        if (CG != 1 || plan.cluster_split != p.splits || p.full_tiles != 0 || plan.sched != 0 ||
            plan.grid != p.num_units) {
            std::snprintf(err, errlen, "cluster split-K plan is inconsistent");
            return GEMM_ERR_INVALID_ARG;
        }
        p.csplit = plan.cluster_split;
        // One owner per tile (an uneven split, plain FP32 C stored by TMA): its
        // receive region, 4 lane quarters x 32 rows x BN FP32, ends where the
        // epilogue staging area ends and takes as many ring stages as needed
        // beyond that area.
        const int rx_bytes = 4 * 32 * BN * 4;
        const int over = rx_bytes > kEpiBytes ? rx_bytes - kEpiBytes : 0;
        const int ring = Cf::STAGES - (over + Cf::STAGE_BYTES - 1) / Cf::STAGE_BYTES;
        if (p.csplit == 2 && plan.kb_split > 0 && !epi.active && plan.tma_store && ring >= 3) {
            p.ring = ring;
            p.csr_rx = Cf::STAGES * Cf::STAGE_BYTES + kEpiBytes - rx_bytes;
        }
    }
    return launch_kernel<DT, CG, BN, BMODE>(plan, ta, tb, tc, tw, p, stream, err, errlen);
}

// One group's descriptor fields that depend on the variant (maps, tile counts).
template <int DT, int CG, int BN, int BMODE>
int encode_group_variant(GroupDesc *d, const void *A, int64_t lda, const void *B, int64_t ldb, void *C, int64_t ldc,
                         int out, int M, int N, int K, char *err, size_t errlen) {
    using Cf = TcCfg<DT, CG, BN, BMODE>;
    const CUresult r = encode_operands<DT, CG, BN, BMODE>(M, N, K, A, lda, B, ldb, C, ldc, out, d->tma_store != 0,
                                                          &d->tmA, &d->tmB, &d->tmC);
    if (r != CUDA_SUCCESS) {
        std::snprintf(err, errlen, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
        return GEMM_ERR_CUDA;
    }
    d->M = M;
    d->N = N;
    d->num_kb = (K + Cf::BK - 1) / Cf::BK;
    d->tiles_m = (M + kBM * CG - 1) / (kBM * CG);
    d->tiles_n = (N + BN - 1) / BN;
    return GEMM_OK;
}

template <int DT, int CG, int BN, int BMODE>
int launch_grouped_variant(const gemm_plan_t &plan, const GroupDesc *groups, int group_count, int num_units,
                           const EpiParams &epi, uint32_t timeout_ms, cudaStream_t stream, char *err, size_t errlen) {
    CUtensorMap unused;
    std::memset(&unused, 0, sizeof unused);
    TcParams p = base_params(plan, epi, timeout_ms);
    p.num_units = num_units;
    p.full_tiles = num_units;
    p.groups = groups;
    p.group_count = group_count;
    return launch_kernel<DT, CG, BN, BMODE>(plan, unused, unused, unused, unused, p, stream, err, errlen);
}

// A (dtype, CTA group, BN, B mode) combination is compiled only if it is legal:
// B read as stored needs every CTA's share of the tile width to be whole
// 128-byte column chunks.
template <int DT, int CG, int BN, int BMODE>
constexpr bool variant_ok() {
    return BMODE == kBKMajor || (BN / CG) % (128 / dt_elem(DT)) == 0;
}

enum VariantValue : int { kValSmem = 0, kValStages = 1, kValHalves = 2 };

template <int DT, int CG, int BN, int BMODE>
int variant_value(int what) {
    if constexpr (variant_ok<DT, CG, BN, BMODE>()) {
        using Cf = TcCfg<DT, CG, BN, BMODE>;
        return what == kValStages ? Cf::STAGES : what == kValHalves ? (Cf::HALVES ? 1 : 0) : Cf::SMEM_BYTES;
    } else {
        return 0;
    }
}


}  // namespace

// The (cta_group, BN) tiles compiled in.  Narrower pair tiles (256 x 128,
// 256 x 192) were measured and dropped: the MMA then re-reads A from shared
// memory twice as often per flop and runs 25-30% slower.
#define TC_VARIANTS(X) X(1, 64) X(1, 128) X(1, 256) X(2, 256)

static int tc_value(int dtype, int cta_group, int bn, int b_kmajor, int what) {
    const int mode = b_kmajor ? kBKMajor : kBNMajor;
#define X(cg, bn_)                                                                                   \
    if (cta_group == cg && bn == bn_) {                                                               \
        if (dtype == GEMM_TF32)                                                                       \
            return mode == kBKMajor ? variant_value<kDtTF32, cg, bn_, kBKMajor>(what)                \
                                    : variant_value<kDtTF32, cg, bn_, kBNMajor>(what);               \
        if (dtype == GEMM_FP16)                                                                       \
            return mode == kBKMajor ? variant_value<kDtFP16, cg, bn_, kBKMajor>(what)                \
                                    : variant_value<kDtFP16, cg, bn_, kBNMajor>(what);               \
        if (dtype == GEMM_E4M3)                                                                       \
            return mode == kBKMajor ? variant_value<kDtE4M3, cg, bn_, kBKMajor>(what)                \
                                    : variant_value<kDtE4M3, cg, bn_, kBNMajor>(what);               \
        if (dtype == GEMM_E5M2)                                                                       \
            return mode == kBKMajor ? variant_value<kDtE5M2, cg, bn_, kBKMajor>(what)                \
                                    : variant_value<kDtE5M2, cg, bn_, kBNMajor>(what);               \
        return mode == kBKMajor ? variant_value<kDtBF16, cg, bn_, kBKMajor>(what)                    \
                                : variant_value<kDtBF16, cg, bn_, kBNMajor>(what);                   \
    }
    TC_VARIANTS(X)
#undef X
    return 0;
}

int tc_smem_bytes(int dtype, int cta_group, int bn, int b_kmajor) {
    return tc_value(dtype, cta_group, bn, b_kmajor, kValSmem);
}

int tc_stages(int dtype, int cta_group, int bn, int b_kmajor) {
    return tc_value(dtype, cta_group, bn, b_kmajor, kValStages);
}

int tc_halves_ok(int dtype, int cta_group, int bn, int b_kmajor) {
    return tc_value(dtype, cta_group, bn, b_kmajor, kValHalves);
}

// Calls f(dt, cg, bn, mode) -- each an std::integral_constant -- for the
// variant the plan names; f returns a gemm_status_t.
template <class F>
static int dispatch_variant(const gemm_plan_t &plan, int dtype, F &&f, char *err, size_t errlen) {
    using std::integral_constant;
#define TC_CALL(DT_, MODE_, CG_, BN_) \
    f(integral_constant<int, DT_>{}, integral_constant<int, CG_>{}, integral_constant<int, BN_>{}, \
      integral_constant<int, MODE_>{})
#define X(cg, bn_)                                                                                       \
    if (plan.cta_group == cg && plan.bn == bn_) {                                                         \
        if (dtype == GEMM_TF32)                                                                           \
            return plan.b_kmajor == kBKMajor ? TC_CALL(kDtTF32, kBKMajor, cg, bn_)                        \
                                             : TC_CALL(kDtTF32, kBNMajor, cg, bn_);                       \
        if (dtype == GEMM_FP16)                                                                           \
            return plan.b_kmajor == kBKMajor ? TC_CALL(kDtFP16, kBKMajor, cg, bn_)                        \
                                             : TC_CALL(kDtFP16, kBNMajor, cg, bn_);                       \
        if (dtype == GEMM_E4M3)                                                                           \
            return plan.b_kmajor == kBKMajor ? TC_CALL(kDtE4M3, kBKMajor, cg, bn_)                        \
                                             : TC_CALL(kDtE4M3, kBNMajor, cg, bn_);                       \
        if (dtype == GEMM_E5M2)                                                                           \
            return plan.b_kmajor == kBKMajor ? TC_CALL(kDtE5M2, kBKMajor, cg, bn_)                        \
                                             : TC_CALL(kDtE5M2, kBNMajor, cg, bn_);                       \
        return plan.b_kmajor == kBKMajor ? TC_CALL(kDtBF16, kBKMajor, cg, bn_)                            \
                                         : TC_CALL(kDtBF16, kBNMajor, cg, bn_);                           \
    }
    do {
        TC_VARIANTS(X)
    } while (0);
#undef X
#undef TC_CALL
    std::snprintf(err, errlen, "no tensor-core variant for cta_group=%d bn=%d b_kmajor=%d", plan.cta_group, plan.bn,
                  plan.b_kmajor);
    return GEMM_ERR_UNSUPPORTED;
}

#define TC_IF_COMPILED(...)                                                                               \
    constexpr int DT = decltype(dt)::value, CG = decltype(cg)::value, BN = decltype(bn)::value,         \
                  MODE = decltype(mode)::value;                                                           \
    if constexpr (variant_ok<DT, CG, BN, MODE>()) {                                                       \
        __VA_ARGS__;                                                                                      \
    } else {                                                                                              \
        std::snprintf(err, errlen, "no tensor-core variant for cta_group=%d bn=%d b_kmajor=%d", CG, BN, MODE); \
        return GEMM_ERR_UNSUPPORTED;                                                                      \
    }

int tc_launch(const gemm_plan_t &plan, int dtype, int M, int N, int K, const void *A, int64_t lda, const void *B,
              int64_t ldb, void *C, int64_t ldc, float *W, const EpiParams &epi, uint32_t timeout_ms,
              cudaStream_t stream, char *err, size_t errlen) {
    return dispatch_variant(
        plan, dtype,
        [&](auto dt, auto cg, auto bn, auto mode) -> int {
            TC_IF_COMPILED(return launch_variant<DT, CG, BN, MODE>(plan, M, N, K, A, lda, B, ldb, C, ldc, W, epi,
                                                                   timeout_ms, stream, err, errlen))
        },
        err, errlen);
}

int tc_encode_group(const gemm_plan_t &plan, int dtype, GroupDesc *d, const void *A, int64_t lda, const void *B,
                    int64_t ldb, void *C, int64_t ldc, int out, int M, int N, int K, char *err, size_t errlen) {
    return dispatch_variant(
        plan, dtype,
        [&](auto dt, auto cg, auto bn, auto mode) -> int {
            TC_IF_COMPILED(return encode_group_variant<DT, CG, BN, MODE>(d, A, lda, B, ldb, C, ldc, out, M, N, K,
                                                                         err, errlen))
        },
        err, errlen);
}

int tc_launch_grouped(const gemm_plan_t &plan, int dtype, const GroupDesc *groups, int group_count, int num_units,
                      const EpiParams &epi, uint32_t timeout_ms, cudaStream_t stream, char *err, size_t errlen) {
    return dispatch_variant(
        plan, dtype,
        [&](auto dt, auto cg, auto bn, auto mode) -> int {
            TC_IF_COMPILED(return launch_grouped_variant<DT, CG, BN, MODE>(plan, groups, group_count, num_units, epi,
                                                                           timeout_ms, stream, err, errlen))
        },
        err, errlen);
}
#undef TC_IF_COMPILED

cudaError_t tc_read_and_clear_status(uint32_t words[4]) {
    cudaError_t e = cudaMemcpyFromSymbol(words, g_tc_status, sizeof(uint32_t) * 4);
    if (e != cudaSuccess) return e;
    static const uint32_t zero[4] = {0, 0, 0, 0};
    return cudaMemcpyToSymbol(g_tc_status, zero, sizeof zero);
}

int tc_max_active_clusters(int device) {
    (void)device;
    using Cf = TcCfg<kDtBF16, 2, 256, kBNMajor>;
    auto kern = tc_gemm_kernel<kDtBF16, 2, 256, kBNMajor>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cf::SMEM_BYTES) != cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = Cf::SMEM_BYTES;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) return 0;
    return n;
}

}  // namespace tcgemm
