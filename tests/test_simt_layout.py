"""Shared-memory access patterns of the SIMT kernel under the 32-bank model.

The bank model (pinned against the page's printed passes in test_analysis.py)
is applied to the index expressions of the kernel in
tiled_tensor_core_gemm_gb300/csrc/simt_fp32.cu: the padded, transposed A tile
[k][BM+4], the B tile [k][BN], and thread (ty, tx) = (tid / TX, tid % TX) with
its RM x RN 4-wide quads BM/RM rows and BN/RN columns apart.  No GPU.
"""
import pytest

from tiled_tensor_core_gemm_gb300.analysis import bank_passes, vector_bank_passes

BK = 8
# (BM, BN, BK, RM, RN) of the compiled variants 1..7
VARIANTS = [(128, 128, 8, 2, 2), (128, 128, 16, 2, 2), (128, 256, 8, 2, 4), (256, 128, 8, 4, 2),
            (64, 64, 8, 2, 2), (128, 256, 16, 2, 4), (64, 64, 16, 2, 2)]


def _threads(BM, BN, RM, RN):
    return (BM // (4 * RM)) * (BN // (4 * RN))


@pytest.mark.parametrize("BM,BN,bk,RM,RN", VARIANTS)
def test_transposed_A_stores(BM, BN, bk, RM, RN):
    """K step 8: conflict-free; K step 16: at most 2-way (four k-quads, two bank halves)."""
    threads = _threads(BM, BN, RM, RN)
    lds_a = BM + 4
    worst = 0
    for warp in range(threads // 32):
        for i in range(BM * bk // 4 // threads):
            for e in range(4):
                def addr(t):
                    f = warp * 32 + t + i * threads
                    r, kq = f // (bk // 4), f % (bk // 4)
                    return (4 * kq + e) * lds_a + r
                worst = max(worst, bank_passes(addr))
    assert worst == (1 if bk == 8 else 2)


@pytest.mark.parametrize("BM,BN", [(128, 128), (64, 64)])
def test_unpadded_transpose_would_conflict(BM, BN):
    # the reason for the +4 pad: with pitch BM the two k-quads share banks
    threads = (BM // 8) * (BN // 8)

    def addr(t):
        r, kq = t // (BK // 4), t % (BK // 4)
        return (4 * kq) * BM + r
    assert bank_passes(addr) == 2
    assert threads >= 32


@pytest.mark.parametrize("BM,BN,bk,RM,RN", VARIANTS)
def test_inner_loop_vector_reads_minimal(BM, BN, bk, RM, RN):
    TX = BN // (4 * RN)
    lds_a = BM + 4
    k = 5
    for warp in range(_threads(BM, BN, RM, RN) // 32):
        for qm in range(RM):
            def a_addr(t):
                ty = (warp * 32 + t) // TX
                return 4 * (k * lds_a + qm * (BM // RM) + ty * 4)
            # one pass per quarter-warp phase is the floor for 16-byte accesses
            assert vector_bank_passes(a_addr, 16) == 4
        for qn in range(RN):
            def b_addr(t):
                tx = (warp * 32 + t) % TX
                return 4 * (k * BN + qn * (BN // RN) + tx * 4)
            assert vector_bank_passes(b_addr, 16) == 4


def test_B_tile_vector_stores_minimal():
    BN, threads = 128, 256
    for warp in range(threads // 32):
        def addr(t):
            f = warp * 32 + t
            kr, c4 = f // (BN // 4), f % (BN // 4)
            return 4 * (kr * BN + 4 * c4)
        assert vector_bank_passes(addr, 16) == 4


def test_tc_epilogue_staging_swizzle_conflict_free():
    # tcgen05 epilogue: lane = row, 16-byte chunk c stored at c ^ (row % 8)
    for c in range(8):
        assert vector_bank_passes(lambda t: t * 128 + ((c ^ (t & 7)) * 16), 16) == 4
    # ordinary-store read-back: lane reads column `lane` of row rr
    for rr in range(32):
        assert bank_passes(lambda t: (rr * 128 + (((t >> 2) ^ (rr & 7)) * 16) + (t & 3) * 4) // 4) == 1
