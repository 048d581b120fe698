"""GPU parity of every path against the fp64 oracle, through the C ABI.

* exact: small-integer inputs (every product and partial sum an exact small
  integer) at tile-edge shapes must give bit-identical C on every path;
* the published workloads, every element of C: 256^3 / 1024^3 FP32, 1024^3
  TF32, 4096^3 FP32/TF32, 8192^3 BF16 and the four ragged BF16 shapes, in
  the launch configuration the benchmark uses (automatic plan); the FP16 and
  FP8 workloads on sampled rows;
* structure: identity, permutation, all-ones, K = 0, guard bands and padded
  leading dimensions, misaligned bases (operand pack), determinism, and every
  compiled tensor-core variant and epilogue.
"""
import numpy as np
import pytest
import torch

import tiled_tensor_core_gemm_gb300 as tg
from tiled_tensor_core_gemm_gb300 import build as tgbuild
from tiled_tensor_core_gemm_gb300.inputs import (C1_FP32_256, C2_FP32_1024, C2_TF32_1024, C3_FP32_4096,
                                                 C3_TF32_4096, C4_BF16_8192, C5_BF16_RAGGED, E4M3_4096, E4M3_8192,
                                                 E5M2_8192, FP16_4096, FP16_8192,
                                                 make_operands, workload_operands)

from gemm_check import TOL, error_ratio, oracle_full, oracle_rows, run_gemm, sample_rows

pytestmark = pytest.mark.gpu

DTYPES = ("fp32", "tf32", "bf16", "fp16", "e4m3", "e5m2")
FP8_TORCH = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}


@pytest.fixture(scope="module", autouse=True)
def lib():
    tgbuild.build()
    tg.load_library()
    for k in ("tc_bn", "tc_cta_group", "tc_group_m", "tc_max_ctas", "tc_tma_store", "simt_variant", "tc_b_major",
              "debug_stall_mma", "tc_splits", "tc_tail_splits", "tc_tail_halves", "tc_split_reduce", "tc_split_lead"):
        tg.gemm_set_option(k, 0)
    yield


def _exact(A, B, dtype, **kw):
    C = run_gemm(A, B, dtype, **kw)
    Cref, _ = oracle_full(A, B, dtype)
    assert np.array_equal(C.astype(np.float64), Cref), f"max |diff| {np.max(np.abs(C - Cref))}"


EDGE = [(1, 1, 1), (15, 17, 16), (16, 16, 16), (17, 15, 17), (63, 65, 64), (127, 129, 63), (128, 128, 128),
        (129, 257, 65), (255, 256, 257), (257, 513, 129), (300, 700, 1000), (384, 640, 192)]


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("shape", EDGE, ids=lambda s: "x".join(map(str, s)))
def test_small_integers_bit_exact(dtype, shape):
    M, N, K = shape
    A, B = make_operands(M, N, K, dtype, "ints", seed=11)
    _exact(A, B, dtype)


@pytest.mark.parametrize("dtype", DTYPES)
def test_identity_and_permutation(dtype):
    n, N = 300, 520
    tdt = {"bf16": torch.bfloat16, "fp16": torch.float16, **FP8_TORCH}.get(dtype, torch.float32)
    _, B = make_operands(n, N, n, dtype, "uniform", seed=12)
    if dtype == "tf32":
        B = B.to(torch.bfloat16).float()   # values the tensor cores read without loss
    eye32 = torch.eye(n, dtype=torch.float32)
    eye = eye32.to(tdt)
    C = run_gemm(eye, B, dtype)
    assert np.array_equal(C, B.float().numpy())
    perm = torch.randperm(n, generator=torch.Generator().manual_seed(3))
    P = eye32[perm].to(tdt)
    C = run_gemm(P, B, dtype)
    assert np.array_equal(C, B.float().numpy()[perm.numpy()])


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("K", [1, 64, 4099])
def test_all_ones_gives_K(dtype, K):
    A, B = make_operands(200, 333, K, dtype, "ones", seed=0)
    C = run_gemm(A, B, dtype)
    assert np.all(C == K)


@pytest.mark.parametrize("dtype", DTYPES)
def test_empty_sum_zero_fills(dtype):
    A, B = make_operands(37, 45, 0, dtype, "uniform", seed=0)
    C = run_gemm(A, B, dtype, ldc_pad=3)
    assert np.all(C == 0)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("shape,pads", [((200, 257, 128), (0, 7, 3)), ((200, 258, 128), (0, 6, 2)),
                                        ((200, 256, 130), (6, 0, 0)), ((200, 260, 132), (4, 4, 4))],
                         ids=["raggedN-ldc260", "raggedN-ldc260b", "raggedK-lda136", "ldc264"])
def test_ragged_edges_with_16_byte_pitches(dtype, shape, pads):
    """Pitches TMA can address (no pack) around ragged edges: NaN in the lda/ldb
    padding must not be read, and nothing may be stored into the ldc padding
    (a TMA store at a ragged right edge would write the whole 16-byte chunk)."""
    (M, N, K), (pa, pb, pc) = shape, pads
    A, B = make_operands(M, N, K, dtype, "ints", seed=15, lda_pad=pa, ldb_pad=pb)
    _exact(A, B, dtype, ldc_pad=pc)


@pytest.mark.parametrize("dtype", DTYPES)
def test_padded_leading_dimensions_and_guard_bands(dtype):
    # NaN in the lda/ldb padding: any read of it would poison C
    A, B = make_operands(200, 300, 130, dtype, "ints", seed=13, lda_pad=8, ldb_pad=8)
    _exact(A, B, dtype, ldc_pad=4)
    A, B = make_operands(199, 301, 129, dtype, "ints", seed=14, lda_pad=3, ldb_pad=5)
    _exact(A, B, dtype, ldc_pad=1)


@pytest.mark.parametrize("dtype", DTYPES)
def test_misaligned_bases(dtype):
    A, B = make_operands(256, 256, 256, dtype, "ints", seed=15)
    _exact(A, B, dtype, a_offset=1, b_offset=3)


@pytest.mark.parametrize("dtype", DTYPES)
def test_deterministic(dtype):
    A, B = make_operands(777, 1024, 1500, dtype, "normal", seed=16)
    C1 = run_gemm(A, B, dtype)
    C2 = run_gemm(A, B, dtype)
    assert np.array_equal(C1, C2)


TC_VARIANTS = [(1, 64), (1, 128), (1, 256), (2, 256)]


# (dtype, B staging): every input type reads B as stored (N-major; TF32 with
# the 32-byte-unit swizzle) or from the K-major transposed copy.
TC_OPERANDS = [("bf16", 2), ("bf16", 1), ("tf32", 2), ("tf32", 1), ("fp16", 2), ("fp16", 1), ("e4m3", 2),
               ("e4m3", 1), ("e5m2", 2), ("e5m2", 1)]


@pytest.mark.parametrize("operands", TC_OPERANDS, ids=lambda o: f"{o[0]}_{'kmajorB' if o[1] == 1 else 'nmajorB'}")
@pytest.mark.parametrize("variant", TC_VARIANTS, ids=lambda v: f"cg{v[0]}_bn{v[1]}")
@pytest.mark.parametrize("tma_store", (1, 2), ids=("tma_store", "plain_store"))
@pytest.mark.parametrize("shape", [(300, 700, 1000), (1024, 768, 333), (2048, 1536, 256)],
                         ids=lambda s: "x".join(map(str, s)))
def test_every_tensor_core_variant_exact(operands, variant, tma_store, shape):
    dtype, b_major = operands
    cg, bn = variant
    if dtype in FP8_TORCH and b_major == 2 and (bn // cg) % 128:
        pytest.skip("FP8 B as stored needs 128 columns per CTA (the planner takes the K-major copy)")
    M, N, K = shape
    A, B = make_operands(M, N, K, dtype, "ints", seed=17)
    try:
        tg.gemm_set_option("tc_cta_group", cg)
        tg.gemm_set_option("tc_bn", bn)
        tg.gemm_set_option("tc_tma_store", tma_store)
        tg.gemm_set_option("tc_b_major", b_major)
        _exact(A, B, dtype)
        # fewer persistent CTAs than tiles: several tiles per CTA, both accumulators
        tg.gemm_set_option("tc_max_ctas", 2 * cg)
        _exact(A, B, dtype)
    finally:
        for k in ("tc_cta_group", "tc_bn", "tc_tma_store", "tc_max_ctas", "tc_b_major"):
            tg.gemm_set_option(k, 0)


@pytest.mark.parametrize("dtype", ("bf16", "tf32", "fp16", "e4m3", "e5m2"))
@pytest.mark.parametrize("variant", TC_VARIANTS, ids=lambda v: f"cg{v[0]}_bn{v[1]}")
@pytest.mark.parametrize("splits", (2, 3, 7))
def test_split_k_exact(dtype, variant, splits):
    """Split-K: partial tiles in the workspace, summed in split order by the
    reduce kernel."""
    cg, bn = variant
    A, B = make_operands(300, 700, 1100, dtype, "ints", seed=20)
    try:
        tg.gemm_set_option("tc_split_reduce", 1)
        tg.gemm_set_option("tc_cta_group", cg)
        tg.gemm_set_option("tc_bn", bn)
        tg.gemm_set_option("tc_splits", splits)
        _exact(A, B, dtype)
        _exact(A, B, dtype, ldc_pad=3)          # C not TMA-addressable: the reduce writes it
        tg.gemm_set_option("tc_max_ctas", 3 * cg)
        _exact(A, B, dtype)
    finally:
        for k in ("tc_cta_group", "tc_bn", "tc_splits", "tc_max_ctas", "tc_b_major", "tc_split_reduce"):
            tg.gemm_set_option(k, 0)


@pytest.mark.parametrize("dtype", ("bf16", "tf32", "fp16", "e4m3"))
@pytest.mark.parametrize("bn", (64, 128, 256))
@pytest.mark.parametrize("shape", [(300, 700, 1100), (128, 2048, 4096), (40, 1000, 777)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("splits", (2, 4))
def test_split_k_summed_in_cluster_shared_memory_exact(dtype, bn, shape, splits):
    """Split-K with the K ranges of a tile on the CTAs of one cluster (2 or
    4), summed through distributed shared memory: exact on small integers,
    with TMA stores, with plain stores (C not TMA-addressable), and with rows
    of a lane quarter past M."""
    M, N, K = shape
    A, B = make_operands(M, N, K, dtype, "ints", seed=33)
    opts = {"tc_cta_group": 1, "tc_bn": bn, "tc_splits": splits, "tc_split_reduce": 1}
    try:
        for k, v in opts.items():
            tg.gemm_set_option(k, v)
        plan = tg.gemm_plan(M, N, K, tg.DTYPES[dtype], 0, K, 0, N, 0, N).as_dict()
        if plan["splits"] != splits or plan["tiles"] * splits > 152:
            pytest.skip(f"K cuts into {plan['splits']} non-empty ranges here, or too many CTAs")
        tg.gemm_set_option("tc_split_reduce", 2)
        plan = tg.gemm_plan(M, N, K, tg.DTYPES[dtype], 0, K, 0, N, 0, N).as_dict()
        assert plan["cluster_split"] == splits and plan["grid"] == splits * plan["tiles"], plan
        _exact(A, B, dtype)
        _exact(A, B, dtype, ldc_pad=3)
    finally:
        for k in opts:
            tg.gemm_set_option(k, 0)


@pytest.mark.parametrize("dtype", ("bf16", "tf32", "e4m3"))
@pytest.mark.parametrize("bn", (64, 128))
@pytest.mark.parametrize("lead", (51, 75, 95))
@pytest.mark.parametrize("shape", [(300, 700, 1100), (40, 1000, 777), (128, 2048, 4096)],
                         ids=lambda s: "x".join(map(str, s)))
def test_cluster_split_one_owner_exact(dtype, bn, lead, shape):
    """Two K ranges of uneven length on the CTAs of a cluster: CTA 0 runs the
    first range, receives CTA 1's partial past its ring and stores the whole
    tile.  Exact on small integers for first ranges from just over half to
    95% of the k-blocks, with rows of a lane quarter past M and ragged
    columns."""
    M, N, K = shape
    A, B = make_operands(M, N, K, dtype, "ints", seed=35)
    opts = {"tc_cta_group": 1, "tc_bn": bn, "tc_splits": 2, "tc_split_reduce": 2, "tc_split_lead": lead}
    try:
        for k, v in opts.items():
            tg.gemm_set_option(k, v)
        plan = tg.gemm_plan(M, N, K, tg.DTYPES[dtype], 0, K, 0, N, 0, N).as_dict()
        if plan["splits"] != 2 or plan["tiles"] * 2 > 152:
            pytest.skip("K does not cut into 2 ranges here, or too many CTAs")
        assert plan["cluster_split"] == 2 and plan["kb_split"] > 0, plan
        _exact(A, B, dtype)
    finally:
        for k in opts:
            tg.gemm_set_option(k, 0)


@pytest.mark.parametrize("dtype,lead", [("bf16", 0), ("bf16", 56), ("bf16", 80), ("tf32", 0)])
def test_cluster_split_k_gives_the_reduce_kernels_bits(dtype, lead):
    """On random data the cluster-summed split gives exactly the bits of the
    workspace-and-reduce-kernel split: both cut K at the same k-block (even,
    or the one-owner split) and add the K ranges' FP32 partials in range
    order."""
    M, N, K = 128, 8192, 8192 if dtype == "bf16" else 4096
    A, B = make_operands(M, N, K, dtype, "normal", seed=34)
    try:
        tg.gemm_set_option("tc_split_lead", lead)
        tg.gemm_set_option("tc_splits", 2)
        tg.gemm_set_option("tc_split_reduce", 1)
        assert tg.gemm_plan(M, N, K, tg.DTYPES[dtype], 0, K, 0, N, 0, N).cluster_split == 0
        C1 = run_gemm(A, B, dtype)
        tg.gemm_set_option("tc_split_reduce", 2)
        assert tg.gemm_plan(M, N, K, tg.DTYPES[dtype], 0, K, 0, N, 0, N).cluster_split == 2
        C2 = run_gemm(A, B, dtype)
        assert np.array_equal(C1, C2)
    finally:
        for k in ("tc_splits", "tc_split_reduce", "tc_split_lead"):
            tg.gemm_set_option(k, 0)


@pytest.mark.parametrize("dtype", ("bf16", "tf32"))
@pytest.mark.parametrize("cg,max_ctas,tail_splits", [(2, 28, 2), (2, 28, 3), (1, 20, 3), (1, 7, 2)])
def test_split_tail_exact(dtype, cg, max_ctas, tail_splits):
    """Whole tiles first, then the last round's tiles split in K (slabs + reduce)."""
    A, B = make_operands(2048, 1536, 1024, dtype, "ints", seed=25)
    try:
        tg.gemm_set_option("tc_cta_group", cg)
        tg.gemm_set_option("tc_bn", 256)
        tg.gemm_set_option("tc_max_ctas", max_ctas)
        tg.gemm_set_option("tc_tail_splits", tail_splits)
        from gemm_check import to_device
        plan = tg.gemm_plan(2048, 1536, 1024, tg.DTYPES[dtype], 0, 1024, 0, 1536, 0, 1536).as_dict()
        assert plan["tail_tiles"] > 0 and plan["splits"] > 1, plan
        _exact(A, B, dtype)
        _exact(A, B, dtype, ldc_pad=1)
    finally:
        for k in ("tc_cta_group", "tc_bn", "tc_max_ctas", "tc_tail_splits", "tc_tail_halves"):
            tg.gemm_set_option(k, 0)


HALF_CASES = [  # dtype, cta_group, BN, tc_b_major, CTAs
    ("bf16", 2, 256, 0, 40), ("fp16", 2, 256, 0, 40), ("tf32", 2, 256, 0, 40), ("tf32", 2, 256, 1, 40),
    ("tf32", 1, 128, 0, 44), ("bf16", 2, 256, 1, 40),
    ("e5m2", 2, 256, 1, 40), ("bf16", 1, 256, 0, 40), ("bf16", 1, 128, 0, 44), ("e4m3", 1, 256, 1, 40)]


@pytest.mark.parametrize("store", ("tma", "plain"))
@pytest.mark.parametrize("dtype,cg,bn,b_major,ctas", HALF_CASES, ids=lambda v: str(v))
def test_tail_halves_exact(dtype, cg, bn, b_major, ctas, store):
    """Whole tiles first, then the last round's tiles as two column halves each.
    1998 x 1440 in tiles of 256 (or 128) rows: the raster's last tiles are the
    right-hand column, whose tiles hold 160 (or 32) of their columns, so one
    half there is partly empty and, with BN = 128, the other has no column at
    all; the bottom row of tiles is ragged too."""
    M, N, K = 1998, 1440, 1024
    A, B = make_operands(M, N, K, dtype, "ints", seed=27)
    opts = {"tc_cta_group": cg, "tc_bn": bn, "tc_max_ctas": ctas, "tc_b_major": b_major,
            "tc_tma_store": 2 if store == "plain" else 0, "tc_tail_halves": 2}
    try:
        for k, v in opts.items():
            tg.gemm_set_option(k, v)
        plan = tg.gemm_plan(M, N, K, tg.DTYPES[dtype], 0, K, 0, N, 0, N).as_dict()
        assert plan["half_tiles"] > 0 and plan["tail_tiles"] == 0 and plan["tma_store"] == (store == "tma"), plan
        _exact(A, B, dtype)
    finally:
        for k in opts:
            tg.gemm_set_option(k, 0)


@pytest.mark.parametrize("K", (1, 65, 129))
@pytest.mark.parametrize("dtype,cg,bn,b_major,ctas", [("bf16", 2, 256, 0, 40), ("tf32", 2, 256, 0, 40), ("bf16", 1, 128, 0, 44)],
                         ids=lambda v: str(v))
def test_tail_halves_short_k(dtype, cg, bn, b_major, ctas, K):
    """Column halves whose K loop is one or two k-blocks (the ring never fills)."""
    M, N = 1998, 1440
    A, B = make_operands(M, N, K, dtype, "ints", seed=29)
    opts = {"tc_cta_group": cg, "tc_bn": bn, "tc_max_ctas": ctas, "tc_b_major": b_major, "tc_tail_halves": 2}
    try:
        for k, v in opts.items():
            tg.gemm_set_option(k, v)
        assert tg.gemm_plan(M, N, K, tg.DTYPES[dtype], 0, K, 0, N, 0, N).half_tiles > 0
        _exact(A, B, dtype)
    finally:
        for k in opts:
            tg.gemm_set_option(k, 0)


@pytest.mark.parametrize("dtype", ("bf16", "tf32"))
def test_tail_halves_equal_whole_tiles(dtype):
    """On random data a tile run as two column halves gives the same bits as
    the tile run whole: every output's sum takes the same K steps in the same
    order; only the MMA width differs."""
    A, B = make_operands(4096, 4096, 1024, dtype, "normal", seed=28)
    try:
        tg.gemm_set_option("tc_tail_halves", 2)
        assert tg.gemm_plan(4096, 4096, 1024, tg.DTYPES[dtype], 0, 1024, 0, 4096, 0, 4096).half_tiles == 28
        C1 = run_gemm(A, B, dtype)
        tg.gemm_set_option("tc_tail_halves", 1)
        tg.gemm_set_option("tc_tail_splits", 1)           # whole tiles (TF32 would split the tail in K)
        assert tg.gemm_plan(4096, 4096, 1024, tg.DTYPES[dtype], 0, 1024, 0, 4096, 0, 4096).tail_tiles == 0
        C2 = run_gemm(A, B, dtype)
    finally:
        tg.gemm_set_option("tc_tail_halves", 0)
        tg.gemm_set_option("tc_tail_splits", 0)
    assert np.array_equal(C1, C2)


def test_split_k_deterministic_on_random_data():
    A, B = make_operands(128, 4096, 8192, "bf16", "normal", seed=24)
    C1 = run_gemm(A, B, "bf16")
    C2 = run_gemm(A, B, "bf16")
    assert np.array_equal(C1, C2)
    # the split tail of a many-tile problem as well
    A, B = make_operands(4096, 4096, 2048, "tf32", "normal", seed=26)
    try:
        tg.gemm_set_option("tc_tail_splits", 2)
        C1 = run_gemm(A, B, "tf32")
        C2 = run_gemm(A, B, "tf32")
    finally:
        tg.gemm_set_option("tc_tail_splits", 0)
    assert np.array_equal(C1, C2)


@pytest.mark.parametrize("pdl", (0, 1), ids=("pdl_on", "pdl_off"))
@pytest.mark.parametrize("n", (512, 2048))
def test_back_to_back_launches_read_the_previous_output(n, pdl):
    """A tensor-core launch starts its set-up while the previous kernel on the
    stream finishes (programmatic dependent launch).  Here each step writes C1
    (BF16) and the next launch reads C1 as its A; the step after that
    overwrites C1 while that reader may still be finishing.  Small integers
    keep every value exact (|C1| <= 256, |D| < 2^24), so a read that came too
    early, or a write that came too soon, would show as a wrong D."""
    k1 = 4
    As = [make_operands(n, n, k1, "bf16", "ints", seed=140 + i)[0] for i in range(2)]
    B1 = make_operands(n, n, k1, "bf16", "ints", seed=142)[1]
    B2 = make_operands(n, n, n, "bf16", "ints", seed=143)[1]
    a_dev = [a.cuda() for a in As]
    b1, b2 = B1.cuda(), B2.cuda()
    c1 = torch.empty((n, n), dtype=torch.bfloat16, device="cuda")
    Ds = [torch.empty((n, n), dtype=torch.float32, device="cuda") for _ in range(8)]
    s = torch.cuda.current_stream().cuda_stream
    ep = tg.make_epilogue(out="bf16")
    assert tg.gemm_set_option("pdl", pdl) == tg.GEMM_OK
    try:
        for i, D in enumerate(Ds):
            a = a_dev[i % 2]
            rc = tg.gemm_run_ex(n, n, k1, tg.GEMM_BF16, a.data_ptr(), k1, b1.data_ptr(), n, c1.data_ptr(), n, ep, s)
            assert rc == tg.GEMM_OK, tg.gemm_last_error()
            rc = tg.gemm_run(n, n, n, tg.GEMM_BF16, c1.data_ptr(), n, b2.data_ptr(), n, D.data_ptr(), n, s)
            assert rc == tg.GEMM_OK, tg.gemm_last_error()
        assert tg.gemm_get_status(s) == tg.GEMM_OK, tg.gemm_last_error()
    finally:
        tg.gemm_set_option("pdl", 0)
    refs = []
    for a in As:
        c_ref, _ = oracle_full(a, B1, "bf16")
        refs.append(oracle_full(torch.from_numpy(c_ref).to(torch.bfloat16), B2, "bf16")[0])
    for i, D in enumerate(Ds):
        assert np.array_equal(D.cpu().double().numpy(), refs[i % 2]), f"step {i}"


def test_back_to_back_chain_through_the_cluster_split():
    """Each step: C1 = A_i . B1 through split-K summed in cluster shared
    memory (its owners' TMA stores are the last writes of that launch), then
    D = C1 . B2 reads C1 as its A (TF32).  The next step overwrites C1 while
    that reader may still be finishing.  Entries in {-1, 0, 1} keep every
    value exact (|C1| <= 512, |D| < 2^24)."""
    M, N1, K1, N2 = 128, 2048, 512, 256
    As = [make_operands(M, N1, K1, "bf16", "ints", seed=160 + i, lo_hi=1)[0] for i in range(2)]
    B1 = make_operands(M, N1, K1, "bf16", "ints", seed=162, lo_hi=1)[1]
    B2 = make_operands(N1, N2, N1, "tf32", "ints", seed=163, lo_hi=1)[1]
    a_dev = [a.cuda() for a in As]
    b1, b2 = B1.cuda(), B2.cuda()
    c1 = torch.empty((M, N1), dtype=torch.float32, device="cuda")
    Ds = [torch.empty((M, N2), dtype=torch.float32, device="cuda") for _ in range(8)]
    s = torch.cuda.current_stream().cuda_stream
    try:
        tg.gemm_set_option("tc_splits", 2)
        assert tg.gemm_plan(M, N1, K1, tg.GEMM_BF16, 0, K1, 0, N1, 0, N1).cluster_split == 2
        for i, D in enumerate(Ds):
            a = a_dev[i % 2]
            rc = tg.gemm_run(M, N1, K1, tg.GEMM_BF16, a.data_ptr(), K1, b1.data_ptr(), N1, c1.data_ptr(), N1, s)
            assert rc == tg.GEMM_OK, tg.gemm_last_error()
            rc = tg.gemm_run(M, N2, N1, tg.GEMM_TF32, c1.data_ptr(), N1, b2.data_ptr(), N2, D.data_ptr(), N2, s)
            assert rc == tg.GEMM_OK, tg.gemm_last_error()
        assert tg.gemm_get_status(s) == tg.GEMM_OK, tg.gemm_last_error()
    finally:
        tg.gemm_set_option("tc_splits", 0)
    refs = []
    for a in As:
        c_ref, _ = oracle_full(a, B1, "bf16")
        refs.append(oracle_full(torch.from_numpy(c_ref.astype(np.float32)), B2, "tf32")[0])
    for i, D in enumerate(Ds):
        assert np.array_equal(D.cpu().numpy().astype(np.float64), refs[i % 2]), i


@pytest.mark.parametrize("case", ("packed", "fp32"))
def test_back_to_back_chain_through_packs_and_simt(case):
    """The same chain where every kernel of the library takes part: with
    leading dimensions the TMA cannot address, the first GEMM of each step
    runs after two pack kernels; in FP32 both GEMMs are the SIMT kernel.
    Each of them may start while the one before it finishes, and must still
    read only finished data."""
    n, k1 = 600, 4
    dtype = "fp32" if case == "fp32" else "bf16"
    pad = 1 if case == "packed" else 0
    As = [make_operands(n, n, k1, dtype, "ints", seed=150 + i)[0] for i in range(2)]
    B1 = make_operands(n, n, k1, dtype, "ints", seed=152)[1]
    B2 = make_operands(n, n, n, dtype, "ints", seed=153)[1]

    def padded(t, ld):
        buf = torch.zeros((t.shape[0], ld), dtype=t.dtype, device="cuda")
        buf[:, :t.shape[1]] = t.cuda()
        return buf

    a_dev = [padded(a, k1 + pad) for a in As]
    b1, b2 = padded(B1, n + pad), B2.cuda()
    c1 = torch.empty((n, n), dtype=torch.float32 if case == "fp32" else torch.bfloat16, device="cuda")
    Ds = [torch.empty((n, n), dtype=torch.float32, device="cuda") for _ in range(8)]
    s = torch.cuda.current_stream().cuda_stream
    code = tg.DTYPES[dtype]
    ep = tg.make_epilogue(out="f32" if case == "fp32" else "bf16")
    if case == "packed":
        plan = tg.gemm_plan(n, n, k1, code, a_dev[0].data_ptr(), k1 + pad, b1.data_ptr(), n + pad, c1.data_ptr(), n)
        assert plan.pack_a and plan.pack_b
    for i, D in enumerate(Ds):
        a = a_dev[i % 2]
        rc = tg.gemm_run_ex(n, n, k1, code, a.data_ptr(), k1 + pad, b1.data_ptr(), n + pad, c1.data_ptr(), n, ep, s)
        assert rc == tg.GEMM_OK, tg.gemm_last_error()
        rc = tg.gemm_run(n, n, n, code, c1.data_ptr(), n, b2.data_ptr(), n, D.data_ptr(), n, s)
        assert rc == tg.GEMM_OK, tg.gemm_last_error()
    assert tg.gemm_get_status(s) == tg.GEMM_OK, tg.gemm_last_error()
    refs = []
    for a in As:
        c_ref, _ = oracle_full(a, B1, dtype)
        c_in = torch.from_numpy(c_ref).float()
        refs.append(oracle_full(c_in if case == "fp32" else c_in.to(torch.bfloat16), B2, dtype)[0])
    for i, D in enumerate(Ds):
        assert np.array_equal(D.cpu().double().numpy(), refs[i % 2]), f"step {i}"


@pytest.mark.parametrize("splits", (0, 2, 3, 8))
@pytest.mark.parametrize("shape", [(513, 389, 1027), (256, 256, 256), (1, 1000, 17), (1000, 7, 1000), (300, 520, 64),
                                   (200, 300, 65), (130, 129, 100), (64, 64, 257)],
                         ids=lambda s: "x".join(map(str, s)))
def test_simt_split_k_exact(shape, splits):
    """FP32 K cut into ranges (automatic, or forced), partials added in order by
    a second kernel: small integers stay exact; the result is the same run to run."""
    M, N, K = shape
    A, B = make_operands(M, N, K, "fp32", "ints", seed=170)
    try:
        tg.gemm_set_option("simt_splits", splits)
        _exact(A, B, "fp32")
        _exact(A, B, "fp32", ldc_pad=3)
        An, Bn = make_operands(M, N, K, "fp32", "normal", seed=171)
        assert np.array_equal(run_gemm(An, Bn, "fp32"), run_gemm(An, Bn, "fp32"))
    finally:
        tg.gemm_set_option("simt_splits", 0)


@pytest.mark.parametrize("variant", (1, 2, 3, 4, 5, 6, 7, 8, 9))
@pytest.mark.parametrize("shape", [(513, 389, 1027), (300, 520, 64), (1, 1000, 17)], ids=lambda s: "x".join(map(str, s)))
def test_simt_variants_exact(variant, shape):
    M, N, K = shape
    A, B = make_operands(M, N, K, "fp32", "ints", seed=18)
    try:
        tg.gemm_set_option("simt_variant", variant)
        _exact(A, B, "fp32")
        _exact(A, B, "fp32", a_offset=1, ldc_pad=1)   # scalar (non-vector) loads and stores
    finally:
        tg.gemm_set_option("simt_variant", 0)


# ------------------------------------------------------- published workloads ---
@pytest.mark.parametrize("w", [C1_FP32_256, C2_FP32_1024, C2_TF32_1024, C5_BF16_RAGGED[0]], ids=lambda w: w.name)
def test_workload_full(w):
    A, B = workload_operands(w)
    C = run_gemm(A, B, w.dtype)
    Cref, D = oracle_full(A, B, w.dtype)
    r = error_ratio(C, Cref, D)
    assert r <= TOL[w.dtype], r


# The oracle's C and D of a full-size workload, kept for the process: the FP32
# and TF32 4096^3 workloads share their inputs (and so one oracle run).
_ORACLE_CACHE = {}


def _oracle_of(w):
    kind = "f32" if w.dtype in ("fp32", "tf32") else w.dtype
    key = (w.M, w.N, w.K, kind, w.dist, w.seed)
    if key not in _ORACLE_CACHE:
        _ORACLE_CACHE.clear()          # one full-size product held at a time (8192^3: 1 GiB of C and D)
        A, B = workload_operands(w)
        _ORACLE_CACHE[key] = oracle_full(A, B, w.dtype)
    return _ORACLE_CACHE[key]


@pytest.mark.parametrize("w", [C3_FP32_4096, C3_TF32_4096, C4_BF16_8192] + list(C5_BF16_RAGGED[1:]),
                         ids=lambda w: w.name)
def test_workload_full_size_every_element(w):
    """The published full-size workloads, every element of C against the
    oracle, in the launch configuration the benchmark times (automatic plan)."""
    A, B = workload_operands(w)
    C = run_gemm(A, B, w.dtype)
    Cref, D = _oracle_of(w)
    r = error_ratio(C, Cref, D)
    assert r <= TOL[w.dtype], r


@pytest.mark.parametrize("w", [FP16_4096, FP16_8192, E4M3_4096, E4M3_8192, E5M2_8192], ids=lambda w: w.name)
def test_workload_sampled_rows(w):
    A, B = workload_operands(w)
    C = run_gemm(A, B, w.dtype)
    assert np.all(np.isfinite(C))
    rows = sample_rows(w.M, extra=8, seed=w.seed)
    Cref, D = oracle_rows(A, B, w.dtype, rows)
    r = error_ratio(C[rows], Cref, D)
    assert r <= TOL[w.dtype], r


# ------------------------------------------------------------ bounded waits ---
@pytest.mark.parametrize("cta_group", (1, 2))
def test_expired_wait_reports_timeout_and_context_survives(cta_group):
    """The MMA thread waits on an mbarrier nothing arrives at; the wait expires
    after wait_timeout_ms, the kernel records GEMM_ERR_TIMEOUT and returns, and
    the next GEMM on the same context is exact."""
    A, B = make_operands(512, 768, 320, "bf16", "ints", seed=19)
    stream = torch.cuda.current_stream().cuda_stream
    try:
        tg.gemm_set_option("tc_cta_group", cta_group)
        tg.gemm_set_option("wait_timeout_ms", 200)
        tg.gemm_set_option("debug_stall_mma", 1)
        from gemm_check import to_device
        a_keep, a_ptr, lda = to_device(A)
        b_keep, b_ptr, ldb = to_device(B)
        C = torch.empty((512, 768), dtype=torch.float32, device="cuda")
        rc = tg.gemm_run(512, 768, 320, tg.GEMM_BF16, a_ptr, lda, b_ptr, ldb, C.data_ptr(), 768, stream)
        assert rc == tg.GEMM_OK, tg.gemm_last_error()
        st = tg.gemm_get_status(stream)
        assert st == tg.GEMM_ERR_TIMEOUT, (st, tg.gemm_last_error())
        assert "role=mma" in tg.gemm_last_error()
        assert tg.gemm_get_status(stream) == tg.GEMM_OK   # the status word was cleared
        tg.gemm_set_option("debug_stall_mma", 0)
        _exact(A, B, "bf16")
    finally:
        tg.gemm_set_option("debug_stall_mma", 0)
        tg.gemm_set_option("wait_timeout_ms", 2000)
        tg.gemm_set_option("tc_cta_group", 0)
