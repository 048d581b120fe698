"""The C ABI without a GPU: the library loads, exports what include/gemm.h
declares, rejects bad arguments before any CUDA call, and plans on the host."""
import ctypes
import os
import re
import subprocess

import pytest

import tiled_tensor_core_gemm_gb300 as tg
from tiled_tensor_core_gemm_gb300 import build as tgbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    tgbuild.build()
    tg.load_library()


def _declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"GEMM_API\s+[\w\s\*]+?\b(gemm_\w+)\s*\(", src))
    return names


def test_exports_every_declared_symbol():
    declared = _declared_symbols()
    assert {"gemm_run", "gemm_last_error", "gemm_get_status", "gemm_set_option", "gemm_get_option",
            "gemm_plan", "gemm_version"} <= declared
    out = subprocess.run(["nm", "-D", "--defined-only", tg.library_path()], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT (gemm_\w+)", out))
    assert declared <= exported, declared - exported
    assert set(tg.EXPORTED) <= exported


def test_built_for_sm_103a_only():
    assert tgbuild.GENCODE == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_version():
    assert tg.gemm_version() == 10000


@pytest.mark.parametrize("args,frag", [
    ((-1, 4, 4, tg.GEMM_FP32, 16, 4, 16, 4, 64, 4), "negative"),
    ((4, 4, 4, 7, 16, 4, 16, 4, 64, 4), "dtype"),
    ((4, 4, 8, tg.GEMM_FP32, 16, 4, 16, 4, 64, 4), "leading dimension"),
    ((4, 8, 4, tg.GEMM_BF16, 16, 4, 16, 8, 64, 4), "leading dimension"),
    ((4, 4, 4, tg.GEMM_FP32, 0, 4, 16, 4, 64, 4), "NULL"),
    ((4, 4, 4, tg.GEMM_FP32, 16, 4, 16, 4, 0, 4), "NULL"),
    ((1 << 31, 4, 4, tg.GEMM_FP32, 16, 4, 16, 4, 64, 4), "2^31"),
])
def test_invalid_arguments_rejected_before_cuda(args, frag):
    rc = tg.gemm_run(*args, 0)
    assert rc == tg.GEMM_ERR_INVALID_ARG
    assert frag in tg.gemm_last_error()


def test_overlap_rejected():
    # C starts inside A's footprint
    rc = tg.gemm_run(8, 8, 8, tg.GEMM_FP32, 4096, 8, 1 << 20, 8, 4096 + 64, 8, 0)
    assert rc == tg.GEMM_ERR_INVALID_ARG and "overlap" in tg.gemm_last_error()


def test_empty_output_is_noop_without_cuda():
    assert tg.gemm_run(0, 5, 3, tg.GEMM_BF16, 0, 3, 0, 5, 0, 5, 0) == tg.GEMM_OK
    assert tg.gemm_run(5, 0, 3, tg.GEMM_FP32, 0, 3, 0, 1, 0, 1, 0) == tg.GEMM_OK


def test_options_roundtrip_and_validation():
    assert tg.gemm_set_option("tc_bn", 128) == tg.GEMM_OK and tg.gemm_get_option("tc_bn") == 128
    assert tg.gemm_set_option("tc_bn", 0) == tg.GEMM_OK
    assert tg.gemm_set_option("tc_bn", 96) == tg.GEMM_ERR_INVALID_ARG
    assert tg.gemm_set_option("tc_bn", 192) == tg.GEMM_ERR_INVALID_ARG
    assert tg.gemm_set_option("no_such_key", 1) == tg.GEMM_ERR_INVALID_ARG
    assert tg.gemm_get_option("no_such_key") == -1
    assert tg.gemm_get_option("wait_timeout_ms") == 2000
    assert tg.gemm_get_option("debug_stall_mma") == 0
    assert tg.gemm_set_option("debug_stall_mma", 2) == tg.GEMM_ERR_INVALID_ARG
    assert tg.gemm_get_option("tc_sched") == 0
    assert tg.gemm_set_option("tc_sched", 3) == tg.GEMM_ERR_INVALID_ARG


def test_every_documented_option_is_implemented_and_no_other():
    """The option keys the header documents (each at the head of a line in
    the gemm_set_option comment, plus "trace_records", described with
    "trace_addr") are exactly the keys gemm_get_option answers and
    gemm_api.cu reads."""
    import re
    header = open(os.path.join(ROOT, "include", "gemm.h")).read()
    documented = set(re.findall(r'^ \*   "([a-z_0-9]+)"', header, re.M)) | {"trace_records"}
    api = open(os.path.join(ROOT, "tiled_tensor_core_gemm_gb300", "csrc", "gemm_api.cu")).read()
    implemented = set(re.findall(r'if \(!std::strcmp\(key, "([a-z_0-9]+)"\)\) return o\.', api))
    assert documented == implemented, (documented ^ implemented)
    for key in documented:
        assert tg.gemm_get_option(key) != -1, key
    assert tg.gemm_get_option("tc_bn_x") == -1


def test_plan_dynamic_schedule_launches_one_cluster_per_unit():
    try:
        assert tg.gemm_set_option("tc_sched", 2) == tg.GEMM_OK
        p = _plan(8192, 8192, 8192, tg.GEMM_BF16)
        assert p["sched"] == 1 and p["cta_group"] == 2 and p["grid"] == 2 * p["tiles"] == 2048
        # column halves are units too: 256 tiles, the last 28 as two halves each
        h = _plan(4096, 4096, 4096, tg.GEMM_BF16)
        assert h["half_tiles"] == 28 and h["grid"] == 2 * (256 + 28)
        q = _plan(128, 8192, 8192, tg.GEMM_BF16)          # split-K units count too
        assert q["grid"] == q["tiles"] * q["splits"]
    finally:
        tg.gemm_set_option("tc_sched", 0)
    assert _plan(8192, 8192, 8192, tg.GEMM_BF16)["sched"] == 0


def _plan(M, N, K, dt, lda=None, ldb=None, ldc=None, a=0, b=0, c=0, sms=152):
    return tg.gemm_plan(M, N, K, dt, a, lda or K, b, ldb or N, c, ldc or N, sms).as_dict()


def test_plan_8192_bf16_uses_cta_pairs_full_machine():
    p = _plan(8192, 8192, 8192, tg.GEMM_BF16)
    assert p["path"] == 1 and p["cta_group"] == 2 and p["bn"] == 256 and p["bk"] == 64
    assert p["tiles"] == 32 * 32 and p["grid"] == 152
    assert not p["pack_a"] and not p["pack_b"] and p["tma_store"]
    assert p["stages"] >= 4 and p["smem_bytes"] <= 232448


def test_plan_tf32_and_fp32_4096():
    p = _plan(4096, 4096, 4096, tg.GEMM_TF32)
    assert p["path"] == 1 and p["bk"] == 32 and p["b_kmajor"] == 0 and p["pack_b"] == 0   # B read as stored
    assert _plan(4096, 4096, 4096, tg.GEMM_BF16)["b_kmajor"] == 0
    # a row pitch that is not a multiple of 16 bytes is packed, not transposed
    r = _plan(512, 1023, 512, tg.GEMM_TF32)
    assert r["b_kmajor"] == 0 and r["pack_b"] == 1
    s = _plan(4096, 4096, 4096, tg.GEMM_FP32)
    assert s["path"] == 0 and s["bm"] == 64 and s["bn"] == 128 and s["bk"] == 16 and s["vec"] == 1
    assert s["grid"] == 64 * 32


def test_plan_fp32_uses_64x128_tiles_at_every_size():
    for n in (256, 1024, 4096):
        p = _plan(n, n, n, tg.GEMM_FP32)
        assert (p["bm"], p["bn"], p["bk"]) == (64, 128, 16), p


def test_plan_fp32_splits_k_when_tiles_are_few():
    # target 6 x 152 blocks: 1024^3 has 128 tiles -> 8 K ranges; 256^3 8 tiles,
    # capped at 8; 2048^3 512 tiles -> 2; 4096^3 fills the machine
    assert _plan(1024, 1024, 1024, tg.GEMM_FP32)["splits"] == 8
    assert _plan(1024, 1024, 1024, tg.GEMM_FP32)["grid"] == 1024
    assert _plan(256, 256, 256, tg.GEMM_FP32)["splits"] == 8
    assert _plan(2048, 2048, 2048, tg.GEMM_FP32)["splits"] == 2
    assert _plan(4096, 4096, 4096, tg.GEMM_FP32)["splits"] == 1
    assert _plan(1000, 1000, 100, tg.GEMM_FP32)["splits"] == 3          # ranges of at least 32
    assert _plan(1000, 1000, 50, tg.GEMM_FP32)["splits"] == 1           # K too short
    assert _plan(513, 389, 1027, tg.GEMM_FP32)["splits"] == 8           # capped at 8
    try:
        assert tg.gemm_set_option("simt_splits", 1) == 0
        assert _plan(1024, 1024, 1024, tg.GEMM_FP32)["splits"] == 1
        assert tg.gemm_set_option("simt_splits", 3) == 0
        assert _plan(4096, 4096, 4096, tg.GEMM_FP32)["splits"] == 3
        assert _plan(64, 64, 16, tg.GEMM_FP32)["splits"] == 1           # never more ranges than K steps
    finally:
        tg.gemm_set_option("simt_splits", 0)
    assert tg.gemm_set_option("simt_splits", 9) == tg.GEMM_ERR_INVALID_ARG


def test_plan_ragged_packs_and_plain_epilogue():
    p = _plan(4097, 4095, 4099, tg.GEMM_BF16)
    assert p["pack_a"] and p["pack_b"] and not p["tma_store"]
    q = _plan(1000, 1000, 1000, tg.GEMM_BF16)   # 2000-byte rows are 16-byte multiples
    assert not q["pack_a"] and not q["pack_b"] and q["tma_store"]


def test_plan_tma_store_needs_whole_16_byte_rows():
    # A TMA store at a ragged right edge writes the whole 16-byte chunk holding
    # column N - 1, so a padded ldc with N * 4 not a multiple of 16 stores plainly.
    assert not _plan(200, 257, 128, tg.GEMM_BF16, ldc=260)["tma_store"]
    assert not _plan(200, 258, 128, tg.GEMM_BF16, ldc=260)["tma_store"]
    assert _plan(200, 260, 128, tg.GEMM_BF16, ldc=264)["tma_store"]


def test_plan_fp8():
    p = _plan(8192, 8192, 8192, tg.GEMM_E4M3)
    assert p["path"] == 1 and p["cta_group"] == 2 and p["bn"] == 256 and p["bk"] == 128
    assert not p["b_kmajor"] and not p["pack_a"] and not p["pack_b"]     # B read as stored
    # a narrow tile (64 columns per CTA) reads B from the K-major copy instead
    q = _plan(128, 8192, 256, tg.GEMM_E5M2)
    assert q["bn"] == 64 and q["b_kmajor"] == 1
    # 8-bit rows need a pitch that is a multiple of 16 elements for TMA (B here
    # goes through the K-major copy, whose pitch is rounded up anyway)
    r = _plan(1000, 1000, 1000, tg.GEMM_E4M3)
    assert r["pack_a"] and r["b_kmajor"] and not r["pack_b"]
    s = _plan(2000, 3000, 1000, tg.GEMM_E4M3)
    assert s["bn"] == 256 and s["pack_a"] and s["pack_b"] and not s["b_kmajor"]
    try:
        tg.gemm_set_option("tc_b_major", 2)
        with pytest.raises(tg.GemmError):
            _plan(128, 8192, 256, tg.GEMM_E5M2)
    finally:
        tg.gemm_set_option("tc_b_major", 0)


def test_plan_misaligned_base_packs():
    p = _plan(256, 256, 256, tg.GEMM_BF16, a=2)
    assert p["pack_a"] and not p["pack_b"]
    s = _plan(256, 256, 256, tg.GEMM_FP32, a=4)
    assert s["vec"] == 0


def test_plan_low_tile_count_splits_k():
    # 32 tiles of 128x256 for 152 SMs and 128 k-blocks: 4 K ranges per tile
    p = _plan(1024, 2048, 8192, tg.GEMM_BF16)
    assert p["cta_group"] == 1 and p["bn"] == 256 and p["splits"] == 2 and p["grid"] == 128
    assert p["tma_store"] == 1 and p["tail_tiles"] == 64        # every tile is split
    # short K: no split, narrow tiles instead
    q = _plan(128, 8192, 256, tg.GEMM_BF16)
    assert q["splits"] == 1 and q["bn"] == 64
    # small problems never split (the reduce would cost more than it saves)
    assert _plan(1000, 1000, 1000, tg.GEMM_BF16)["splits"] == 1


@pytest.mark.parametrize("M,N,K,bn,splits", [
    # B streams from HBM past at most 256 rows of A: 128-column tiles, K split to fill the SMs
    (128, 8192, 8192, 128, 2), (64, 8192, 8192, 128, 2), (256, 8192, 8192, 128, 1), (128, 4096, 16384, 128, 4),
    # 512 and more rows: 256-column tiles (measured faster there)
    (512, 4096, 8192, 256, 2), (1024, 2048, 8192, 256, 2)])
def test_plan_streaming_b_takes_128_column_tiles(M, N, K, bn, splits):
    for dt in (tg.GEMM_BF16, tg.GEMM_FP16):
        p = _plan(M, N, K, dt)
        assert (p["cta_group"], p["bn"], p["splits"]) == (1, bn, splits), (M, N, K, p)
        assert p["grid"] == p["tiles"] * p["splits"]
    # a forced tile width is kept
    try:
        tg.gemm_set_option("tc_bn", 256)
        assert _plan(M, N, K, tg.GEMM_BF16)["bn"] == 256
    finally:
        tg.gemm_set_option("tc_bn", 0)


@pytest.mark.parametrize("M,N,K,dt,bn,splits,cluster", [
    # too few 256-column tiles: two K ranges of 128-column tiles summed in cluster
    # shared memory where they fit one round of clusters and keep as many CTAs busy
    (256, 4096, 4096, "bf16", 128, 2, 2), (1024, 1024, 2048, "bf16", 128, 2, 2),
    (512, 2048, 2048, "fp16", 128, 2, 2), (768, 1536, 3072, "bf16", 128, 2, 2),
    (512, 2048, 2048, "tf32", 128, 2, 2), (512, 2048, 2048, "e4m3", 128, 2, 2),
    # ... not where they would not fit one round, or keep fewer CTAs busy
    (1024, 1536, 4096, "bf16", 256, 3, 0), (256, 2048, 8192, "bf16", 256, 9, 0),
    (2048, 1024, 2048, "bf16", 256, 2, 2), (1536, 1536, 1536, "bf16", 256, 2, 2),
    # little work: TF32 and 8-bit inputs take them instead of 64-column tiles, 16-bit inputs do not
    (1024, 1024, 1024, "tf32", 128, 2, 2), (1024, 1024, 1024, "e4m3", 128, 2, 2),
    (1024, 1024, 1024, "e5m2", 128, 2, 2), (1024, 1024, 1024, "bf16", 64, 1, 0),
    (1000, 1000, 1000, "bf16", 64, 1, 0), (1024, 1024, 512, "tf32", 64, 1, 0)])
def test_plan_two_k_ranges_in_cluster_shared_memory(M, N, K, dt, bn, splits, cluster):
    p = _plan(M, N, K, tg.DTYPES[dt])
    assert (p["cta_group"], p["bn"], p["splits"], p["cluster_split"]) == (1, bn, splits, cluster), (M, N, K, dt, p)
    assert p["b_kmajor"] == 0
    try:
        tg.gemm_set_option("tc_split_reduce", 1)           # the workspace path: the old choice stands
        q = _plan(M, N, K, tg.DTYPES[dt])
        assert q["cluster_split"] == 0
        tg.gemm_set_option("tc_split_reduce", 0)
        tg.gemm_set_option("tc_splits", 1)                  # no split at all
        assert _plan(M, N, K, tg.DTYPES[dt])["splits"] == 1
    finally:
        tg.gemm_set_option("tc_split_reduce", 0)
        tg.gemm_set_option("tc_splits", 0)


def test_plan_two_k_ranges_with_one_owner():
    """Two K ranges summed in cluster shared memory: of equal length unless
    asked; on request (128-column tiles, C stored by TMA) the first range
    takes that share of the k-blocks and its CTA owns the tile, and the
    forced workspace path cuts K at the same k-block."""
    p = _plan(128, 8192, 8192, tg.GEMM_BF16)
    assert (p["cluster_split"], p["splits"], p["bn"], p["kb_split"]) == (2, 2, 128, 0), p
    try:
        tg.gemm_set_option("tc_split_lead", 56)
        assert _plan(128, 8192, 8192, tg.GEMM_BF16)["kb_split"] == 72
        assert _plan(128, 8192, 8256, tg.GEMM_BF16)["kb_split"] == 72          # 129 k-blocks
        assert _plan(128, 8192, 8192, tg.GEMM_BF16, ldc=8195)["kb_split"] == 0  # C by ordinary stores
        assert _plan(128, 8192, 8192, tg.GEMM_TF32)["kb_split"] == 143         # 256 k-blocks
        assert _plan(1024, 2048, 8192, tg.GEMM_BF16)["kb_split"] == 0          # 256-column tiles
        assert _plan(128, 4096, 16384, tg.GEMM_BF16)["kb_split"] == 0          # 4 ranges
        assert _plan(8192, 8192, 8192, tg.GEMM_BF16)["kb_split"] == 0
        for lead, kb in ((0, 0), (50, 0), (51, 65), (75, 96), (95, 122)):
            assert tg.gemm_set_option("tc_split_lead", lead) == tg.GEMM_OK
            assert _plan(128, 8192, 8192, tg.GEMM_BF16)["kb_split"] == kb, lead
        tg.gemm_set_option("tc_split_lead", 56)
        tg.gemm_set_option("tc_split_reduce", 1)
        q = _plan(128, 8192, 8192, tg.GEMM_BF16)
        assert q["cluster_split"] == 0 and q["kb_split"] == 72, q
        for bad in (1, 49, 96, -1):
            assert tg.gemm_set_option("tc_split_lead", bad) == tg.GEMM_ERR_INVALID_ARG
    finally:
        tg.gemm_set_option("tc_split_lead", 0)
        tg.gemm_set_option("tc_split_reduce", 0)


def test_plan_struct_layout_matches_the_header(tmp_path):
    src = tmp_path / "plan.c"
    src.write_text('#include <stddef.h>\n#include <stdio.h>\n#include "gemm.h"\n'
                   'int main(void) { printf("%zu %zu %zu\\n", sizeof(gemm_plan_t),'
                   ' offsetof(gemm_plan_t, cluster_split), offsetof(gemm_plan_t, kb_split)); return 0; }\n')
    exe = tmp_path / "plan"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    P = tg.GemmPlan
    assert got == [ctypes.sizeof(P), P.cluster_split.offset, P.kb_split.offset]


def test_plan_runs_the_last_round_as_column_halves():
    # 256 pair tiles over 76 pairs: 3 rounds and 28 tiles left, which as 56
    # halves fit one round; on by default for 16-bit inputs on short schedules
    for dt in (tg.GEMM_BF16, tg.GEMM_FP16):
        q = _plan(4096, 4096, 4096, dt)
        assert q["half_tiles"] == 28 and q["tail_tiles"] == 0 and q["splits"] == 1 and q["grid"] == 152, (dt, q)
    assert _plan(16384, 1024, 4096, tg.GEMM_BF16)["half_tiles"] == 28
    # not by default on 14 rounds (8192^3: neutral) nor for TF32 (its K split is faster)
    assert _plan(8192, 8192, 8192, tg.GEMM_BF16)["half_tiles"] == 0
    t = _plan(4096, 4096, 4096, tg.GEMM_TF32)
    assert t["half_tiles"] == 0 and t["tail_tiles"] == 28
    try:
        assert tg.gemm_set_option("tc_tail_halves", 2) == 0          # 2: wherever the tile allows it
        # 1024 tiles: 13 rounds and 36 left, 72 halves
        p = _plan(8192, 8192, 8192, tg.GEMM_BF16)
        assert p["half_tiles"] == 36 and p["tail_tiles"] == 0 and p["grid"] == 152
        t = _plan(4096, 4096, 4096, tg.GEMM_TF32)                   # TF32 B as stored halves too
        assert t["half_tiles"] == 28 and t["tail_tiles"] == 0
        # 272 tiles leave 44: 88 halves would not fit one round
        assert _plan(4097, 4095, 4099, tg.GEMM_BF16)["half_tiles"] == 0
        # FP8 B as stored comes in one 128-column chunk per CTA: no halves
        assert _plan(8192, 8192, 8192, tg.GEMM_E4M3)["half_tiles"] == 0
        # a whole number of rounds: no tail
        assert _plan(256, 256 * 76, 4096, tg.GEMM_BF16)["half_tiles"] == 0
    finally:
        tg.gemm_set_option("tc_tail_halves", 0)
    # 1-CTA 128 x 256 tiles halve too; 64-column tiles do not
    try:
        assert tg.gemm_set_option("tc_cta_group", 1) == 0
        assert tg.gemm_set_option("tc_max_ctas", 100) == 0
        r = _plan(128 * 130, 256, 1024, tg.GEMM_BF16)             # 130 tiles on 100 CTAs: 30 left
        assert r["bn"] == 256 and r["half_tiles"] == 30 and r["grid"] == 100
        assert tg.gemm_set_option("tc_bn", 64) == 0
        assert _plan(128 * 130, 64, 1024, tg.GEMM_BF16)["half_tiles"] == 0
    finally:
        for k in ("tc_cta_group", "tc_max_ctas", "tc_bn"):
            tg.gemm_set_option(k, 0)
    try:
        assert tg.gemm_set_option("tc_tail_halves", 1) == 0          # 1: off
        assert _plan(4096, 4096, 4096, tg.GEMM_BF16)["half_tiles"] == 0
    finally:
        tg.gemm_set_option("tc_tail_halves", 0)
    assert tg.gemm_set_option("tc_tail_halves", 3) == tg.GEMM_ERR_INVALID_ARG
    assert tg.gemm_get_option("tc_tail_halves") == 0
    assert tg.gemm_get_option("pdl") == 0
    assert tg.gemm_set_option("pdl", 1) == 0 and tg.gemm_get_option("pdl") == 1
    assert tg.gemm_set_option("pdl", 2) == tg.GEMM_ERR_INVALID_ARG
    assert tg.gemm_set_option("pdl", 0) == 0


def test_plan_splits_the_last_round_in_k_only_on_request():
    try:
        assert tg.gemm_set_option("tc_tail_halves", 1) == 0
        # without column halves: off by default for 16- and 8-bit inputs
        # (measured: no gain or a loss) ...
        assert _plan(8192, 8192, 8192, tg.GEMM_BF16)["tail_tiles"] == 0
        assert _plan(4096, 4096, 4096, tg.GEMM_BF16)["tail_tiles"] == 0
        assert _plan(4096, 4096, 4096, tg.GEMM_E4M3)["tail_tiles"] == 0
        # ... on, two K ranges, for TF32
        auto = _plan(4096, 4096, 4096, tg.GEMM_TF32)
        assert auto["tail_tiles"] == 28 and auto["splits"] == 2 and auto["half_tiles"] == 0
    finally:
        tg.gemm_set_option("tc_tail_halves", 0)
    try:
        assert tg.gemm_set_option("tc_tail_splits", 1) == 0          # 1: off for every dtype
        assert _plan(4096, 4096, 4096, tg.GEMM_TF32)["tail_tiles"] == 0
        # 1024 pair tiles over 76 pairs: 13 full rounds and 36 tiles left
        assert tg.gemm_set_option("tc_tail_splits", 2) == 0          # a K split takes precedence
        p = _plan(8192, 8192, 8192, tg.GEMM_BF16)
        assert p["tail_tiles"] == 36 and p["splits"] == 2 and p["grid"] == 152 and p["half_tiles"] == 0
        # TF32 4096^3: 256 pair tiles, 28 left after 3 rounds
        q = _plan(4096, 4096, 4096, tg.GEMM_TF32)
        assert q["tail_tiles"] == 28 and q["splits"] == 2
        assert tg.gemm_set_option("tc_tail_splits", 3) == 0
        t = _plan(8192, 8192, 8192, tg.GEMM_BF16)
        assert t["tail_tiles"] == 36 and t["splits"] == 3
        # no partly idle round: nothing to split
        assert _plan(256, 256 * 76, 4096, tg.GEMM_BF16)["tail_tiles"] == 0
    finally:
        tg.gemm_set_option("tc_tail_splits", 0)


@pytest.mark.parametrize("kb,req,eff", [(9, 4, 3), (10, 4, 4), (16, 3, 3), (5, 8, 5), (128, 32, 32)])
def test_forced_splits_leave_no_empty_k_range(kb, req, eff):
    try:
        assert tg.gemm_set_option("tc_splits", req) == 0
        p = _plan(256, 256, kb * 64, tg.GEMM_BF16)
        assert p["splits"] == eff
        per = -(-kb // eff)
        assert (eff - 1) * per < kb          # the last K range is not empty
    finally:
        tg.gemm_set_option("tc_splits", 0)


def test_plan_forced_options():
    try:
        assert tg.gemm_set_option("tc_b_major", 1) == 0
        assert _plan(512, 512, 512, tg.GEMM_BF16)["b_kmajor"] == 1
        assert _plan(512, 512, 512, tg.GEMM_TF32)["b_kmajor"] == 1
        assert tg.gemm_set_option("tc_b_major", 2) == 0
        assert _plan(512, 512, 512, tg.GEMM_BF16)["b_kmajor"] == 0
        assert _plan(512, 512, 512, tg.GEMM_TF32)["b_kmajor"] == 0
        assert tg.gemm_set_option("tc_b_major", 0) == 0
        assert tg.gemm_set_option("tc_cta_group", 1) == 0
        assert tg.gemm_set_option("tc_bn", 128) == 0
        p = _plan(8192, 8192, 8192, tg.GEMM_BF16)
        assert p["cta_group"] == 1 and p["bn"] == 128
        assert tg.gemm_set_option("tc_max_ctas", 10) == 0
        assert _plan(8192, 8192, 8192, tg.GEMM_BF16)["grid"] == 10
    finally:
        for k in ("tc_cta_group", "tc_bn", "tc_max_ctas", "tc_b_major"):
            tg.gemm_set_option(k, 0)


def test_python_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    monkeypatch.setattr(tg, "_lib", None)
    monkeypatch.setattr(tg, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no fallback"):
        tg.gemm_version()


# ------------------------------------------------------------ gemm_run_ex ---
def _ex(M, N, K, dtype, A, lda, B, ldb, C, ldc, **epi):
    return tg.gemm_run_ex(M, N, K, dtype, A, lda, B, ldb, C, ldc, tg.make_epilogue(**epi), 0)


def test_epilogue_struct_layout_matches_the_header(tmp_path):
    src = tmp_path / "layout.c"
    src.write_text('#include <stddef.h>\n#include <stdio.h>\n#include "gemm.h"\n'
                   'int main(void) { printf("%zu %zu %zu %zu %zu %zu\\n", sizeof(gemm_epilogue_t),'
                   ' offsetof(gemm_epilogue_t, alpha), offsetof(gemm_epilogue_t, beta),'
                   ' offsetof(gemm_epilogue_t, bias), offsetof(gemm_epilogue_t, activation),'
                   ' offsetof(gemm_epilogue_t, out_dtype)); return 0; }\n')
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    E = tg.GemmEpilogue
    assert got == [ctypes.sizeof(E), E.alpha.offset, E.beta.offset, E.bias.offset, E.activation.offset,
                   E.out_dtype.offset]


def test_epilogue_enumerations_match_the_header():
    src = open(os.path.join(ROOT, "include", "gemm.h")).read()
    for name, value in (("GEMM_ACT_NONE", 0), ("GEMM_ACT_RELU", 1), ("GEMM_ACT_GELU", 2), ("GEMM_OUT_F32", 0),
                        ("GEMM_OUT_BF16", 1), ("GEMM_OUT_F16", 2)):
        assert re.search(rf"\b{name}\s*=\s*{value}\b", src), name
        assert getattr(tg, name) == value


def test_epilogue_rejects_unknown_activation_and_output_type():
    ep = tg.GemmEpilogue(1.0, 0.0, None, 7, 0)
    assert tg.gemm_run_ex(8, 8, 8, tg.GEMM_BF16, 1 << 20, 8, 1 << 21, 8, 1 << 22, 8, ep, 0) == tg.GEMM_ERR_INVALID_ARG
    assert "activation" in tg.gemm_last_error()
    ep = tg.GemmEpilogue(1.0, 0.0, None, 0, 9)
    assert tg.gemm_run_ex(8, 8, 8, tg.GEMM_BF16, 1 << 20, 8, 1 << 21, 8, 1 << 22, 8, ep, 0) == tg.GEMM_ERR_INVALID_ARG
    assert "output type" in tg.gemm_last_error()


def test_epilogue_argument_checks_before_cuda():
    A, B = 1 << 20, 1 << 21
    # bias inside C's footprint
    rc = _ex(8, 8, 8, tg.GEMM_BF16, A, 8, B, 8, 1 << 22, 8, bias=(1 << 22) + 16, act="relu", out="bf16")
    assert rc == tg.GEMM_ERR_INVALID_ARG and "bias overlaps C" in tg.gemm_last_error()
    # a BF16 C at an odd address, a bias that is not 4-byte aligned
    rc = _ex(8, 8, 8, tg.GEMM_BF16, A, 8, B, 8, (1 << 22) + 1, 8, out="bf16")
    assert rc == tg.GEMM_ERR_INVALID_ARG and "aligned" in tg.gemm_last_error()
    rc = _ex(8, 8, 8, tg.GEMM_BF16, A, 8, B, 8, 1 << 22, 8, bias=(1 << 23) + 2, out="bf16")
    assert rc == tg.GEMM_ERR_INVALID_ARG and "bias is not 4-byte aligned" in tg.gemm_last_error()
    # a BF16 C half the size of an FP32 one: C right after A's footprint is fine
    # for the overlap check, C one element earlier overlaps
    a_end = A + (7 * 8 + 8) * 2
    rc = _ex(8, 8, 8, tg.GEMM_BF16, A, 8, B, 8, a_end - 2, 8, out="bf16")
    assert rc == tg.GEMM_ERR_INVALID_ARG and "overlap" in tg.gemm_last_error()


def test_null_epilogue_behaves_as_gemm_run():
    assert tg.gemm_run_ex(0, 5, 3, tg.GEMM_BF16, 0, 3, 0, 5, 0, 5, None, 0) == tg.GEMM_OK
    assert tg.gemm_run_ex(4, 4, 4, 7, 16, 4, 16, 4, 64, 4, None, 0) == tg.GEMM_ERR_INVALID_ARG


# ------------------------------------------------------- gemm_run_grouped ---
def _grp(M, N, K, A, lda, B, ldb, C, ldc, bias=0):
    return tg.GemmGroup(M, N, K, A, lda, B, ldb, C, ldc, bias or None)


def test_group_struct_layout_matches_the_header(tmp_path):
    src = tmp_path / "glayout.c"
    fields = ("M", "N", "K", "A", "lda", "B", "ldb", "C", "ldc", "bias")
    src.write_text('#include <stddef.h>\n#include <stdio.h>\n#include "gemm.h"\n'
                   'int main(void) { printf("%zu' + ' %zu' * len(fields) + '\\n", sizeof(gemm_group_t)'
                   + "".join(f", offsetof(gemm_group_t, {f})" for f in fields) + '); return 0; }\n')
    exe = tmp_path / "glayout"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    assert got == [ctypes.sizeof(tg.GemmGroup)] + [getattr(tg.GemmGroup, f).offset for f in fields]


def test_grouped_argument_checks_before_cuda():
    BF = tg.GEMM_BF16
    ok = _grp(8, 8, 8, 1 << 20, 8, 1 << 21, 8, 1 << 22, 8)
    assert tg.gemm_run_grouped(BF, []) == tg.GEMM_OK                                  # nothing to do
    assert tg.gemm_run_grouped(BF, [_grp(0, 8, 8, 0, 8, 0, 8, 0, 8)]) == tg.GEMM_OK   # only empty groups
    lib = tg.load_library()
    assert lib.gemm_run_grouped(BF, -1, None, None, None) == tg.GEMM_ERR_INVALID_ARG
    assert lib.gemm_run_grouped(BF, 3, None, None, None) == tg.GEMM_ERR_INVALID_ARG
    assert "NULL" in tg.gemm_last_error()
    # the shared epilogue may not carry a bias
    ep = tg.make_epilogue(1.0, 0.0, 1 << 23, "none", "f32")
    assert tg.gemm_run_grouped(BF, [ok], ep) == tg.GEMM_ERR_INVALID_ARG and "bias" in tg.gemm_last_error()
    # a bad group anywhere in the list
    assert tg.gemm_run_grouped(BF, [ok, _grp(8, 8, 8, 1 << 24, 4, 1 << 25, 8, 1 << 26, 8)]) == tg.GEMM_ERR_INVALID_ARG
    assert "leading dimension" in tg.gemm_last_error()
    # two groups writing overlapping C
    two = [ok, _grp(8, 8, 8, 1 << 24, 8, 1 << 25, 8, (1 << 22) + 64, 8)]
    assert tg.gemm_run_grouped(BF, two) == tg.GEMM_ERR_INVALID_ARG and "C overlap" in tg.gemm_last_error()
    # one group's C over another group's A
    cross = [ok, _grp(8, 8, 8, 1 << 24, 8, 1 << 25, 8, (1 << 20) + 16, 8)]
    assert tg.gemm_run_grouped(BF, cross) == tg.GEMM_ERR_INVALID_ARG and "overlaps" in tg.gemm_last_error()
    # a bias inside some C, a misaligned bias
    bad_bias = [ok, _grp(8, 8, 8, 1 << 24, 8, 1 << 25, 8, 1 << 26, 8, bias=(1 << 22) + 8)]
    assert tg.gemm_run_grouped(BF, bad_bias) == tg.GEMM_ERR_INVALID_ARG and "bias" in tg.gemm_last_error()
    mis = [_grp(8, 8, 8, 1 << 24, 8, 1 << 25, 8, 1 << 26, 8, bias=(1 << 27) + 2)]
    assert tg.gemm_run_grouped(BF, mis) == tg.GEMM_ERR_INVALID_ARG and "aligned" in tg.gemm_last_error()
    assert tg.gemm_run_grouped(9, [ok]) == tg.GEMM_ERR_INVALID_ARG and "dtype" in tg.gemm_last_error()


def test_torch_wrappers_check_their_tensors_before_the_library():
    """The torch-level calls reject host tensors, a C of the wrong type or
    shape, a malformed bias and mismatched group lists with a Python error,
    before anything reaches the C ABI (these tensors live on the CPU)."""
    import torch
    A = torch.zeros(8, 16)
    B = torch.zeros(16, 4)
    with pytest.raises(ValueError, match="CUDA tensors"):
        tg.gemm(A, B)
    with pytest.raises(TypeError, match="float32 tensor"):
        tg.gemm(A, B, C=torch.zeros(8, 5))
    with pytest.raises(TypeError, match="float32 tensor"):
        tg.gemm(A, B, C=torch.zeros(8, 4, dtype=torch.float16))
    with pytest.raises(ValueError, match="inner dimensions"):
        tg.gemm(A, torch.zeros(15, 4))
    with pytest.raises(TypeError, match="operands"):
        tg.gemm(A, B, dtype="bf16")
    with pytest.raises(ValueError, match="CUDA tensors"):
        tg.gemm_ex(A, B, bias=torch.zeros(4))
    with pytest.raises(TypeError, match="bias"):
        tg.gemm_ex(A, B, bias=torch.zeros(5))
    with pytest.raises(TypeError, match="bias"):
        tg.gemm_ex(A, B, bias=torch.zeros(4, dtype=torch.float64))
    with pytest.raises(ValueError, match="differ in length"):
        tg.gemm_grouped([A, A], [B])
    with pytest.raises(ValueError, match="differ in length"):
        tg.gemm_grouped([A], [B], Cs=[torch.zeros(8, 4), torch.zeros(8, 4)])
    with pytest.raises(TypeError, match="bias"):
        tg.gemm_grouped([A], [B], biases=[torch.zeros(3)])
    with pytest.raises(ValueError, match="CUDA tensors"):
        tg.gemm_grouped([A], [B])
    assert tg.gemm_grouped([], []) == []
