"""The kernel's timeline trace (options "trace_addr" / "trace_records"):
one record per work unit for the TMA producer and the MMA issuer, one per
unit and lane quarter for the epilogue warps, one per CTA; spans ordered
within a unit (loads start before the MMAs end, the epilogue ends after the
MMAs); overflow drops records without harm; a bad buffer is refused before
any launch.  The conversion to Chrome-trace JSON runs on the CPU."""
import numpy as np
import pytest
import torch

import tiled_tensor_core_gemm_gb300 as tg
from tiled_tensor_core_gemm_gb300 import build as tgbuild
from tiled_tensor_core_gemm_gb300 import trace as tt
from tiled_tensor_core_gemm_gb300.inputs import make_operands


def test_chrome_trace_layout_on_cpu():
    recs = np.zeros(3, dtype=tt.RECORD)
    recs[0] = (1000, 5000, -1, 4, 3, 7, 0)
    recs[1] = (1200, 4000, 12, 2, 3, 7, 16)
    recs[2] = (4100, 4900, 12, 3, 3, 7, 6)
    ev = tt.chrome_trace(recs)["traceEvents"]
    assert [e["ts"] for e in ev] == [0.0, 0.2, 3.1] and [e["dur"] for e in ev] == [4.0, 2.8, 0.8]
    assert ev[2]["name"] == "epilogue (to peer) u12" and ev[2]["tid"] == 36 and ev[0]["pid"] == 3
    s = tt.summary(recs)
    assert s["launch_us"] == 4.0 and s["mma_us_per_unit"] == 2.8
    assert tt.RECORD.itemsize == 32


@pytest.fixture(scope="module")
def lib():
    tgbuild.build()
    tg.load_library()
    yield


def _run(A, B, dtype):
    Ad, Bd = A.cuda(), B.cuda()
    out = {}

    def go():
        out["C"] = tg.gemm(Ad, Bd, dtype=dtype)
    return out, go


@pytest.mark.gpu
def test_trace_records_every_unit_and_role(lib):
    M, N, K = 2048, 2048, 1024
    A, B = make_operands(M, N, K, "bf16", "ints", seed=41)
    plan = tg.gemm_plan(M, N, K, tg.GEMM_BF16, 0, K, 0, N, 0, N).as_dict()
    units = plan["tiles"]                      # whole tiles only on this shape
    assert plan["tail_tiles"] == 0 and plan["half_tiles"] == 0 and plan["cta_group"] == 1, plan
    out, go = _run(A, B, "bf16")
    recs, count = tt.capture(go)
    assert len(recs) <= count          # (slots are reserved 16 at a time per recording thread)
    per_role = np.bincount(recs["role"], minlength=7)
    assert per_role[1] == per_role[2] == units and per_role[3] == 4 * units
    assert per_role[4] == plan["grid"] and per_role[5] == 2 * plan["grid"]
    assert per_role[6] == 4 * plan["grid"]           # each epilogue warp's last store -> its reads done
    for role, per_unit in ((1, 1), (2, 1), (3, 4)):
        sel = recs[recs["role"] == role]
        assert sorted(np.bincount(sel["unit"], minlength=units).tolist()) == [per_unit] * units, role
    assert np.all(recs["t_end_ns"] >= recs["t_begin_ns"])
    assert sorted(recs[recs["role"] == 3]["sub"].tolist()) == sorted([0, 1, 2, 3] * units)
    # within each unit: loads start before the MMAs end, which end before the epilogue does
    by = {(int(r["role"]), int(r["unit"])): r for r in recs if r["role"] in (1, 2)}
    for r in recs[recs["role"] == 3]:
        u = int(r["unit"])
        assert by[(1, u)]["t_begin_ns"] <= by[(2, u)]["t_end_ns"] <= r["t_end_ns"]
    # every unit span lies inside its CTA's life
    assert np.sum(recs["role"] == 5) == 2 * plan["grid"]
    life = {int(r["cta"]): r for r in recs[recs["role"] == 4]}
    assert len(life) == plan["grid"]
    for r in recs[recs["role"] != 4]:
        c = life[int(r["cta"])]
        assert c["t_begin_ns"] <= r["t_begin_ns"] and r["t_end_ns"] <= c["t_end_ns"]
    import oracle
    from tiled_tensor_core_gemm_gb300.inputs import as_oracle_array
    assert np.array_equal(out["C"].cpu().numpy().astype(np.float64),
                          oracle.gemm(as_oracle_array(A), as_oracle_array(B), bf16=True))


@pytest.mark.gpu
@pytest.mark.parametrize("lead", (0, 56), ids=("quarters_shared", "one_owner"))
def test_trace_shows_cluster_split_senders(lib, lead):
    M, N, K = 128, 2048, 4096
    A, B = make_operands(M, N, K, "bf16", "ints", seed=42)
    try:
        tg.gemm_set_option("tc_splits", 2)
        tg.gemm_set_option("tc_split_lead", lead)
        plan = tg.gemm_plan(M, N, K, tg.GEMM_BF16, 0, K, 0, N, 0, N).as_dict()
        assert plan["cluster_split"] == 2 and (plan["kb_split"] > 0) == (lead > 50), plan
        out, go = _run(A, B, "bf16")
        recs, count = tt.capture(go)
    finally:
        tg.gemm_set_option("tc_splits", 0)
        tg.gemm_set_option("tc_split_lead", 0)
    epi = recs[recs["role"] == 3]
    sends, stores = epi[epi["sub"] >= 4], epi[epi["sub"] < 4]
    # four lane quarters per tile are sent and four stored, per cluster of two CTAs
    assert len(sends) == len(stores) == 2 * plan["grid"]
    if lead <= 50:
        # each CTA sends two lane quarters to its peer and stores the other two
        for half in (sends, stores):
            assert np.all(np.bincount(half["cta"], minlength=plan["grid"]) == 2)
    else:
        # CTA 1 of each cluster sends all four, CTA 0 stores all four
        assert np.all(sends["cta"] % 2 == 1) and np.all(stores["cta"] % 2 == 0)
    # an owning warp's detail: to the first partial chunk, to the last, to its last store
    detail = recs[(recs["role"] == 6) & (recs["sub"] < 3)]
    assert len(detail) == 3 * 2 * plan["grid"] and np.all(detail["t_end_ns"] >= detail["t_begin_ns"])
    import oracle
    from tiled_tensor_core_gemm_gb300.inputs import as_oracle_array
    assert np.array_equal(out["C"].cpu().numpy().astype(np.float64),
                          oracle.gemm(as_oracle_array(A), as_oracle_array(B), bf16=True))


@pytest.mark.gpu
def test_trace_overflow_and_bad_buffer(lib):
    A, B = make_operands(1024, 1024, 512, "bf16", "ints", seed=43)
    out, go = _run(A, B, "bf16")
    recs, count = tt.capture(go, capacity=10)
    assert 0 < len(recs) <= 10 and count > 10
    host = torch.zeros(64, dtype=torch.uint8).pin_memory()
    assert tg.gemm_set_option("trace_addr", host.data_ptr()) == tg.GEMM_OK
    try:
        with pytest.raises(tg.GemmError, match="trace buffer"):
            tg.gemm(A.cuda(), B.cuda())
    finally:
        tg.gemm_set_option("trace_addr", 0)
    assert tg.gemm_set_option("trace_addr", 12) == tg.GEMM_ERR_INVALID_ARG      # not 8-byte aligned
