"""The row-sharded GEMM's host logic across ranks, on CPU with gloo (world
size 2).  The per-rank product is the oracle here (no GPU); what is checked
is everything around it: the row partition (ragged M, a rank with no rows),
the broadcast of B into each rank's own buffer, and the all-gather of the row
slabs, whose result must equal the oracle's product of the whole A and B."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from tiled_tensor_core_gemm_gb300.sharded import gather_rows, gemm_sharded, row_shards


def test_row_shards_cover_m_in_order_and_balance():
    for M in (0, 1, 2, 7, 128, 4097, 8192):
        for world in (1, 2, 3, 8):
            s = row_shards(M, world)
            assert len(s) == world
            assert s[0][0] == 0 and all(a[0] + a[1] == b[0] for a, b in zip(s, s[1:]))
            assert sum(rows for _, rows in s) == M
            assert max(r for _, r in s) - min(r for _, r in s) <= 1
    assert row_shards(1, 2) == [(0, 1), (1, 0)]
    assert row_shards(4097, 2) == [(0, 2049), (2049, 2048)]
    with pytest.raises(ValueError):
        row_shards(-1, 2)
    with pytest.raises(ValueError):
        row_shards(4, 0)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _oracle_gemm(a, b, dtype):
    import oracle
    return torch.from_numpy(oracle.gemm(a.numpy(), b.numpy()).astype(np.float32))


def _worker(rank, world, port, cases, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        for i, (M, N, K) in enumerate(cases):
            g = torch.Generator().manual_seed(100 + i)
            A = torch.rand((M, K), generator=g) * 2 - 1
            B_root = torch.rand((K, N), generator=g) * 2 - 1
            # every rank has its own B buffer; only rank 0's holds the values
            B = B_root.clone() if rank == 0 else torch.zeros((K, N))
            row0, rows = row_shards(M, world)[rank]
            C = gemm_sharded(A[row0:row0 + rows].contiguous(), B, M, dtype="fp32", b_src=0, gather=True,
                             local_gemm=_oracle_gemm)
            out[(rank, i)] = (C.numpy(), bool(torch.equal(B, B_root)), rows)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_sharded_gemm_gloo_world2_matches_the_whole_product():
    import oracle
    world = 2
    cases = [(37, 19, 23), (1, 8, 5), (2, 3, 4), (64, 33, 17)]       # ragged M, and M = 1: rank 1 has no rows
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_worker, args=(world, _free_port(), cases, out), nprocs=world, join=True)
    for i, (M, N, K) in enumerate(cases):
        g = torch.Generator().manual_seed(100 + i)
        A = torch.rand((M, K), generator=g) * 2 - 1
        B = torch.rand((K, N), generator=g) * 2 - 1
        want = oracle.gemm(A.numpy(), B.numpy()).astype(np.float32)
        for rank in range(world):
            C, b_ok, rows = out[(rank, i)]
            assert b_ok, (rank, i)                          # B arrived in this rank's own buffer
            assert rows == row_shards(M, world)[rank][1]
            assert C.shape == (M, N) and np.array_equal(C, want), (rank, i)


def test_single_process_runs_as_world_one():
    A = torch.arange(12, dtype=torch.float32).reshape(3, 4)
    B = torch.ones((4, 2))
    C = gemm_sharded(A, B, 3, dtype="fp32", b_src=0, gather=True, local_gemm=lambda a, b, d: a @ b)
    assert torch.equal(C, A @ B)
    assert gather_rows(C, 3) is C
    with pytest.raises(ValueError):
        gemm_sharded(A[:2], B, 3, local_gemm=lambda a, b, d: a @ b)


@pytest.mark.gpu
def test_row_slabs_through_the_library_match_the_oracle():
    """On one GPU: the library's product on each rank's row slab of a ragged
    A (views into one buffer, as each rank would hold them), concatenated,
    equals the oracle's product of the whole A; and gemm_sharded at world
    size 1 runs the library itself."""
    import tiled_tensor_core_gemm_gb300 as tg
    from tiled_tensor_core_gemm_gb300 import build as tgbuild
    from tiled_tensor_core_gemm_gb300.inputs import as_oracle_array, make_operands
    import oracle
    tgbuild.build()
    tg.load_library()
    M, N, K = 1000, 768, 512
    A, B = make_operands(M, N, K, "bf16", "ints", seed=31)
    Ad, Bd = A.cuda(), B.cuda()
    want = oracle.gemm(as_oracle_array(A), as_oracle_array(B), bf16=True)
    for world in (2, 3, 7):
        parts = [tg.gemm(Ad[row0:row0 + rows], Bd) for row0, rows in row_shards(M, world) if rows > 0]
        C = torch.cat(parts).cpu().numpy().astype(np.float64)
        assert np.array_equal(C, want), world
    C1 = gemm_sharded(Ad, Bd, M, b_src=0, gather=True)
    assert np.array_equal(C1.cpu().numpy().astype(np.float64), want)
