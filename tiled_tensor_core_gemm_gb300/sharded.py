"""Row-sharded GEMM over the ranks of a process group (one GPU per rank).

C = A.B splits along M with no exchange inside the product: rank r owns rows
[row0_r, row0_r + rows_r) of A and of C, and every rank holds all of B.  The
pages define the product ("Shared memory and tensor cores", section 13.1:
C = A @ B, each output row the product of one row of A with B), so a block of
rows of C needs only the same rows of A and the whole of B.

What crosses ranks, and when:
  * B, once, before the product: a broadcast from one rank into every rank's
    own buffer (``broadcast_b``).  Each rank's kernels and TMA descriptors then
    read only that rank's own device memory -- no peer-memory operand and no
    multicast.
  * C, optionally, once, after the product: an all-gather of the row slabs
    (``gather_rows``), for callers that want the whole of C on every rank.
Nothing is exchanged while the kernels run.

The partition (``row_shards``) is balanced: the first M mod world ranks get
one row more; with M < world the last ranks get no rows and skip the call.
Without an initialised process group everything runs as world size 1.
"""
from __future__ import annotations


def row_shards(M: int, world: int):
    """[(row0, rows)] for every rank: contiguous, in rank order, covering
    [0, M) exactly, sizes differing by at most one."""
    if M < 0 or world < 1:
        raise ValueError(f"bad partition request M={M} world={world}")
    base, extra = divmod(M, world)
    out, row0 = [], 0
    for r in range(world):
        rows = base + (1 if r < extra else 0)
        out.append((row0, rows))
        row0 += rows
    return out


def _group_info(group):
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return None, 1, 0
    return dist, dist.get_world_size(group), dist.get_rank(group)


def broadcast_b(B, src: int = 0, group=None):
    """Copy B from rank `src` into B on every rank of `group` (in place: each
    rank passes its own buffer of the same shape and type).  A no-op at world
    size 1."""
    dist, world, _ = _group_info(group)
    if world > 1:
        dist.broadcast(B, src=src, group=group)
    return B


def gather_rows(C_local, M: int, group=None):
    """The whole M x N C on every rank from the ranks' row slabs (row_shards
    order).  Slabs are padded to the largest slab for the collective and cut
    back afterwards."""
    import torch

    dist, world, rank = _group_info(group)
    if world == 1:
        return C_local
    shards = row_shards(M, world)
    if C_local.shape[0] != shards[rank][1]:
        raise ValueError(f"rank {rank} holds {C_local.shape[0]} rows, its shard has {shards[rank][1]}")
    width = max(rows for _, rows in shards)
    N = C_local.shape[1]
    pad = torch.zeros((width, N), dtype=C_local.dtype, device=C_local.device)
    pad[:C_local.shape[0]].copy_(C_local)
    parts = [torch.empty_like(pad) for _ in range(world)]
    dist.all_gather(parts, pad, group=group)
    return torch.cat([p[:rows] for p, (_, rows) in zip(parts, shards)], dim=0)


def gemm_sharded(A_local, B, M: int, dtype=None, group=None, b_src=None, gather=False, local_gemm=None):
    """This rank's rows of C = A.B, computed by the library on this rank's GPU.

    A_local   this rank's row slab of A (row_shards(M, world)[rank] rows).
    B         the whole of B in this rank's own memory; with b_src set, it is
              first overwritten by rank b_src's B (broadcast_b).
    M         total rows of A and C across the group.
    gather    return the whole of C on every rank instead of this rank's slab.
    local_gemm  the per-rank product, (A_slab, B, dtype) -> C_slab; default:
              the library's gemm (gemm_run on the current stream).
    """
    from . import gemm as library_gemm

    _, world, rank = _group_info(group)
    row0, rows = row_shards(M, world)[rank]
    if A_local.shape[0] != rows:
        raise ValueError(f"rank {rank} of {world}: A slab has {A_local.shape[0]} rows, its shard {rows}")
    if b_src is not None:
        broadcast_b(B, b_src, group)
    run = local_gemm or (lambda a, b, d: library_gemm(a, b, dtype=d))
    if rows > 0:
        C_local = run(A_local, B, dtype)
    else:
        import torch
        C_local = torch.empty((0, B.shape[1]), dtype=torch.float32, device=B.device)
    return gather_rows(C_local, M, group) if gather else C_local
