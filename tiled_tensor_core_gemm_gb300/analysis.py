"""Closed-form models used to design and report the GEMM kernels.

* FLOP count and compulsory bytes of C = A.B -- "Shared memory and tensor
  cores" (ml-compiler-from-scratch ch. 13), section 13.1.
* DRAM reads of a BM x BN block tiling with no cache reuse, and its arithmetic
  intensity BM*BN / (2 (BM + BN)) flop per byte -- same section.
* The shared-memory bank model (32 banks of 4 bytes, one word per bank per
  pass, equal words broadcast) -- same page, section 13.6.
* Peak arithmetic rates derived from unit counts and clocks.

These are pure host arithmetic: no GPU, no oracle.
"""
from __future__ import annotations

from typing import Callable, Iterable


def gemm_flops(M: int, N: int, K: int) -> int:
    """One multiply and one add per (i, j, k): 2*M*N*K."""
    return 2 * M * N * K


def compulsory_bytes(M: int, N: int, K: int, in_bytes: int, out_bytes: int = 4) -> int:
    """Read A and B once, write C once."""
    return (M * K + K * N) * in_bytes + M * N * out_bytes


def compulsory_read_bytes(M: int, N: int, K: int, in_bytes: int) -> int:
    return (M * K + K * N) * in_bytes


def naive_read_bytes(M: int, N: int, K: int, in_bytes: int = 4) -> int:
    """One A element and one B element loaded per multiply-add."""
    return 2 * M * N * K * in_bytes


def block_tile_read_bytes(M: int, N: int, K: int, BM: int, BN: int, in_bytes: int = 4) -> int:
    """Each of the ceil(M/BM)*ceil(N/BN) blocks reads a BM x K panel of A and a
    K x BN panel of B once; no reuse between blocks is assumed."""
    tiles_m = -(-M // BM)
    tiles_n = -(-N // BN)
    return tiles_m * tiles_n * (BM + BN) * K * in_bytes


def block_tile_intensity(BM: int, BN: int, in_bytes: int = 4) -> float:
    """Flop per byte of DRAM reads for a block tile: 2*BM*BN*K / ((BM+BN)*K*in_bytes)."""
    return 2.0 * BM * BN / ((BM + BN) * in_bytes)


def bank_passes(addr_of_lane: Callable[[int], int], lanes: int = 32,
                banks: int = 32, word_bytes: int = 4, byte_addresses: bool = False) -> int:
    """Worst-case shared-memory passes for one warp access.

    addr_of_lane(t) gives the 4-byte word index (or byte address with
    byte_addresses=True) that lane t touches.  Lanes touching the same word are
    served together; distinct words in one bank serialise.
    """
    words = set()
    for t in range(lanes):
        a = addr_of_lane(t)
        words.add(a // word_bytes if byte_addresses else a)
    per_bank: dict[int, set] = {}
    for w in words:
        per_bank.setdefault(w % banks, set()).add(w)
    return max(len(s) for s in per_bank.values())


def vector_bank_passes(byte_addr_of_lane: Callable[[int], int], vec_bytes: int,
                       lanes: int = 32) -> int:
    """Passes for a warp-wide vector access of vec_bytes per lane (8 or 16).

    The hardware splits a 16-byte access into quarter-warp phases (8 lanes,
    128 bytes each) and an 8-byte access into half-warp phases; each phase is
    scored with the scalar model over every word it touches.
    """
    lanes_per_phase = 128 // vec_bytes
    total = 0
    for p in range(0, lanes, lanes_per_phase):
        words = set()
        for t in range(p, min(p + lanes_per_phase, lanes)):
            base = byte_addr_of_lane(t)
            for w in range(vec_bytes // 4):
                words.add(base // 4 + w)
        per_bank: dict[int, set] = {}
        for w in words:
            per_bank.setdefault(w % 32, set()).add(w)
        total += max(len(s) for s in per_bank.values())
    return total


def fp32_simt_peak_tflops(sms: int, sm_mhz: float, fp32_lanes_per_sm: int = 128) -> float:
    """FP32 FMA-pipe peak: SMs x lanes x 2 flop x clock."""
    return sms * fp32_lanes_per_sm * 2 * sm_mhz * 1e6 / 1e12


def tflops(flops: float, seconds: float) -> float:
    return flops / seconds / 1e12


def traffic_table(N: int, tiles: Iterable[tuple[int, int]] = ((16, 16), (32, 32), (64, 64), (128, 128))):
    """Rows (scheme, DRAM read bytes, flop/byte) for an N^3 FP32 GEMM."""
    flops = gemm_flops(N, N, N)
    rows = [("naive", naive_read_bytes(N, N, N), flops / naive_read_bytes(N, N, N))]
    for bm, bn in tiles:
        b = block_tile_read_bytes(N, N, N, bm, bn)
        rows.append((f"{bm}x{bn}", b, flops / b))
    return rows
