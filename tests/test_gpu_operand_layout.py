"""The shared-memory operand layouts the tensor-core kernel relies on,
measured on the GPU and checked against their closed forms.

A probe program (tests/probes/operand_layout.cu) runs one tcgen05.mma per
descriptor with a one-hot A and a B region whose every element holds its own
index, so the product tells which shared-memory element the MMA read for each
(k, n); and it TMA-loads a box of values equal to their global index, so the
shared-memory image tells where the TMA engine put each element.  The kernel
needs the two to agree for every way it stages B: as stored with the
128-byte swizzle of 16-byte units (16-bit inputs), as stored with the 128-byte
swizzle of 32-byte units (TF32: atoms of 4 K-rows, 512 bytes apart), and
K-major.
"""
import os
import subprocess

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "probes", "operand_layout.cu")
EXE = os.path.join(HERE, "probes", "_build", "operand_layout")


@pytest.fixture(scope="module")
def probe():
    os.makedirs(os.path.dirname(EXE), exist_ok=True)
    if not os.path.exists(EXE) or os.path.getmtime(EXE) < os.path.getmtime(SRC):
        nvcc = os.environ.get("NVCC", "nvcc")
        subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17", "-o", EXE, SRC],
                       check=True)
    r = subprocess.run([EXE], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    out = {}
    for line in r.stdout.splitlines():
        name, *vals = line.split()
        out[name] = np.array([int(v) for v in vals], dtype=np.int64)
    return out


def _mma_bytes(probe, name, n_cols, uk, elem):
    """Byte offset the MMA read for each (k, n), checked consistent over the
    rows m that share k = m % uk."""
    idx = probe[name].reshape(128, n_cols)
    assert np.all(idx >= 0), name
    for m in range(uk, 128):
        assert np.array_equal(idx[m], idx[m % uk]), (name, m)
    return idx[:uk] * elem


@pytest.mark.parametrize("name,lbo,sbo,n_cols", [("umma_bf16_mn_sw128_lbo2048_sbo1024_n128", 2048, 1024, 128)])
def test_mma_reads_16_bit_b_as_stored_from_16_byte_units(probe, name, lbo, sbo, n_cols):
    got = _mma_bytes(probe, name, n_cols, 16, 2)
    k, n = np.meshgrid(np.arange(16), np.arange(n_cols), indexing="ij")
    want = (n // 64) * lbo + (k // 8) * sbo + (k % 8) * 128 + (((n % 64) // 8) ^ (k % 8)) * 16 + (n % 8) * 2
    assert np.array_equal(got, want)


@pytest.mark.parametrize("name,lbo,sbo,n_cols", [("umma_tf32_mn_sw128a32_lbo2048_sbo1024_n64", 2048, 1024, 64),
                                                 ("umma_tf32_mn_sw128a32_lbo4096_sbo512_n128", 4096, 512, 128)])
def test_mma_reads_tf32_b_as_stored_from_32_byte_units(probe, name, lbo, sbo, n_cols):
    """Atoms of 4 K-rows of 128 bytes; row r's 32-byte units permuted by r % 4;
    32-column chunks LBO apart, atoms SBO apart."""
    got = _mma_bytes(probe, name, n_cols, 8, 4)
    k, n = np.meshgrid(np.arange(8), np.arange(n_cols), indexing="ij")
    want = (n // 32) * lbo + (k // 4) * sbo + (k % 4) * 128 + (((n % 32) // 8) ^ (k % 4)) * 32 + (n % 8) * 4
    assert np.array_equal(got, want)


@pytest.mark.parametrize("name,uk,elem", [("umma_bf16_k_sw128_n64", 16, 2), ("umma_tf32_k_sw128_n64", 8, 4)])
def test_mma_reads_k_major_b(probe, name, uk, elem):
    got = _mma_bytes(probe, name, 64, uk, elem)
    k, n = np.meshgrid(np.arange(uk), np.arange(64), indexing="ij")
    kb = k * elem
    want = (n // 8) * 1024 + (n % 8) * 128 + ((kb // 16) ^ (n % 8)) * 16 + kb % 16
    assert np.array_equal(got, want)


def _tma_position(probe, name):
    """Shared-memory word of box element (row, col), from the dumped image."""
    img = probe[name]
    assert sorted(img.tolist()) == sorted((r * 64 + c) for r in range(32) for c in range(32))
    pos = np.empty((32, 32), np.int64)
    for word, g in enumerate(img):
        pos[g // 64, g % 64] = word
    return pos


def test_tma_writes_16_byte_units_permuted_by_row_mod_8(probe):
    r, c = np.meshgrid(np.arange(32), np.arange(32), indexing="ij")
    assert np.array_equal(_tma_position(probe, "tma_sw128"), r * 32 + ((c // 4) ^ (r % 8)) * 4 + c % 4)


def test_tma_writes_32_byte_units_permuted_by_row_mod_4(probe):
    r, c = np.meshgrid(np.arange(32), np.arange(32), indexing="ij")
    assert np.array_equal(_tma_position(probe, "tma_sw128a32"), r * 32 + ((c // 8) ^ (r % 4)) * 8 + c % 8)


def test_tf32_b_chunk_as_the_tma_writes_it_is_what_the_mma_reads(probe):
    """A TF32 B chunk (K-rows of 32 columns, 128 bytes each) loaded with the
    32-byte-unit swizzle, read by MMAs whose descriptor starts 1024 bytes
    further per 8 K-rows with SBO 512: the byte the MMA takes for (k, n) is
    the byte the TMA wrote element (k, n) to."""
    tma_word = _tma_position(probe, "tma_sw128a32")           # (K-row, column) -> word within the box
    got = _mma_bytes(probe, "umma_tf32_mn_sw128a32_lbo4096_sbo512_n128", 128, 8, 4)
    for kstep in range(4):                                     # the 4 MMAs of a 32-row stage
        for k in range(8):
            row = 8 * kstep + k
            mma = kstep * 1024 + got[k, :32]                   # first 32 columns: one chunk
            assert np.array_equal(mma, tma_word[row] * 4), (kstep, k)
