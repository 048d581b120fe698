"""The grouped tile raster (csrc/tile_order.cuh), checked on the host (no GPU).

The tensor-core kernel and the split-K reduction both map a tile index t to
(tile row, tile column) through tile_coords; a mistake there computes some
tiles twice and leaves others unwritten.  The header is host-compilable, so a
small C++ program includes it and checks, for every grid of 1..64 x 1..64
tiles and group heights 1..20 (ragged last groups included), that t ->
(tm, tn) is a bijection onto the grid, that a group covers `group_m` tile
rows (fewer in the last group) and is walked down its rows first, and that
groups follow one another top to bottom."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "tiled_tensor_core_gemm_gb300", "csrc")

PROGRAM = r"""
#define __host__
#define __device__
#define __forceinline__ inline
#include "tile_order.cuh"
#include <cstdio>
#include <vector>

int main() {
    long checked = 0;
    for (int tiles_m = 1; tiles_m <= 64; ++tiles_m)
        for (int tiles_n = 1; tiles_n <= 64; ++tiles_n)
            for (int group_m = 1; group_m <= 20; ++group_m) {
                const int tiles = tiles_m * tiles_n;
                std::vector<int> seen(tiles, 0);
                int prev_tm = -1, prev_tn = 0, prev_g = 0;
                for (int t = 0; t < tiles; ++t) {
                    int tm = -1, tn = -1;
                    tcgemm::tile_coords(t, tiles_m, tiles_n, group_m, tm, tn);
                    if (tm < 0 || tm >= tiles_m || tn < 0 || tn >= tiles_n) {
                        printf("out of range: grid %dx%d group %d t %d -> (%d, %d)\n", tiles_m, tiles_n, group_m, t, tm, tn);
                        return 1;
                    }
                    if (seen[tm * tiles_n + tn]++) {
                        printf("tile visited twice: grid %dx%d group %d t %d -> (%d, %d)\n", tiles_m, tiles_n, group_m, t, tm, tn);
                        return 1;
                    }
                    const int g = tm / group_m;                 // the group of tile rows tm falls in
                    const int first = g * group_m;
                    const int rows = tiles_m - first < group_m ? tiles_m - first : group_m;
                    if (t > 0) {
                        const bool same_group = g == prev_g;
                        // inside a group: next row in the same column, or the group's first row of the next column
                        const bool down = same_group && tn == prev_tn && tm == prev_tm + 1;
                        const bool across = same_group && tn == prev_tn + 1 && tm == first && prev_tm == first + rows - 1;
                        // next group: its first row, first column, after the previous group's last tile
                        const bool next = g == prev_g + 1 && tm == first && tn == 0 && prev_tn == tiles_n - 1;
                        if (!(down || across || next)) {
                            printf("order broken: grid %dx%d group %d t %d -> (%d, %d) after (%d, %d)\n", tiles_m, tiles_n,
                                   group_m, t, tm, tn, prev_tm, prev_tn);
                            return 1;
                        }
                    } else if (tm != 0 || tn != 0) {
                        printf("tile 0 is not (0, 0)\n");
                        return 1;
                    }
                    prev_tm = tm, prev_tn = tn, prev_g = g;
                    ++checked;
                }
            }
    printf("ok %ld\n", checked);
    return 0;
}
"""


@pytest.mark.skipif(shutil.which("g++") is None, reason="needs g++")
def test_tile_raster_is_a_grouped_bijection(tmp_path):
    src = tmp_path / "tile_order_check.cc"
    exe = tmp_path / "tile_order_check"
    src.write_text(PROGRAM)
    subprocess.run(["g++", "-O2", "-std=c++17", "-I", CSRC, str(src), "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.startswith("ok ")
