"""The decode activation layout (act_index in csrc/flint_common.cuh), compiled
from the library's own header as host code and run on the CPU.

The gate/up kernels write a = silu(g) * u through act_index; the down kernels
copy one token tile (8 pairs x one 256-column half) with a single 4 KiB bulk
copy and read its MMA B fragments with the row's chunk swizzle.  These tests
pin the properties that contract relies on: every (pair, column) has its own
element inside the buffer, a tile is one contiguous 4 KiB range for any first
pair, and the fragment reads of the 8 rows of a tile fall in 32 distinct
shared-memory banks."""
import os
import shutil
import subprocess

import numpy as np
import pytest

from sparse_moe_transformer_03_b300 import build as flint_build

CSRC = os.path.join(os.path.dirname(flint_build.__file__), "csrc")
PAIRS = 32 * 7          # DEC_PAIRS: T <= 32 tokens x (6 routed + shared)
ROWS = PAIRS + 8        # DEC_ACT_ROWS
PROG = r"""
#include <cstdio>
#include "flint_common.cuh"
int main() {
    static_assert(flint::DEC_ACT_ROWS == %d, "rows");
    std::printf("%%zu\n", flint::DEC_ACT_BYTES);
    for (int p = 0; p < flint::DEC_ACT_ROWS; ++p)
        for (int j = 0; j < flint::I; ++j) std::printf("%%zu\n", flint::act_index(p, j));
    return 0;
}
""" % ROWS


@pytest.fixture(scope="module")
def table(tmp_path_factory):
    nvcc = flint_build.nvcc()
    if not shutil.which(nvcc) and not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    d = tmp_path_factory.mktemp("act_layout")
    src, exe = d / "act.cu", d / "act"
    src.write_text(PROG)
    subprocess.check_call([nvcc, "-std=c++17", "-I", CSRC, "-o", str(exe), str(src)])
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()
    nbytes = int(out[0])
    idx = np.array(out[1:], dtype=np.int64).reshape(ROWS, 512)
    return nbytes, idx


def test_every_element_has_its_own_place_in_the_buffer(table):
    nbytes, idx = table
    assert nbytes == 2 * ROWS * 256 * 2          # two halves of [ROWS][256] bf16
    flat = idx.ravel()
    assert flat.min() >= 0 and flat.max() < nbytes // 2
    assert len(np.unique(flat)) == flat.size      # one-to-one


@pytest.mark.parametrize("half", [0, 1])
def test_a_token_tile_is_one_contiguous_4kib_copy(table, half):
    _, idx = table
    for p0 in range(0, PAIRS):                    # any first pair of a tile that starts inside the batch
        tile = idx[p0:p0 + 8, 256 * half:256 * (half + 1)]
        base = (half * ROWS + p0) * 256
        assert sorted(tile.ravel().tolist()) == list(range(base, base + 8 * 256)), (p0, half)
        # row g of the tile is the g-th 512-byte run
        for g in range(8):
            assert tile[g].min() == base + 256 * g and tile[g].max() == base + 256 * g + 255


@pytest.mark.parametrize("half", [0, 1])
def test_fragment_reads_of_a_tile_use_32_distinct_banks(table, half):
    """Lane (g, cq) of a warp reads the 4-byte word holding columns kb*16 + 2cq,
    +1 (first B register) and kb*16 + 8 + 2cq, +1 (second) of row g."""
    _, idx = table
    for p0 in range(0, PAIRS, 3):
        base = (half * ROWS + p0) * 256
        for kb in range(16):
            for off in (0, 8):
                banks = set()
                for g in range(8):
                    for cq in range(4):
                        j = 256 * half + kb * 16 + off + 2 * cq
                        e0, e1 = idx[p0 + g, j] - base, idx[p0 + g, j + 1] - base
                        assert e1 == e0 + 1 and e0 % 2 == 0          # both columns in one 4-byte word
                        banks.add((e0 * 2 // 4) % 32)
                assert len(banks) == 32, (p0, kb, off)
