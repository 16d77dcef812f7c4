"""Capacity of the decode kernels' per-CTA work-item lists, checked on the
host: the item count of a batch is DEC_UNITS x (its 8-token tiles), and no
routing of T <= 32 tokens can give a CTA of the smallest gate/up grid more
items than its list holds.  So the kernels' FLINT_ERR_INTERNAL path (an item
list that does not fit) cannot be reached by any input.  The constants are
read from the library's own header, compiled as host code."""
import os
import shutil
import subprocess
from collections import Counter

import numpy as np
import pytest

from sparse_moe_transformer_03_b300 import build as flint_build

CSRC = os.path.join(os.path.dirname(flint_build.__file__), "csrc")
PROG = r"""
#include <cstdio>
#include "routing.cuh"
int main() {
    std::printf("%d %d %d %d %d %d\n", flint::DEC_UNITS, flint::DEC_MAX_TILES, flint::DEC_MAX_CTA_ITEMS,
                flint::DEC_MIN_GRID, flint::DEC_T, flint::TOPK);
    return 0;
}
"""


@pytest.fixture(scope="module")
def consts(tmp_path_factory):
    nvcc = flint_build.nvcc()
    if not shutil.which(nvcc) and not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    d = tmp_path_factory.mktemp("capacity")
    src, exe = d / "cap.cu", d / "cap"
    src.write_text(PROG)
    subprocess.check_call([nvcc, *flint_build.ARCH, "-std=c++17", "-I", CSRC, "-o", str(exe), str(src)])
    units, max_tiles, max_items, min_grid, dec_t, topk = map(
        int, subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split())
    return dict(units=units, max_tiles=max_tiles, max_items=max_items, min_grid=min_grid, dec_t=dec_t, topk=topk)


def tiles_of(T, idx):
    """8-token tiles of a batch: the shared slot's ceil(T/8), then each
    touched expert's ceil(tokens/8) (the table builder's slot_tile0 scan)."""
    counts = Counter(np.asarray(idx).ravel().tolist())
    return (T + 7) // 8 + sum((n + 7) // 8 for n in counts.values())


def spread_routing(T, rng):
    """Every token takes 6 experts no other token takes while experts last
    (the most distinct experts, each with one token: the most tiles)."""
    perm = rng.permutation(256)
    return np.array([[perm[(6 * t + j) % 256] for j in range(6)] for t in range(T)])


def test_worst_case_routing_fits_every_cta_list(consts):
    rng = np.random.default_rng(0)
    for T in range(1, consts["dec_t"] + 1):
        worst = tiles_of(T, spread_routing(T, rng))
        assert worst <= consts["max_tiles"], T
        items = consts["units"] * worst
        per_cta = -(-items // consts["min_grid"])       # CTA 0 gets the most: ceil(items / G)
        assert per_cta <= consts["max_items"], (T, per_cta)


def test_random_and_clustered_routings_stay_below_the_bound(consts):
    rng = np.random.default_rng(1)
    for _ in range(2000):
        T = int(rng.integers(1, consts["dec_t"] + 1))
        pool = int(rng.integers(6, 257))
        idx = np.stack([rng.choice(pool, 6, replace=False) for _ in range(T)])
        assert tiles_of(T, idx) <= consts["max_tiles"]


def test_bound_is_reached(consts):
    """The bound is tight: 32 tokens on 192 distinct experts reach it."""
    rng = np.random.default_rng(2)
    T = consts["dec_t"]
    assert tiles_of(T, spread_routing(T, rng)) == consts["max_tiles"]
