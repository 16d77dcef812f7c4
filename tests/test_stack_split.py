"""Host checks of the persistent stack kernel's static plan (csrc/stack_decode.cu,
compiled as host code): the routed gate/up units are dealt to the CTAs in
contiguous, non-decreasing ranges that cover every unit exactly once, every
CTA gets the same number of gate/up units to within one, and the shared-memory layout
fits the device limit with a ring deep enough for every T <= 8."""
import os
import shutil
import subprocess

import numpy as np
import pytest

from sparse_moe_transformer_03_b300 import build as flint_build

CSRC = os.path.join(os.path.dirname(flint_build.__file__), "csrc")
PROG = r"""
#include "stack_decode.cu"
#include <cstdio>
int main() {
    using namespace flint;
    for (int G : {128, 132, 148, 160, 256})
        for (int U = 1; U <= 48; ++U) {
            std::printf("R %d %d", G, U);
            for (int c = -1; c < G; ++c) std::printf(" %d", sk_rcum(c, G, U));
            std::printf("\n");
        }
    for (int nv = 0; nv < 2; ++nv)
        for (int T = 1; T <= 8; ++T) {
            SkLayout L = sk_layout(T, 232448, nv != 0);
            std::printf("L %d %d %d %u %u %u\n", nv, T, L.nslot, L.ubuf_off, L.sh_off, L.total);
        }
    return 0;
}
"""


@pytest.fixture(scope="module")
def plan(tmp_path_factory):
    nvcc = flint_build.nvcc()
    if not shutil.which(nvcc) and not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    d = tmp_path_factory.mktemp("stack_split")
    src, exe = d / "plan.cu", d / "plan"
    src.write_text(PROG)
    subprocess.check_call([nvcc, *flint_build.ARCH, "-std=c++17", "--expt-relaxed-constexpr", "-I", CSRC,
                           "-I", os.path.join(CSRC, "..", "..", "include"), "-o", str(exe), str(src)])
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.splitlines()
    ranges, layouts = {}, {}
    for ln in out:
        f = ln.split()
        if f[0] == "R":
            ranges[(int(f[1]), int(f[2]))] = np.array(f[3:], dtype=np.int64)
        else:
            layouts[(int(f[1]), int(f[2]))] = tuple(int(v) for v in f[3:])
    return ranges, layouts


def test_routed_units_are_dealt_once_in_order(plan):
    ranges, _ = plan
    for (G, U), r in ranges.items():
        assert r[0] == 0 and r[-1] == 64 * U, (G, U)
        assert (np.diff(r) >= 0).all(), (G, U)


def test_every_cta_gets_about_the_same_gate_up_units(plan):
    """Gate/up units per CTA (routed ones of its range plus its shared one,
    CTA c < 64): the work that precedes the activation barrier."""
    ranges, _ = plan
    for (G, U), r in ranges.items():
        c = np.arange(G)
        units = np.diff(r) + (c < 64)
        mean = 64 * (U + 1) / G
        assert units.max() - mean < 1.0 and mean - units.min() < 1.0, (G, U, units.min(), units.max(), mean)


def test_shared_memory_fits_with_a_deep_ring(plan):
    """bf16 slots are 16 KiB tensor boxes, NVFP4 slots 4608-byte chunks; the
    ring holds at least two gate/up units (8 / 16 slots)."""
    _, layouts = plan
    for (nv, T), (nslot, ubuf_off, sh_off, total) in layouts.items():
        assert total <= 232448, (nv, T)
        assert nslot >= (16 if nv else 8), (nv, T, nslot)
        assert ubuf_off >= nslot * (4608 if nv else 16384) and ubuf_off % 128 == 0
