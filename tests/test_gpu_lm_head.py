"""The 4-bit output layer (flint_lm_head_*) against the fp64 oracle on the
same NVFP4 codes.

Bar (from the arithmetic, not from a run): every weight code x block scale
is exact in f16, x is staged as f16 x 2^e_t (exact for bf16 values within 28
binades of the token's largest), the MMA accumulates 2048 exact products in
fp32 and one fp32 multiply applies s_tensor x 2^-e_t.  The error is fp32
accumulation alone: |err| <= 2048 x 2^-23 x sum_h |x_h W_vh| in the worst
case, about 2^-23 x sqrt(2048) x that sum for random signs.  The test bounds
every logit by 2^-10 x sum_h |x_h W_vh| (a quarter of the worst case) and
the relative L2 error of each call by 1e-5."""
import numpy as np
import pytest
import torch

import oracle
from sparse_moe_transformer_03_b300 import flint
from synth import device, gen
from tests.gpu_common import to_dev_bf16, x_for

pytestmark = pytest.mark.gpu

V_FULL = 131072          # the assumed vocabulary (not on the pages): 2^17 rows


class Head:
    """A seeded bf16 head [V][2048] quantised to NVFP4 on the device, its
    handle and the oracle's view of the same codes."""

    def __init__(self, V, seed=3):
        device.build()
        w = torch.empty((V, gen.H), dtype=torch.bfloat16, device="cuda")
        device.fill_normal_bf16(w, seed, 0, gen.T_LM_HEAD, gen.WEIGHT_STD)
        pk, sc, ts = device.nvfp4_quantize(w)
        del w
        self.V = V
        self.ts = float(ts[0].item())
        self.h = flint.flint_lm_head_create((pk[0], sc[0], self.ts), V)
        self.pk, self.sc = pk[0].cpu().numpy(), sc[0].cpu().numpy()
        self.mat = oracle.Mat(packed=self.pk, scales=self.sc, tensor_scale=self.ts)
        self.absmat = oracle.Mat(packed=self.pk & 0x77, scales=self.sc & 0x7F, tensor_scale=abs(self.ts))

    def logits(self, xb):
        T = xb.shape[0]
        x = to_dev_bf16(xb)
        out = torch.full((T, self.V), float("nan"), dtype=torch.float32, device="cuda")
        flint.flint_lm_head_forward(self.h, x, T, out)
        torch.cuda.synchronize()
        return out.cpu().numpy().astype(np.float64)

    def check(self, xb, got, rows=None):
        ref = oracle.lm_head(xb, self.mat, rows)
        # sum_h |x_h| |W_vh|: the oracle on |x| and on the codes with their sign bits cleared
        xa = xb & np.uint16(0x7FFF)
        mag = oracle.lm_head(xa, self.absmat, rows)
        g = got if rows is None else got[:, rows]
        assert np.isfinite(g).all()
        err = np.abs(g - ref)
        rel_l2 = np.linalg.norm(g - ref) / np.linalg.norm(ref)
        worst = float((err / np.maximum(mag, 1e-30)).max())
        assert (err <= 2.0 ** -10 * mag).all(), worst
        assert rel_l2 <= 1e-5, rel_l2
        return {"rel_l2": float(rel_l2), "worst_err_over_abs_sum": worst}

    def close(self):
        flint.flint_lm_head_destroy(self.h)


@pytest.fixture(scope="module")
def small():
    hd = Head(2160)          # 135 units: fewer units than SMs, one per CTA
    yield hd
    hd.close()


@pytest.fixture(scope="module")
def ragged():
    hd = Head(16016, seed=4)  # 1001 units: ragged per-CTA ranges and a partial last round
    yield hd
    hd.close()


@pytest.fixture(scope="module")
def full():
    hd = Head(V_FULL, seed=5)
    yield hd
    hd.close()


@pytest.mark.parametrize("T,kind", [(1, "gauss"), (3, "gauss"), (8, "clustered"), (9, "gauss"),
                                    (17, "clustered"), (32, "gauss")])
def test_small_head_every_logit(small, T, kind):
    xb = x_for(kind, 800 + T, T)
    print(small.check(xb, small.logits(xb)))


@pytest.mark.parametrize("T", [1, 8, 25, 32])
def test_ragged_head_every_logit(ragged, T):
    xb = x_for("gauss", 900 + T, T)
    print(ragged.check(xb, ragged.logits(xb)))


def sampled_rows(V, grid=148, extra=512, seed=0):
    """Each CTA's first and last unit's rows plus random rows."""
    units = V // 16
    rows = []
    for c in range(grid):
        u0, u1 = units * c // grid, units * (c + 1) // grid
        rows += [16 * u0, 16 * u0 + 15, 16 * u1 - 16, 16 * u1 - 1]
    rows += list(np.random.default_rng(seed).integers(0, V, extra))
    return np.unique(np.array(rows, dtype=np.int64))


@pytest.mark.parametrize("T", [1, 32])
def test_full_vocabulary_sampled_rows(full, T):
    """V = 2^17 in the configuration the benchmark times: sampled rows."""
    xb = x_for("gauss", 950 + T, T)
    got = full.logits(xb)
    print(full.check(xb, got, sampled_rows(full.V)))


def test_repeat_is_bit_identical_and_arguments(small):
    xb = x_for("clustered", 31, 32)
    a = small.logits(xb)
    assert np.array_equal(a, small.logits(xb))
    x = to_dev_bf16(xb)
    out = torch.empty((33, small.V), dtype=torch.float32, device="cuda")
    with pytest.raises(flint.FlintError):
        flint.flint_lm_head_forward(small.h, x, 33, out)          # T above the limit
    with pytest.raises(flint.FlintError):
        flint.flint_lm_head_forward(small.h, x, 0, out)
