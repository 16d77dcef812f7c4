"""Pins of the oracle's output-layer GEMV (oracle.lm_head) to things outside
the oracle: closed forms on matrices with one nonzero weight per row, the
published E2M1 code table with torch's float8 E4M3 decoding and a library
matmul, and the row-subset contract.  A dropped tensor scale, a swapped
nibble, a transposed operand or a wrong row index fails one of them."""
import os

import numpy as np
import pytest
import torch

import oracle
from synth import gen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
E4M3_ONE = 0x38          # E4M3 code of 1.0: exponent field 7 (bias 7), mantissa 0


def e2m1_table():
    """Code -> value from the OCP MX table (tests/golden/e2m1_values.txt)."""
    vals = {}
    for ln in open(os.path.join(GOLDEN, "e2m1_values.txt")):
        if ln.startswith("#") or not ln.strip():
            continue
        c, v = ln.split()
        vals[int(c, 16)] = float(v)
    return np.array([vals[c] for c in range(16)])


def e4m3_values(codes):
    """E4M3 codes -> float64 through torch's float8_e4m3fn."""
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def x_bits(seed, T, H):
    return gen.normal_bf16(seed, 0, gen.T_X, (T, H), 1.0)


def x_values(bits):
    return gen.bf16_bits_to_f32(bits).astype(np.float64)


def test_one_weight_per_row_picks_that_column():
    """Row v holds a single code at column j_v (1.0 or -1.0, even and odd
    nibbles, several 16-column blocks), block scale 1.0, tensor scale 0.5:
    logits[t][v] = +-0.5 * x[t][j_v] exactly."""
    V, H, T = 9, 64, 4
    cols = [0, 1, 15, 16, 17, 31, 32, 62, 63]
    sign = [1, -1, 1, 1, -1, 1, -1, 1, -1]
    packed = np.zeros((V, H // 2), dtype=np.uint8)
    scales = np.full((V, H // 16), E4M3_ONE, dtype=np.uint8)
    for v, (j, sg) in enumerate(zip(cols, sign)):
        code = 0x2 if sg > 0 else 0xA           # +1.0 / -1.0
        packed[v, j // 2] = code if j % 2 == 0 else code << 4
    xb = x_bits(3, T, H)
    got = oracle.lm_head(xb, oracle.Mat(packed=packed, scales=scales, tensor_scale=0.5))
    want = 0.5 * x_values(xb)[:, cols] * np.array(sign)
    assert got.shape == (T, V)
    assert np.array_equal(got, want)


def test_block_scales_weight_their_own_16_columns():
    """Every code 1.0, block b scaled by 2^(b-2): logits = sum over blocks of
    2^(b-2) * (sum of x over the block's 16 columns)."""
    V, H, T = 3, 128, 2
    packed = np.full((V, H // 2), 0x22, dtype=np.uint8)           # 1.0 in both nibbles
    scales = np.zeros((V, H // 16), dtype=np.uint8)
    for b in range(H // 16):
        scales[:, b] = (b - 2 + 7) << 3                           # 2^(b-2)
    xb = x_bits(4, T, H)
    got = oracle.lm_head(xb, oracle.Mat(packed=packed, scales=scales, tensor_scale=1.0))
    xs = x_values(xb).reshape(T, H // 16, 16).sum(axis=2)
    want = (xs * 2.0 ** (np.arange(H // 16) - 2)).sum(axis=1)
    assert np.allclose(got, want[:, None], rtol=1e-14, atol=0)


def test_random_matrix_against_table_decode_and_matmul():
    """Random codes and scales: the oracle equals x @ W^T with W decoded from
    the published E2M1 table and torch's E4M3 (numpy float64 matmul)."""
    rng = np.random.default_rng(7)
    V, H, T = 37, 96, 5
    packed = rng.integers(0, 256, (V, H // 2), dtype=np.uint8)
    scales = rng.integers(0, 0x7F, (V, H // 16), dtype=np.uint8)   # finite E4M3 codes
    ts = np.float32(0.013)
    tab = e2m1_table()
    codes = np.empty((V, H), dtype=np.uint8)
    codes[:, 0::2] = packed & 0xF
    codes[:, 1::2] = packed >> 4
    W = tab[codes] * np.repeat(e4m3_values(scales), 16, axis=1) * float(ts)
    xb = x_bits(5, T, H)
    got = oracle.lm_head(xb, oracle.Mat(packed=packed, scales=scales, tensor_scale=ts))
    want = x_values(xb) @ W.T
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12 * np.abs(want).max())


def test_bf16_matrix_and_row_subset():
    """A bf16 head: equals the widened matmul; a row subset returns exactly
    those columns of the full result, in the order asked."""
    V, H, T = 21, 64, 3
    Wb = gen.normal_bf16(9, 0, gen.T_LM_HEAD, (V, H), 0.02)
    xb = x_bits(6, T, H)
    full = oracle.lm_head(xb, oracle.Mat(bf16=Wb))
    want = x_values(xb) @ gen.bf16_bits_to_f32(Wb).astype(np.float64).T
    assert np.allclose(full, want, rtol=1e-12, atol=1e-14)
    rows = np.array([20, 0, 7, 7, 13])
    sub = oracle.lm_head(xb, oracle.Mat(bf16=Wb), rows=rows)
    assert np.array_equal(sub, full[:, rows])
    with pytest.raises(AssertionError):
        oracle.lm_head(xb, oracle.Mat(bf16=Wb), rows=[V])
