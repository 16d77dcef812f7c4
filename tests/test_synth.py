"""Properties of the seeded input generator (host side)."""
import numpy as np
import scipy.stats
import torch

from synth import gen


def test_normals_are_standard_normal_and_deterministic():
    z = gen.normals(5, 3, gen.gate_up_tensor(7), 200_000)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1) < 0.01
    assert scipy.stats.kstest(z, "norm").pvalue > 1e-3
    assert np.array_equal(z, gen.normals(5, 3, gen.gate_up_tensor(7), 200_000))
    # any window of the stream equals the same slice of the whole stream
    for start, n in [(1, 10), (2, 7), (12345, 999), (3, 1)]:
        assert np.array_equal(gen.normals(5, 3, 9, n, start), gen.normals(5, 3, 9, start + n)[start:])


def test_streams_are_independent():
    a = gen.normals(1, 0, 100, 50_000)
    for other in [gen.normals(2, 0, 100, 50_000), gen.normals(1, 1, 100, 50_000), gen.normals(1, 0, 101, 50_000)]:
        assert abs(np.corrcoef(a, other)[0, 1]) < 0.02


def test_bf16_rounding_matches_torch():
    f = np.random.default_rng(0).normal(0, 3, 100_000).astype(np.float32)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(gen.f32_to_bf16_bits(f), ref)


def test_x_is_rms_normalised():
    x = gen.bf16_bits_to_f32(gen.x_gaussian(11, 16)).astype(np.float64)
    rms = np.sqrt((x * x).mean(1))
    assert np.allclose(rms, 1.0, atol=5e-3)


def test_clustered_tokens_share_clusters():
    x, cid = gen.x_clustered(13, 64)
    xf = gen.bf16_bits_to_f32(x).astype(np.float64)
    xn = xf / np.linalg.norm(xf, axis=1, keepdims=True)
    cos = xn @ xn.T
    same = cid[:, None] == cid[None, :]
    off = ~np.eye(64, dtype=bool)
    assert cos[same & off].mean() > 0.8 and abs(cos[~same].mean()) < 0.1
    assert set(cid.tolist()) <= {0, 1, 2, 3}


def test_e4m3_encoder_matches_torch_cast():
    v = np.abs(np.random.default_rng(1).normal(0, 50, 50_000)).astype(np.float32)
    v = np.concatenate([v, np.float32([0, 2 ** -10, 2 ** -9, 0.0029296875, 448, 440, 464])])
    v = v[v <= 448]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(gen.e4m3_encode_rn_sat(v), ref)
    assert gen.e4m3_encode_rn_sat(np.float32([1000.0]))[0] == 0x7E


def test_e2m1_encoder_ties_to_even():
    vals = np.float32([0, 0.25, 0.5, 0.75, 1, 1.25, 1.5, 1.75, 2, 2.5, 3, 3.5, 4, 5, 6, 7, -0.75, -5.0, -0.1])
    codes = gen.e2m1_encode_rn(vals)
    assert codes.tolist() == [0, 0, 1, 2, 2, 2, 3, 4, 4, 4, 5, 6, 6, 6, 7, 7, 10, 14, 0]
