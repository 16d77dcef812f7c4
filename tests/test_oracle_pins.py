"""Pins of the fp64 oracle against facts that do not come from the oracle.

Each test checks the oracle against a closed form, a textbook or library
routine, a brute-force evaluation written differently, an invariant of the
method, or a published table (tests/golden).  They are chosen so that a
dropped term, a wrong sign, a swapped index or a transposed operand in the
oracle fails at least one of them.
"""
import heapq
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from synth import gen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16_bits(vals):
    return gen.to_bf16_bits(np.asarray(vals, dtype=np.float64))


# ---------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------

def test_bf16_widening_matches_torch():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 2**16, size=4096, dtype=np.uint32).astype(np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]   # finite only
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    got = np.array([oracle.bf16_to_double(b) for b in bits])
    assert np.array_equal(got, ref)


def test_e4m3_decode_matches_torch_float8():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    got = np.array([oracle.e4m3_decode(c) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert nan.sum() == 2                      # S.1111.111 only
    assert np.array_equal(got[~nan], ref[~nan])
    assert oracle.e4m3_decode(0x7E) == 448.0   # largest finite
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9


def test_e2m1_decode_matches_published_table():
    rows = []
    with open(os.path.join(GOLDEN, "e2m1_values.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                c, v = line.split()
                rows.append((int(c, 16), float(v)))
    assert len(rows) == 16
    for c, v in rows:
        got = oracle.e2m1_decode(c)
        assert got == v and math.copysign(1.0, got) == math.copysign(1.0, v), (c, got, v)


def test_sigmoid_and_silu_against_scipy():
    z = np.linspace(-30, 30, 601)
    s = np.array([oracle.sigmoid(v) for v in z])
    assert np.allclose(s, scipy.special.expit(z), rtol=1e-15, atol=1e-300)
    si = np.array([oracle.silu(v) for v in z])
    assert np.allclose(si, z * scipy.special.expit(z), rtol=1e-14, atol=1e-300)
    assert oracle.sigmoid(0.0) == 0.5 and oracle.silu(0.0) == 0.0
    # symmetry sigma(-z) = 1 - sigma(z)
    assert np.allclose([oracle.sigmoid(-v) for v in z], 1.0 - s, atol=1e-15)


# ---------------------------------------------------------------------------
# router and selection
# ---------------------------------------------------------------------------

def test_router_one_hot_rows_give_textbook_top_k():
    """W_r[e] = c * e_{pi(e)} and no bias: logit[e] = c * x[pi(e)], so the
    chosen set is the 6 largest coordinates x[pi(e)] (a plain partial sort)."""
    E, H, T = 32, 64, 16
    rng = np.random.default_rng(7)
    pi = rng.permutation(H)[:E]
    c = 0.5
    Wr = np.zeros((E, H))
    Wr[np.arange(E), pi] = c
    x = gen.x_gaussian(3, T, H)
    xf = gen.bf16_bits_to_f32(x).astype(np.float64)
    l = oracle.router_logits(x, bf16_bits(Wr))
    assert np.array_equal(l, c * xf[:, pi])
    idx, w = oracle.select(l, 6)
    for t in range(T):
        top = heapq.nlargest(6, range(E), key=lambda e: (xf[t, pi[e]], -e))
        assert list(idx[t]) == top
        s = scipy.special.expit(c * xf[t, pi[top]])
        assert np.allclose(w[t], s / s.sum(), rtol=1e-14)


def test_router_bias_only_and_logits_against_numpy():
    E, H, T = 48, 96, 5
    rng = np.random.default_rng(11)
    x = gen.x_gaussian(5, T, H)
    Wr = gen.router_weight(5, 0, E, H)
    b = rng.normal(0, 0.5, E).astype(np.float32)
    l = oracle.router_logits(x, Wr, b)
    ref = gen.bf16_bits_to_f32(x).astype(np.float64) @ gen.bf16_bits_to_f32(Wr).astype(np.float64).T + b
    assert np.allclose(l, ref, rtol=1e-13, atol=1e-13)
    # with a zero router the bias alone decides
    l0 = oracle.router_logits(x, np.zeros((E, H), np.uint16), b)
    assert np.array_equal(l0, np.broadcast_to(b.astype(np.float64), (T, E)))
    idx, _ = oracle.select(l0, 6)
    assert all(list(r) == list(np.argsort(-b, kind="stable")[:6]) for r in idx)


def test_selection_invariants_and_ties():
    rng = np.random.default_rng(3)
    T, E, k = 200, 256, 6
    l = rng.normal(0, 1, (T, E))
    l[0, :] = 0.0                                 # all equal: lowest indices win
    l[1, [3, 9, 200, 201, 250, 7, 100]] = 5.0     # 7 equal maxima
    idx, w = oracle.select(l, k)
    for t in range(T):
        s = set(idx[t].tolist())
        assert len(s) == k and all(0 <= e < E for e in s)
        assert abs(w[t].sum() - 1.0) <= 1e-12
        unsel = np.delete(l[t], idx[t])
        assert l[t, idx[t]].min() >= unsel.max()
        assert np.all(w[t] > 0)
    assert list(idx[0]) == [0, 1, 2, 3, 4, 5]
    assert sorted(idx[1].tolist()) == [3, 7, 9, 100, 200, 201]
    assert np.allclose(w[0], 1.0 / 6)


# ---------------------------------------------------------------------------
# the layer: brute force, closed forms, textbook special case
# ---------------------------------------------------------------------------

def dense_brute_force(x, Wr, b, Wgu, Wd, sh, k):
    """Evaluate every expert on every token with numpy matrix products, choose
    by a full stable sort of the sigmoid scores, mask and combine."""
    xf = gen.bf16_bits_to_f32(x).astype(np.float64)
    W = gen.bf16_bits_to_f32(Wr).astype(np.float64)
    logits = xf @ W.T + (0 if b is None else b.astype(np.float64))
    scores = scipy.special.expit(logits)
    E = W.shape[0]
    T = xf.shape[0]
    mask = np.zeros((T, E))
    for t in range(T):
        order = np.argsort(-logits[t], kind="stable")
        mask[t, order[:k]] = 1.0
    gates = mask * scores
    gates /= gates.sum(axis=1, keepdims=True)

    def ffn(gu, d):
        G = gen.bf16_bits_to_f32(gu).astype(np.float64)
        D = gen.bf16_bits_to_f32(d).astype(np.float64)
        I = G.shape[0] // 2
        h = xf @ G.T
        a = h[:, :I] * scipy.special.expit(h[:, :I]) * h[:, I:]
        return a @ D.T

    y = np.zeros_like(xf)
    for e in range(E):
        y += gates[:, e:e + 1] * ffn(Wgu[e], Wd[e])
    if sh is not None:
        y += ffn(sh[0], sh[1])
    return y, mask


@pytest.mark.parametrize("E,H,I,T,with_bias", [(16, 32, 8, 8, False), (16, 32, 8, 8, True),
                                               (256, 64, 16, 4, True)])
def test_layer_matches_dense_brute_force(E, H, I, T, with_bias):
    seed = 21
    x = gen.x_gaussian(seed, T, H)
    Wr = gen.router_weight(seed, 0, E, H)
    b = gen.router_bias(seed, 0, E) if with_bias else None
    Wgu = [gen.normal_bf16(seed, 0, gen.gate_up_tensor(e), (2 * I, H), 0.2) for e in range(E)]
    Wd = [gen.normal_bf16(seed, 0, gen.down_tensor(e), (H, I), 0.2) for e in range(E)]
    sh = (gen.normal_bf16(seed, 0, gen.gate_up_tensor(E), (2 * I, H), 0.2),
          gen.normal_bf16(seed, 0, gen.down_tensor(E), (H, I), 0.2))
    r = oracle.moe_forward(x, Wr, b, [oracle.Mat(m) for m in Wgu], [oracle.Mat(m) for m in Wd],
                           (oracle.Mat(sh[0]), oracle.Mat(sh[1])), k=6)
    ref, mask = dense_brute_force(x, Wr, b, Wgu, Wd, sh, 6)
    assert np.allclose(r["y"], ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    for t in range(T):
        assert set(r["idx"][t].tolist()) == set(np.nonzero(mask[t])[0].tolist())
    # without the shared expert the result changes by exactly its output
    r2 = oracle.moe_forward(x, Wr, b, [oracle.Mat(m) for m in Wgu], [oracle.Mat(m) for m in Wd],
                            None, k=6)
    ref2, _ = dense_brute_force(x, Wr, b, Wgu, Wd, None, 6)
    assert np.allclose(r2["y"], ref2, rtol=1e-12, atol=1e-12 * np.abs(ref2).max())


def test_identity_like_experts_closed_form():
    """W_g[e][i] = alpha_e * e_{p(i)}, W_u[e][i] = beta_e * e_{p(i)},
    W_d[e][q(i)][i] = 1: then y[q(i)] = sum_j w_j beta_j x_{p(i)} silu(alpha_j x_{p(i)})
    (+ the shared expert's term) and y is zero off q(I).  p and q are distinct
    random injections, so a transposed or mis-indexed operand is caught."""
    E, H, I, T, k = 12, 40, 10, 6, 6
    rng = np.random.default_rng(5)
    p = rng.permutation(H)[:I]
    q = rng.permutation(H)[:I]
    alphas = np.array([0.5, 1.0, 1.5, 2.0, -1.0, 0.75, 1.25, 3.0, -0.5, 0.25, 2.5, 1.75])
    betas = np.array([1.0, -2.0, 0.5, 1.5, 2.0, -1.0, 0.25, 1.0, 3.0, -0.75, 0.5, 1.0])
    sa, sb = 1.5, -0.5
    x = gen.x_gaussian(9, T, H)
    xf = gen.bf16_bits_to_f32(x).astype(np.float64)
    Wr = gen.router_weight(9, 0, E, H)

    def mats(al, be):
        G = np.zeros((2 * I, H))
        G[np.arange(I), p] = al
        G[I + np.arange(I), p] = be
        D = np.zeros((H, I))
        D[q, np.arange(I)] = 1.0
        return bf16_bits(G), bf16_bits(D)

    ms = [mats(alphas[e], betas[e]) for e in range(E)]
    shm = mats(sa, sb)
    r = oracle.moe_forward(x, Wr, None, [oracle.Mat(m[0]) for m in ms], [oracle.Mat(m[1]) for m in ms],
                           (oracle.Mat(shm[0]), oracle.Mat(shm[1])), k=k)
    silu = lambda z: z * scipy.special.expit(z)
    for t in range(T):
        xp = xf[t, p]
        exp = np.zeros(H)
        for j in range(k):
            e = r["idx"][t, j]
            exp[q] += r["w"][t, j] * betas[e] * xp * silu(alphas[e] * xp)
        exp[q] += sb * xp * silu(sa * xp)
        assert np.allclose(r["y"][t], exp, rtol=1e-13, atol=1e-15)
        assert np.all(np.delete(r["y"][t], q) == 0.0)


def test_single_expert_reduces_to_x_silu_x():
    """One routed expert, k = 1, alpha = beta = 1, identity maps, no shared
    expert: the renormalised weight is 1 and y = x * silu(x) = x^2 sigma(x)."""
    H = I = 16
    T = 8
    x = gen.x_gaussian(4, T, H)
    xf = gen.bf16_bits_to_f32(x).astype(np.float64)
    G = np.vstack([np.eye(I, H), np.eye(I, H)])
    D = np.eye(H, I)
    r = oracle.moe_forward(x, gen.router_weight(4, 0, 1, H), None,
                           [oracle.Mat(bf16_bits(G))], [oracle.Mat(bf16_bits(D))], None, k=1)
    assert np.allclose(r["w"], 1.0)
    assert np.allclose(r["y"], xf * xf * scipy.special.expit(xf), rtol=1e-14, atol=0)


def test_fixed_selection_uses_that_set_and_renormalises():
    E, H, I, T = 16, 32, 8, 3
    x = gen.x_gaussian(8, T, H)
    Wr = gen.router_weight(8, 0, E, H)
    Wgu = [gen.normal_bf16(8, 0, gen.gate_up_tensor(e), (2 * I, H), 0.2) for e in range(E)]
    Wd = [gen.normal_bf16(8, 0, gen.down_tensor(e), (H, I), 0.2) for e in range(E)]
    base = oracle.moe_forward(x, Wr, None, [oracle.Mat(m) for m in Wgu], [oracle.Mat(m) for m in Wd], None)
    # the runner-up set: replace the 6th choice with the 7th-ranked expert
    alt = base["idx"].copy()
    for t in range(T):
        order = np.argsort(-base["logits"][t], kind="stable")
        alt[t, 5] = order[6]
    r = oracle.moe_forward(x, Wr, None, [oracle.Mat(m) for m in Wgu], [oracle.Mat(m) for m in Wd], None,
                           idx_in=alt)
    assert np.array_equal(r["idx"], alt)
    s = scipy.special.expit(np.take_along_axis(base["logits"], alt.astype(np.int64), 1))
    assert np.allclose(r["w"], s / s.sum(1, keepdims=True), rtol=1e-14)
    assert not np.allclose(r["y"], base["y"])


def test_absent_selected_expert_is_an_error():
    E, H, I = 8, 16, 4
    x = gen.x_gaussian(2, 1, H)
    with pytest.raises(ValueError):
        oracle.moe_forward(x, gen.router_weight(2, 0, E, H), None,
                           [oracle.Mat.absent()] * E, [oracle.Mat.absent()] * E, None)


# ---------------------------------------------------------------------------
# permutation
# ---------------------------------------------------------------------------

def test_permutation_is_a_stable_counting_sort():
    rng = np.random.default_rng(2)
    T, k, E = 300, 6, 256
    idx = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    off, gat = oracle.permutation(idx, E)
    flat = idx.ravel()
    assert np.array_equal(gat, np.argsort(flat, kind="stable"))
    assert np.array_equal(off, np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=E))]))


# ---------------------------------------------------------------------------
# NVFP4
# ---------------------------------------------------------------------------

def test_nvfp4_dequant_of_exactly_representable_matrix_is_lossless():
    """Build a matrix whose elements are e2m1 values times an E4M3 block scale
    times a power-of-two tensor scale, such that the encoder's own choices
    (s_t = amax / (6*448), s_b = amax_b / (6*s_t)) land on those scales
    exactly; encoding then decoding must give the matrix back bit for bit."""
    R, K = 8, 64
    rng = np.random.default_rng(12)
    e2m1 = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    codes = rng.integers(0, 8, (R, K))
    sign = rng.choice([-1.0, 1.0], (R, K))
    vals = sign * e2m1[codes]
    vals[:, ::16] = 6.0 * sign[:, ::16]           # every block reaches |q| = 6
    s_t = 2.0 ** -6
    bs = 2.0 ** rng.integers(-3, 6, (R, K // 16)).astype(np.float64)
    bs[0, 0] = 448.0                              # largest block: amax = 6 * 448 * s_t
    w = vals * np.repeat(bs, 16, axis=1) * s_t
    bits = bf16_bits(w)
    assert np.array_equal(gen.bf16_bits_to_f32(bits), w.astype(np.float32))
    packed, scales, ts = gen.nvfp4_quantize(bits)
    assert float(ts) == s_t
    assert np.array_equal([[oracle.e4m3_decode(c) for c in row] for row in scales], bs)
    deq = oracle.nvfp4_dequant(packed, scales, ts)
    assert np.array_equal(deq, w)


def test_nvfp4_roundtrip_error_within_half_step():
    R, K = 16, 256
    bits = gen.normal_bf16(30, 0, gen.gate_up_tensor(0), (R, K), 0.02)
    w = gen.bf16_bits_to_f32(bits).astype(np.float64)
    packed, scales, ts = gen.nvfp4_quantize(bits)
    deq = oracle.nvfp4_dequant(packed, scales, ts)
    blk_scale = np.repeat(np.array([[oracle.e4m3_decode(c) for c in row] for row in scales]), 16, 1) * float(ts)
    # e2m1 spacing: 0.5 below 2, 1 in [2, 4), 2 in [4, 6]; clamp error is 0 as |w|/scale <= 6 (+rounding)
    mag = np.abs(w) / blk_scale
    half_step = np.where(mag < 2, 0.25, np.where(mag < 4, 0.5, 1.0)) * blk_scale
    assert np.all(np.abs(deq - w) <= half_step * (1 + 1e-6) + 1e-12)
    rel = np.linalg.norm(deq - w) / np.linalg.norm(w)
    assert rel < 0.15


def test_nvfp4_layer_uses_dequantised_weights():
    """The oracle on NVFP4 matrices equals the oracle on bf16 matrices that hold
    the same (exactly representable) dequantised values."""
    E, H, I, T = 8, 64, 16, 3
    x = gen.x_gaussian(31, T, H)
    Wr = gen.router_weight(31, 0, E, H)
    q_gu, q_d, b_gu, b_d = [], [], [], []
    for e in range(E):
        for (shape, tens, qs, bs) in [((2 * I, H), gen.gate_up_tensor(e), q_gu, b_gu),
                                      ((H, I), gen.down_tensor(e), q_d, b_d)]:
            bits = gen.normal_bf16(31, 0, tens, shape, 0.02)
            pk, sc, ts = gen.nvfp4_quantize(bits)
            qs.append(oracle.Mat(packed=pk, scales=sc, tensor_scale=ts))
            deq = oracle.nvfp4_dequant(pk, sc, ts)
            # tensor scale is not a power of two, so the dequantised value need
            # not be a bf16 number: compare against numpy on the doubles instead
            bs.append(deq)
    r = oracle.moe_forward(x, Wr, None, q_gu, q_d, None)
    xf = gen.bf16_bits_to_f32(x).astype(np.float64)
    y = np.zeros((T, H))
    for t in range(T):
        for j in range(6):
            e = r["idx"][t, j]
            h = b_gu[e] @ xf[t]
            a = h[:I] * scipy.special.expit(h[:I]) * h[I:]
            y[t] += r["w"][t, j] * (b_d[e] @ a)
    assert np.allclose(r["y"], y, rtol=1e-12, atol=1e-15)


# ---------------------------------------------------------------------------
# the layer sizes against the pages' totals
# ---------------------------------------------------------------------------

def test_assumed_sizes_reproduce_published_parameter_totals():
    facts = json.load(open(os.path.join(GOLDEN, "flint_model_facts.json")))
    E = facts["routed_experts"]["value"]
    L = facts["moe_layers"]["value"]
    k = facts["top_k"]["value"]
    n_shared = facts["shared_experts"]["value"]
    per_expert = 3 * gen.H * gen.I
    moe_total = L * ((E + n_shared) * per_expert + E * gen.H)
    total = facts["total_params_billion"]["value"] * 1e9
    # the MoE stack is most of the model; attention (GQA 32/4, head 128) over
    # 49 layers and the 2 dense layers + embeddings take the rest
    attn = facts["layers"]["value"] * gen.H * (32 * 128 * 2 + 4 * 128 * 2)
    assert 0.90 * total < moe_total < total
    assert moe_total + attn < total * 1.01
    active_moe = L * (k + n_shared) * per_expert
    assert active_moe + attn < facts["active_params_billion"]["value"] * 1e9 * 1.1
    # bf16 bytes of the whole model within 1% of the checkpoint size
    assert abs(total * 2 / 1e9 - facts["bf16_checkpoint_gb"]["value"]) / 79.6 < 0.01
    # NVFP4 bytes of the expert stack (4.5 bits/weight) stay under the 4-bit build's size
    nvfp4_stack = L * (E + n_shared) * (per_expert // 2 + per_expert // 16)
    assert nvfp4_stack / 1e9 < facts["four_bit_checkpoint_gb"]["range"][1]
