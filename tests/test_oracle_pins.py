"""Pins of the fp64 oracle against facts that do not come from the oracle itself:
closed forms, hand-worked examples, exact integer arithmetic, invariants of
the mathematics, and the GQA partition worked example printed on the Ulysses
KV-head-count pull request (DeepSpeed #8316, "The change").

Each pin is chosen so that a plausible slip (a dropped term, a wrong sign, a
swapped index or a transposed operand) breaks at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
import synth

HERE = os.path.dirname(os.path.abspath(__file__))


def bits(a):
    """Exact bf16 bit patterns of values that bf16 represents exactly (asserted)."""
    f = np.asarray(a, dtype=np.float32)
    u = f.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "value not exactly representable in bf16"
    return (u >> 16).astype(np.uint16)


# ----------------------------------------------------------------------------- bf16

def test_bf16_widening_is_exact():
    assert oracle.bf16_to_f64(0x3F80) == 1.0
    assert oracle.bf16_to_f64(0xC000) == -2.0
    assert oracle.bf16_to_f64(0x3F81) == 1.0 + 2.0 ** -7
    assert oracle.bf16_to_f64(0x0001) == 2.0 ** -133
    assert oracle.bf16_to_f64(0x7F7F) == (2 - 2.0 ** -7) * 2.0 ** 127


@pytest.mark.parametrize("x,expect", [
    (1.0, 0x3F80),
    (1.0 + 2.0 ** -8, 0x3F80),            # halfway, even neighbour below
    (1.0 + 3 * 2.0 ** -8, 0x3F82),        # halfway, even neighbour above
    (1.0 + 2.0 ** -8 + 2.0 ** -40, 0x3F81),  # just above halfway
    (-1.0 - 2.0 ** -8 - 2.0 ** -40, 0xBF81),
    (0.0, 0x0000),
    (-0.0, 0x8000),
    (2.0 ** -133, 0x0001),                # smallest subnormal
    (1.5 * 2.0 ** -133, 0x0002),          # subnormal tie to even
    (3.5e38, 0x7F80),                     # overflow to +inf
])
def test_bf16_rounding_cases(x, expect):
    assert oracle.f64_to_bf16(x) == expect


def test_bf16_rounding_matches_float32_bit_trick():
    # For doubles that are exact float32 values, one-step rounding equals the
    # classic float32 round-to-nearest-even bit trick (an independent method).
    rng = np.random.default_rng(1)
    f = (rng.standard_normal(4000) * np.exp(rng.uniform(-20, 20, 4000))).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    ref = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    got = oracle.round_bf16(f.astype(np.float64))
    np.testing.assert_array_equal(got, ref)


# ----------------------------------------------------------------------------- RMSNorm

def test_rmsnorm_constant_vector_closed_form():
    H, c, eps = 16, 0.75, 1e-6
    gamma = synth.normal_bf16(3, "g", (H,), 1.0, 0.1)
    _, y = oracle.rmsnorm(np.full(H, c), gamma, eps)
    g = synth.bf16_to_f64(gamma)
    np.testing.assert_allclose(y, g * c / math.sqrt(c * c + eps), rtol=1e-15)


def test_rmsnorm_hand_example():
    # r = (3, 4): mean of squares 12.5; gains (1, 2); eps = 0
    _, y = oracle.rmsnorm(np.array([3.0, 4.0]), bits([1.0, 2.0]), 0.0)
    s = math.sqrt(12.5)
    np.testing.assert_allclose(y, [3 / s, 8 / s], rtol=1e-15)


def test_rmsnorm_scale_invariance_without_eps():
    r = np.random.default_rng(2).standard_normal(64)
    gamma = synth.normal_bf16(4, "g", (64,), 1.0, 0.1)
    _, y1 = oracle.rmsnorm(r, gamma, 0.0)
    _, y2 = oracle.rmsnorm(37.5 * r, gamma, 0.0)
    np.testing.assert_allclose(y1, y2, rtol=1e-13)


def test_add_rmsnorm_updates_residual_then_normalises():
    r = np.array([1.0, -2.0, 0.5, 4.0])
    x = np.array([0.5, 2.0, -0.5, -1.0])
    r2, y = oracle.rmsnorm(r, bits([1, 1, 1, 1]), 0.0, x=x)
    np.testing.assert_array_equal(r2, r + x)
    s = math.sqrt(np.mean((r + x) ** 2))
    np.testing.assert_allclose(y, (r + x) / s, rtol=1e-15)


# ----------------------------------------------------------------------------- GEMV

def test_linear_integer_exact_nonsquare():
    rng = np.random.default_rng(5)
    W = rng.integers(-8, 9, size=(7, 9))
    x = rng.integers(-5, 6, size=9)
    y = oracle.linear(bits(W), x)
    np.testing.assert_array_equal(y, (W @ x).astype(np.float64))
    y2 = oracle.linear(bits(W.T.copy()), rng.integers(-5, 6, size=7))
    assert y2.shape == (9,)


def test_linear_permutation_matrix():
    perm = np.array([3, 0, 4, 1, 2])
    W = np.eye(5)[perm]
    x = np.array([1.5, -2.0, 3.25, 7.0, -0.125])
    np.testing.assert_array_equal(oracle.linear(bits(W), x), x[perm])


# ----------------------------------------------------------------------------- RoPE

def test_rope_two_dims_closed_form():
    # one pair, frequency theta^0 = 1: a counter-clockwise turn by p radians
    np.testing.assert_allclose(oracle.rope([1.0, 0.0], 1, 1e4), [math.cos(1), math.sin(1)], rtol=1e-15)
    np.testing.assert_allclose(oracle.rope([0.0, 1.0], 1, 1e4), [-math.sin(1), math.cos(1)], rtol=1e-15)


def test_rope_pairs_i_with_i_plus_half_and_frequency():
    # D = 8: element 1 pairs with element 5 and turns at theta^(-2/8)
    v = np.zeros(8)
    v[1] = 1.0
    out = oracle.rope(v, 7, 1e4)
    ang = 7 * 1e4 ** (-2 / 8)
    expect = np.zeros(8)
    expect[1], expect[5] = math.cos(ang), math.sin(ang)
    np.testing.assert_allclose(out, expect, atol=1e-15)


def test_rope_position_zero_is_identity_and_norm_preserving():
    v = np.random.default_rng(6).standard_normal((3, 64))
    np.testing.assert_array_equal(oracle.rope(v, 0, 1e6), v)
    out = oracle.rope(v, 12345, 1e6)
    h = 32
    np.testing.assert_allclose(out[:, :h] ** 2 + out[:, h:] ** 2, v[:, :h] ** 2 + v[:, h:] ** 2, rtol=1e-12)


def test_rope_relative_position_and_composition():
    rng = np.random.default_rng(7)
    q, k = rng.standard_normal(128), rng.standard_normal(128)
    d1 = oracle.rope(q, 100, 1e6) @ oracle.rope(k, 40, 1e6)
    d2 = oracle.rope(q, 1060, 1e6) @ oracle.rope(k, 1000, 1e6)
    assert abs(d1 - d2) < 1e-10
    np.testing.assert_allclose(oracle.rope(oracle.rope(q, 300, 1e6), 77, 1e6), oracle.rope(q, 377, 1e6),
                               atol=1e-12)


# ----------------------------------------------------------------------------- attention

def _cache(rows_k, rows_v, Hkv=1, S_max=None):
    rows_k = np.asarray(rows_k, dtype=np.float64)
    S, D = rows_k.shape
    S_max = S_max or S
    K = np.zeros((Hkv, S_max, D), dtype=np.uint16)
    V = np.zeros((Hkv, S_max, D), dtype=np.uint16)
    K[:, :S] = bits(rows_k)
    V[:, :S] = bits(rows_v)
    return K, V


def test_attention_hand_example():
    # scores (0, ln 3) -> weights (1/4, 3/4); values (4,0), (0,8) -> (1, 6)
    K, V = _cache([[0, 0], [1, 0]], [[4, 0], [0, 8]])
    q = np.array([[math.log(3) * math.sqrt(2), 0.0]])
    np.testing.assert_allclose(oracle.attention(q, K, V, 2), [[1.0, 6.0]], rtol=1e-14)


def test_attention_single_key_returns_value_and_ignores_later_slots():
    K, V = _cache([[1, 2, 3, 4]], [[0.5, -1, 2, 8]], S_max=3)
    V[0, 1:] = bits(np.full((2, 4), 100.0))  # beyond S: must not be read
    q = np.random.default_rng(8).standard_normal((1, 4))
    np.testing.assert_array_equal(oracle.attention(q, K, V, 1), [[0.5, -1, 2, 8]])


def test_attention_identical_keys_average_values():
    rng = np.random.default_rng(9)
    Vrows = rng.integers(-4, 5, size=(5, 8)).astype(float)
    K, V = _cache(np.tile([1.0, -2.0, 0.5, 0, 0, 0, 0, 3], (5, 1)), Vrows)
    q = rng.standard_normal((1, 8))
    np.testing.assert_allclose(oracle.attention(q, K, V, 5), Vrows.mean(0, keepdims=True), atol=1e-14)


def test_attention_dominant_key_selects_its_value():
    K, V = _cache([[0, 0], [64, 0], [0, 0]], [[1, 1], [5, -3], [2, 2]])
    q = np.array([[4.0, 0.0]])  # score 256/sqrt(2) vs 0: weight of the rest ~ e^-181
    np.testing.assert_allclose(oracle.attention(q, K, V, 3), [[5.0, -3.0]], atol=1e-12)


@pytest.mark.parametrize("S", [1, 2, 7, 33])
def test_online_splitk_equals_two_pass_for_every_split_count(S):
    rng = np.random.default_rng(10 + S)
    Hq, Hkv, D = 4, 2, 16
    K = synth.normal_bf16(S, "k", (Hkv, S + 3, D))
    V = synth.normal_bf16(S, "v", (Hkv, S + 3, D))
    q = 3 * rng.standard_normal((Hq, D))
    ref = oracle.attention(q, K, V, S)
    for n in range(1, S + 1):
        np.testing.assert_allclose(oracle.attention(q, K, V, S, n_splits=n), ref, rtol=1e-12, atol=1e-13)


# ----------------------------------------------------------------------------- GQA mapping

def test_gqa_mapping_distinct_constant_values():
    Hq, Hkv, D, S = 6, 3, 8, 5
    K = synth.normal_bf16(11, "k", (Hkv, S, D))
    V = np.zeros((Hkv, S, D), dtype=np.uint16)
    for g in range(Hkv):
        V[g] = bits(np.full((S, D), float(g + 1)))
    q = np.random.default_rng(12).standard_normal((Hq, D))
    o = oracle.attention(q, K, V, S)
    groups = [int(round(o[h, 0])) - 1 for h in range(Hq)]
    np.testing.assert_allclose(o, np.repeat(np.array(groups, float)[:, None] + 1, D, 1), atol=1e-14)
    assert groups == [0, 0, 1, 1, 2, 2]
    assert groups != [h % Hkv for h in range(Hq)]  # the interleaved reading is wrong


def test_gqa_partition_worked_example_from_ulysses_pr():
    with open(os.path.join(HERE, "golden", "gqa_partition.json")) as f:
        fx = json.load(f)
    for case in fx["cases"]:
        Hq, Hkv = case["n_q_heads"], case["n_kv_heads"]
        bounds = np.cumsum([0] + case["kv_split"])
        q_split = []
        for r in range(len(case["kv_split"])):
            q_split.append(sum(1 for h in range(Hq) if bounds[r] <= oracle.kv_head(h, Hq, Hkv) < bounds[r + 1]))
        assert q_split == case["q_split"], case["note"]


# ----------------------------------------------------------------------------- SiLU, GLU, argmax

def test_silu_closed_forms_and_identity():
    assert oracle.silu(0.0) == 0.0
    assert oracle.silu(1.0) == pytest.approx(1 / (1 + math.exp(-1)), rel=1e-15)
    assert oracle.silu(40.0) == pytest.approx(40.0, rel=1e-15)
    for z in (0.3, 1.7, 5.0, 11.0):
        assert oracle.silu(-z) == pytest.approx(oracle.silu(z) - z, abs=1e-14)


def test_glu_integer_inputs():
    rng = np.random.default_rng(13)
    Wg = rng.integers(-3, 4, size=(6, 5))
    Wu = rng.integers(-3, 4, size=(6, 5))
    y = rng.integers(-2, 3, size=5).astype(float)
    g, u = Wg @ y, Wu @ y
    expect = [gi / (1 + math.exp(-gi)) * ui for gi, ui in zip(g, u)]
    np.testing.assert_allclose(oracle.glu(bits(Wg), bits(Wu), y), expect, rtol=1e-15, atol=1e-300)


def test_argmax_ties_pick_lowest_index():
    assert oracle.argmax([1.0, 3.0, 3.0, 2.0]) == 1
    assert oracle.argmax([5.0, 5.0, 5.0]) == 0
    assert oracle.argmax([-np.inf, -1.0, -1.0]) == 1
    assert oracle.argmax([0.0, -0.0, 0.0]) == 0


# ----------------------------------------------------------------------------- layer and step

def _tiny_model(seed=0, S_max=40, p=20, B=1):
    w = synth.workload("tiny")
    m = w.model
    lay = synth.make_layer(seed, m, 0)
    K = np.zeros((B, m.n_kv_heads, S_max, m.head_dim), dtype=np.uint16)
    V = np.zeros_like(K)
    for b in range(B):
        synth.make_kv_prefix(seed, m, 0, b, p, "k", K[b])
        synth.make_kv_prefix(seed, m, 0, b, p, "v", V[b])
    return m, lay, K, V


def test_layer_equals_composition_of_pinned_primitives():
    m, lay, K, V = _tiny_model()
    p = 20
    r0 = synth.make_residual(0, 1, m.hidden)[0].astype(np.float64)
    K1, V1 = K[0].copy(), V[0].copy()
    r1, taps = oracle.layer(m, lay, K1, V1, p, r0, taps=True)

    # the same layer written out from the primitives
    H, Hq, Hkv, D = m.hidden, m.n_heads, m.n_kv_heads, m.head_dim
    K2, V2 = K[0].copy(), V[0].copy()
    _, y = oracle.rmsnorm(r0, lay["attn_norm"], m.rms_eps)
    q = oracle.rope(oracle.linear(lay["wq"], y).reshape(Hq, D), p, m.rope_theta)
    k = oracle.rope(oracle.linear(lay["wk"], y).reshape(Hkv, D), p, m.rope_theta)
    v = oracle.linear(lay["wv"], y).reshape(Hkv, D)
    K2[:, p] = oracle.round_bf16(k)
    V2[:, p] = oracle.round_bf16(v)
    o = oracle.attention(q, K2, V2, p + 1)
    r = r0 + oracle.linear(lay["wo"], o.reshape(-1))
    _, y2 = oracle.rmsnorm(r, lay["mlp_norm"], m.rms_eps)
    r = r + oracle.linear(lay["wd"], oracle.glu(lay["wg"], lay["wu"], y2))

    np.testing.assert_array_equal(K1, K2)
    np.testing.assert_array_equal(V1, V2)
    np.testing.assert_allclose(taps["q"], q.reshape(-1), rtol=1e-15, atol=1e-15)
    np.testing.assert_allclose(taps["o"], o.reshape(-1), rtol=1e-15, atol=1e-15)
    np.testing.assert_allclose(r1, r, rtol=1e-14, atol=1e-14)


def test_layer_with_zero_output_projections_keeps_residual():
    m, lay, K, V = _tiny_model()
    lay = dict(lay)
    lay["wo"] = np.zeros_like(lay["wo"])
    lay["wd"] = np.zeros_like(lay["wd"])
    r0 = synth.make_residual(1, 1, m.hidden)[0].astype(np.float64)
    K1, V1 = K[0].copy(), V[0].copy()
    r1, taps = oracle.layer(m, lay, K1, V1, 20, r0, taps=True)
    np.testing.assert_array_equal(r1, r0)
    np.testing.assert_array_equal(K1[:, 20], oracle.round_bf16(taps["k"].reshape(m.n_kv_heads, -1)))
    np.testing.assert_array_equal(K1[:, :20], K[0][:, :20])  # older slots untouched


def test_step_one_hot_embedding_repeats_its_input_token():
    # Embedding rows are permuted unit vectors, attention and MLP outputs are
    # zero: the final norm of e_pi(t) is e_pi(t) / sqrt(1/H + eps) and the tied
    # head scores row t highest, so greedy decoding returns the input token.
    m = synth.ModelShape(2, 16, 2, 1, 8, 8, 16, gain_std=0.0)
    perm = np.random.default_rng(14).permutation(16)
    E = bits(np.eye(16)[perm])
    layers = []
    for l in range(m.n_layers):
        lay = synth.make_layer(5, m, l)
        lay["wo"] = np.zeros_like(lay["wo"])
        lay["wd"] = np.zeros_like(lay["wd"])
        layers.append(lay)
    S_max = 4
    Kc = [np.zeros((1, 1, S_max, 8), np.uint16) for _ in range(2)]
    Vc = [np.zeros((1, 1, S_max, 8), np.uint16) for _ in range(2)]
    model = oracle.Model(m, layers, E, bits(np.ones(16)), E, Kc, Vc)
    for t in (0, 5, 11):
        tok, logits, _ = model.step(0, 1, token=t)
        assert tok == t
        assert logits[t] == pytest.approx(1 / math.sqrt(1 / 16 + m.rms_eps), rel=1e-12)


def test_step_equals_layers_then_head():
    m, lay, K, V = _tiny_model()
    E = synth.make_embedding(0, m)
    fn = synth.make_final_norm(0, m)
    model = oracle.Model(m, [lay], E, fn, E, [K.copy()], [V.copy()])
    tok, logits, r_fin = model.step(0, 20, token=77)
    r, _ = oracle.layer(m, lay, K[0].copy(), V[0].copy(), 20, synth.bf16_to_f64(E[77]))
    np.testing.assert_allclose(r_fin, r, rtol=1e-15, atol=1e-15)
    t2, l2 = oracle.head(r, fn, E, m.rms_eps)
    assert t2 == tok
    np.testing.assert_allclose(logits, l2, rtol=1e-15, atol=1e-15)
