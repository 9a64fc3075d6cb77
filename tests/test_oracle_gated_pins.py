"""Pins of the oracle's gated attention variant: the decode-path review "Two
more decode-path suggestions" (item 1) on the segment-KI pull request runs
q/k RMSNorm(1+w), partial NeoX RoPE and an output gate (* sigmoid(gate))
before o_proj.  Each pin ties a part to a closed form, to an already pinned
primitive it must reduce to, or to an invariant it must have.
"""
import dataclasses
import math

import numpy as np

import oracle
import synth


def bits(a):
    f = np.asarray(a, dtype=np.float32)
    u = f.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "value not exactly representable in bf16"
    return (u >> 16).astype(np.uint16)


def tiny(seed=0, S_max=40, p=20, eps=None):
    m = synth.workload("tiny").model
    if eps is not None:
        m = dataclasses.replace(m, rms_eps=eps)
    lay = synth.make_layer(seed, m, 0)
    K = np.zeros((m.n_kv_heads, S_max, m.head_dim), dtype=np.uint16)
    V = np.zeros_like(K)
    synth.make_kv_prefix(seed, m, 0, 0, p, "k", K)
    synth.make_kv_prefix(seed, m, 0, 0, p, "v", V)
    r0 = synth.make_residual(seed + 3, 1, m.hidden)[0].astype(np.float64)
    return m, lay, K, V, r0


# ----------------------------------------------------------------------------- partial RoPE

def test_partial_rope_hand_example():
    # r = 4 of D = 8 at p = 3, theta = 1e4: pair (0, 2) turns by 3 rad, pair (1, 3)
    # by 3 * 1e4^(-1/2) = 0.03 rad, dims 4..7 stay
    v = np.arange(8.0)
    got = oracle.rope_partial(v, 4, 3, 1e4)
    c3, s3, c, s = math.cos(3), math.sin(3), math.cos(0.03), math.sin(0.03)
    want = [0 * c3 - 2 * s3, 1 * c - 3 * s, 2 * c3 + 0 * s3, 3 * c + 1 * s, 4, 5, 6, 7]
    np.testing.assert_allclose(got, want, rtol=1e-15, atol=1e-15)


def test_partial_rope_leaves_the_tail_and_reduces_to_the_full_rope():
    rng = np.random.default_rng(1)
    v = rng.standard_normal((3, 64))
    for r in (2, 16, 32):
        got = oracle.rope_partial(v, r, 77, 1e6)
        np.testing.assert_array_equal(got[:, r:], v[:, r:])
        # the rotated part is the full RoPE of an r-wide head
        np.testing.assert_array_equal(got[:, :r], oracle.rope(v[:, :r], 77, 1e6))
    np.testing.assert_array_equal(oracle.rope_partial(v, 64, 77, 1e6), oracle.rope(v, 77, 1e6))


def test_partial_rope_scores_depend_on_relative_position_only():
    rng = np.random.default_rng(2)
    q, k = rng.standard_normal(32), rng.standard_normal(32)
    s = [oracle.rope_partial(q, 16, p + 9, 1e4) @ oracle.rope_partial(k, 16, p, 1e4) for p in (0, 5, 300)]
    assert abs(s[0] - s[1]) < 1e-12 and abs(s[0] - s[2]) < 1e-12


# ----------------------------------------------------------------------------- per-head norm, gate

def test_head_rmsnorm_closed_form_and_independent_heads():
    g = bits([1.0, 2.0, 0.5, 1.0])
    v = np.array([[3.0, 3.0, 3.0, 3.0], [-2.0, -2.0, -2.0, -2.0]])
    got = oracle.head_rmsnorm(v, g, 0.0)
    np.testing.assert_allclose(got, [[1, 2, 0.5, 1], [-1, -2, -0.5, -1]], rtol=1e-15)
    # eps enters once per head: c / sqrt(c^2 + eps)
    got = oracle.head_rmsnorm(np.full((1, 4), 0.5), bits([1, 1, 1, 1]), 0.25)
    np.testing.assert_allclose(got, np.full((1, 4), 0.5 / math.sqrt(0.5)), rtol=1e-15)
    # changing one head leaves the other as it was
    rng = np.random.default_rng(3)
    a = rng.standard_normal((2, 4))
    b = a.copy()
    b[1] *= 7.0
    np.testing.assert_array_equal(oracle.head_rmsnorm(a, g, 1e-6)[0], oracle.head_rmsnorm(b, g, 1e-6)[0])


def test_sigmoid_closed_forms_and_silu_identity():
    assert oracle.sigmoid(0.0) == 0.5
    for z in (0.3, 2.0, 11.0):
        assert abs(oracle.sigmoid(-z) - (1.0 - oracle.sigmoid(z))) < 1e-15
        # the pinned SiLU is z * sigmoid(z)
        assert abs(oracle.silu(z) - z * oracle.sigmoid(z)) < 1e-15 * max(1.0, z)
    assert oracle.sigmoid(800.0) == 1.0 and oracle.sigmoid(-800.0) == 0.0


# ----------------------------------------------------------------------------- the gated layer

def test_zero_gate_weights_halve_the_attention_output():
    # sigmoid(0) = 1/2 on every element: the plain layer with Wo / 2 (exact in bf16)
    m, lay, K, V, r0 = tiny()
    var = {"rot_dim": m.head_dim, "wgate": np.zeros((m.n_heads * m.head_dim, m.hidden), np.uint16)}
    K1, V1 = K.copy(), V.copy()
    r1, _ = oracle.layer(m, lay, K1, V1, 20, r0, variant=var)
    half = dict(lay)
    half["wo"] = bits(synth.bf16_to_f32(lay["wo"]) * np.float32(0.5))
    K2, V2 = K.copy(), V.copy()
    r2, _ = oracle.layer(m, half, K2, V2, 20, r0)
    np.testing.assert_array_equal(r1, r2)
    np.testing.assert_array_equal(K1, K2)


def test_gate_closes_one_head_and_opens_the_others():
    # gate rows +-64 y (y the layer's normed input) give gates of about +-16,000:
    # sigmoid is then exactly 1 or exactly 0; closing head 0 equals zeroing
    # head 0's columns of Wo
    m, lay, K, V, r0 = tiny()
    Hq, D = m.n_heads, m.head_dim
    _, t = oracle.layer(m, lay, K.copy(), V.copy(), 20, r0, taps=True)
    row = oracle.round_bf16(64.0 * t["y_attn"])
    wgate = np.tile(row, (Hq * D, 1))
    neg = oracle.round_bf16(-64.0 * t["y_attn"])
    wgate[:D] = neg
    r1, t1 = oracle.layer(m, lay, K.copy(), V.copy(), 20, r0, taps=True, variant={"wgate": wgate})
    closed = dict(lay)
    wo = lay["wo"].copy()
    wo[:, :D] = 0
    closed["wo"] = wo
    r2, t2 = oracle.layer(m, closed, K.copy(), V.copy(), 20, r0, taps=True)
    np.testing.assert_array_equal(r1, r2)
    assert np.all(t1["o"][:D] == 0) and np.array_equal(t1["o"][D:], t2["o"][D:])


def test_qk_norm_makes_the_layer_blind_to_the_scale_of_wq_and_wk():
    # with eps = 0, doubling Wq or Wk (exact in bf16) changes nothing once q and
    # k are normalised per head; without the norm it changes the scores
    m, lay, K, V, r0 = tiny(eps=0.0)
    gq = synth.normal_bf16(5, "qn", (m.head_dim,), 1.0, 0.1)
    gk = synth.normal_bf16(5, "kn", (m.head_dim,), 1.0, 0.1)
    var = {"q_norm": gq, "k_norm": gk}
    base, _ = oracle.layer(m, lay, K.copy(), V.copy(), 20, r0, variant=var)
    for name in ("wq", "wk"):
        doubled = dict(lay)
        doubled[name] = bits(synth.bf16_to_f32(lay[name]) * np.float32(2.0))
        got, _ = oracle.layer(m, doubled, K.copy(), V.copy(), 20, r0, variant=var)
        np.testing.assert_array_equal(got, base)
        plain_a, _ = oracle.layer(m, lay, K.copy(), V.copy(), 20, r0)
        plain_b, _ = oracle.layer(m, doubled, K.copy(), V.copy(), 20, r0)
        assert not np.array_equal(plain_a, plain_b)


def test_partial_rotary_leaves_the_key_tail_independent_of_position():
    m, lay, K, V, r0 = tiny()
    var = {"rot_dim": 16, "k_norm": synth.normal_bf16(6, "kn", (m.head_dim,), 1.0, 0.1)}
    _, ta = oracle.layer(m, lay, K.copy(), V.copy(), 0, r0, taps=True, variant=var)
    _, tb = oracle.layer(m, lay, K.copy(), V.copy(), 25, r0, taps=True, variant=var)
    ka = ta["k"].reshape(m.n_kv_heads, m.head_dim)
    kb = tb["k"].reshape(m.n_kv_heads, m.head_dim)
    np.testing.assert_array_equal(ka[:, 16:], kb[:, 16:])
    assert not np.allclose(ka[:, :16], kb[:, :16])
    # at p = 0 the rotation is the identity: the tap is the per-head-normed key
    y = ta["y_attn"]
    k0 = oracle.head_rmsnorm(oracle.linear(lay["wk"], y).reshape(m.n_kv_heads, m.head_dim), var["k_norm"],
                             m.rms_eps)
    np.testing.assert_allclose(ka, k0, rtol=1e-14, atol=1e-14)


def test_gated_layer_equals_composition_of_pinned_primitives():
    m, lay, K, V, r0 = tiny()
    H, Hq, Hkv, D, p = m.hidden, m.n_heads, m.n_kv_heads, m.head_dim, 20
    var = {"rot_dim": 16, "q_norm": synth.normal_bf16(7, "qn", (D,), 1.0, 0.1),
           "k_norm": synth.normal_bf16(7, "kn", (D,), 1.0, 0.1),
           "wgate": synth.normal_bf16(7, "gate", (Hq * D, H), 0.0, 0.05)}
    K1, V1 = K.copy(), V.copy()
    r1, taps = oracle.layer(m, lay, K1, V1, p, r0, taps=True, variant=var)

    K2, V2 = K.copy(), V.copy()
    _, y = oracle.rmsnorm(r0, lay["attn_norm"], m.rms_eps)
    q = oracle.head_rmsnorm(oracle.linear(lay["wq"], y).reshape(Hq, D), var["q_norm"], m.rms_eps)
    k = oracle.head_rmsnorm(oracle.linear(lay["wk"], y).reshape(Hkv, D), var["k_norm"], m.rms_eps)
    q = oracle.rope_partial(q, 16, p, m.rope_theta)
    k = oracle.rope_partial(k, 16, p, m.rope_theta)
    v = oracle.linear(lay["wv"], y).reshape(Hkv, D)
    K2[:, p] = oracle.round_bf16(k)
    V2[:, p] = oracle.round_bf16(v)
    o = oracle.attention(q, K2, V2, p + 1).reshape(-1)
    gate = oracle.linear(var["wgate"], y)
    o = o * np.array([oracle.sigmoid(g) for g in gate])
    r = r0 + oracle.linear(lay["wo"], o)
    _, y2 = oracle.rmsnorm(r, lay["mlp_norm"], m.rms_eps)
    r = r + oracle.linear(lay["wd"], oracle.glu(lay["wg"], lay["wu"], y2))

    np.testing.assert_array_equal(K1, K2)
    np.testing.assert_array_equal(V1, V2)
    np.testing.assert_allclose(taps["o"], o, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(r1, r, rtol=1e-14, atol=1e-14)


def test_gated_step_equals_its_layers_then_the_head():
    m = synth.workload("tiny").model
    m = dataclasses.replace(m, n_layers=2)
    S_max, p = 24, 9
    lays = [synth.make_layer(0, m, l) for l in range(2)]
    vars_ = [synth.make_gated_attention(0, m, l, 16) for l in range(2)]
    E = synth.make_embedding(0, m)
    fn = synth.make_final_norm(0, m)
    Ks = [np.zeros((1, m.n_kv_heads, S_max, m.head_dim), np.uint16) for _ in range(2)]
    Vs = [np.zeros_like(k) for k in Ks]
    for l in range(2):
        synth.make_kv_prefix(0, m, l, 0, p, "k", Ks[l][0])
        synth.make_kv_prefix(0, m, l, 0, p, "v", Vs[l][0])
    Ka, Va = [k.copy() for k in Ks], [v.copy() for v in Vs]
    model = oracle.Model(m, lays, E, fn, E, Ka, Va, variants=vars_)
    tok, logits, r_out = model.step(0, p, token=123)

    r = synth.bf16_to_f64(E[123])
    Kb, Vb = [k[0].copy() for k in Ks], [v[0].copy() for v in Vs]
    for l in range(2):
        r, _ = oracle.layer(m, lays[l], Kb[l], Vb[l], p, r, variant=vars_[l])
    t2, logits2 = oracle.head(r, fn, E, m.rms_eps)
    np.testing.assert_array_equal(r_out, r)
    np.testing.assert_array_equal(logits, logits2)
    assert tok == t2
    for l in range(2):
        np.testing.assert_array_equal(Ka[l][0], Kb[l])
    # without variants the model is the plain dense step
    plain = oracle.Model(m, lays, E, fn, E, [k.copy() for k in Ks], [v.copy() for v in Vs])
    _, _, r_plain = plain.step(0, p, token=123)
    r = synth.bf16_to_f64(E[123])
    Kc, Vc = [k[0].copy() for k in Ks], [v[0].copy() for v in Vs]
    for l in range(2):
        r, _ = oracle.layer(m, lays[l], Kc[l], Vc[l], p, r)
    np.testing.assert_array_equal(r_plain, r)
    assert not np.array_equal(r_plain, r_out)
