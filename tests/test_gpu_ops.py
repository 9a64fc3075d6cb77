"""Parity of each single-op C-ABI call against the fp64 oracle on the same
seeded inputs: the one-layer workload shapes (tiny: H=256, 4/2 heads, D=64;
4B-class: H=2560, 32/8 heads, D=128, I=9728), ragged tails, several batch
sizes and the edge cases of each op."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import (MARGIN, TOL, assert_close, dev_bf16, dev_f32, dev_i32, host_bits, rel_err)

pytestmark = pytest.mark.gpu

gd = pytest.importorskip("greedy_decode_step_gb300")

SHAPES = {
    "tiny": dict(H=256, Hq=4, Hkv=2, D=64, I=704, V=1024),
    "4b": dict(H=2560, Hq=32, Hkv=8, D=128, I=9728, V=151936),
    "gqa12x3": dict(H=1536, Hq=12, Hkv=3, D=128, I=8960, V=151936),
}


def f32_of_bits(bits):
    return synth.bf16_to_f32(bits)


def act(seed, name, shape):
    """fp32 activations holding bf16-representable N(0,1) values."""
    return f32_of_bits(synth.normal_bf16(seed, name, shape))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    gd.lib()
    assert gd.device_error(clear=True) == 0
    yield
    assert gd.device_error(clear=True) == 0


# ----------------------------------------------------------------------------- RMSNorm

@pytest.mark.parametrize("B,H", [(1, 256), (3, 2560), (16, 1536), (1, 8), (2, 9728)])
@pytest.mark.parametrize("with_add", [False, True])
def test_add_rmsnorm(B, H, with_add):
    r0 = act(1, "r", (B, H)) * 3.0
    x = act(2, "x", (B, H)) if with_add else None
    gamma = synth.normal_bf16(3, "g", (H,), 1.0, 0.1)
    r = dev_f32(r0)
    y = torch.empty_like(r)
    gd.dec_add_rmsnorm(dev_f32(x) if x is not None else None, r, dev_bf16(gamma), y, 1e-6)
    r_ref, y_ref = oracle.rmsnorm(r0, gamma, 1e-6, x=x)
    assert_close(r.cpu().numpy(), r_ref, 1e-6, "residual")
    assert_close(y.cpu().numpy(), y_ref, TOL, "y")
    assert rel_err(y.cpu().numpy(), y_ref) < 1e-5


# ----------------------------------------------------------------------------- QKV + RoPE + cache store

@pytest.mark.parametrize("shape", ["tiny", "4b", "gqa12x3"])
@pytest.mark.parametrize("B", [1, 3])
def test_qkv_gemv_rope(shape, B):
    s = SHAPES[shape]
    H, Hq, Hkv, D = s["H"], s["Hq"], s["Hkv"], s["D"]
    S_max = 5000
    Wq = synth.normal_bf16(0, "wq", (Hq * D, H), 0, 0.02)
    Wk = synth.normal_bf16(0, "wk", (Hkv * D, H), 0, 0.02)
    Wv = synth.normal_bf16(0, "wv", (Hkv * D, H), 0, 0.02)
    y = act(5, "y", (B, H))
    pos = np.array([0, 4096, 4999, 17, 1][:B], dtype=np.int32)
    K = torch.zeros((B, Hkv, S_max, D), dtype=torch.bfloat16, device="cuda")
    V = torch.zeros_like(K)
    K[:, :, 10] = 1.5  # a slot nobody writes must keep its contents
    q = torch.empty((B, Hq * D), dtype=torch.float32, device="cuda")
    gd.dec_qkv_gemv_rope(dev_f32(y), dev_bf16(Wq), dev_bf16(Wk), dev_bf16(Wv), dev_i32(pos), 1e6, q, K, V)
    torch.cuda.synchronize()
    Kh, Vh = host_bits(K), host_bits(V)
    for b in range(B):
        qr = oracle.rope(oracle.linear(Wq, y[b]).reshape(Hq, D), int(pos[b]), 1e6)
        kr = oracle.rope(oracle.linear(Wk, y[b]).reshape(Hkv, D), int(pos[b]), 1e6)
        vr = oracle.linear(Wv, y[b]).reshape(Hkv, D)
        assert rel_err(q[b].cpu().numpy(), qr) < 1e-4
        assert_close(f32_of_bits(Kh[b, :, pos[b]]), kr, TOL, "k slot")
        assert_close(f32_of_bits(Vh[b, :, pos[b]]), vr, TOL, "v slot")
        # the bf16 store agrees with the oracle's own rounding except at rounding ties of the fp32 value
        same = np.mean(Kh[b, :, pos[b]] == oracle.round_bf16(kr))
        assert same > 0.99
    # untouched slots
    mask = np.ones((B, S_max), bool)
    mask[np.arange(B), pos] = False
    assert np.all(Kh[:, :, 10][mask[:, 10]] == 0x3FC0)
    written = np.zeros((B, Hkv, S_max), bool)
    written[np.arange(B), :, pos] = True
    written[:, :, 10] = True
    assert np.all(Kh[~written] == 0) and np.all(Vh[~written] == 0)


def test_qkv_position_outside_cache_is_refused_on_device():
    H, Hq, Hkv, D, S_max = 256, 4, 2, 64, 16
    W = [dev_bf16(synth.normal_bf16(0, n, (r * D, H), 0, 0.02)) for n, r in (("q", Hq), ("k", Hkv), ("v", Hkv))]
    K = torch.zeros((1, Hkv, S_max, D), dtype=torch.bfloat16, device="cuda")
    V = torch.zeros_like(K)
    q = torch.empty((1, Hq * D), dtype=torch.float32, device="cuda")
    gd.dec_qkv_gemv_rope(dev_f32(act(1, "y", (1, H))), *W, dev_i32([S_max]), 1e6, q, K, V)
    assert gd.device_error(clear=True) & 4
    assert int((K != 0).sum()) == 0 and int((V != 0).sum()) == 0


# ----------------------------------------------------------------------------- attention

def _attn_case(B, Hq, Hkv, D, S_max, pos, seed=0, scale_q=1.0):
    Kb = synth.normal_bf16(seed, "K", (B, Hkv, S_max, D))
    Vb = synth.normal_bf16(seed, "V", (B, Hkv, S_max, D))
    q = act(seed + 1, "q", (B, Hq, D)) * scale_q
    o = torch.empty((B, Hq, D), dtype=torch.float32, device="cuda")
    return Kb, Vb, q, o


@pytest.mark.parametrize("D,Hq,Hkv", [(64, 4, 2), (128, 32, 8), (128, 12, 3), (128, 16, 1), (64, 8, 8)])
@pytest.mark.parametrize("S", [1, 2, 31, 32, 33, 64, 65, 129, 700, 4097])
def test_attention_lengths(D, Hq, Hkv, S):
    B, S_max = 1, 4200
    Kb, Vb, q, o = _attn_case(B, Hq, Hkv, D, S_max, S - 1)
    gd.dec_gqa_decode_attn(dev_f32(q), dev_bf16(Kb), dev_bf16(Vb), dev_i32([S - 1]), o)
    ref = oracle.attention(q[0], Kb[0], Vb[0], S)
    e = assert_close(o[0].cpu().numpy(), ref, TOL, f"S={S}")
    assert e < 1e-4


@pytest.mark.parametrize("splits", [1, 2, 3, 7, 64])
def test_attention_split_count_invariance(splits):
    B, Hq, Hkv, D, S_max = 3, 32, 8, 128, 3000
    pos = [2999, 0, 1500]
    Kb, Vb, q, o = _attn_case(B, Hq, Hkv, D, S_max, pos, seed=4, scale_q=2.0)
    gd.dec_gqa_decode_attn(dev_f32(q), dev_bf16(Kb), dev_bf16(Vb), dev_i32(pos), o, num_splits=splits)
    for b in range(B):
        ref = oracle.attention(q[b], Kb[b], Vb[b], pos[b] + 1)
        assert rel_err(o[b].cpu().numpy(), ref) < 1e-4


def test_attention_ragged_batch_and_reuse_of_workspace():
    B, Hq, Hkv, D, S_max = 8, 32, 8, 128, 9000
    pos = synth.uniform_int(7, "pos", (B,), 0, S_max - 1)
    Kb, Vb, q, o = _attn_case(B, Hq, Hkv, D, S_max, pos, seed=7)
    Kd, Vd, qd, pd = dev_bf16(Kb), dev_bf16(Vb), dev_f32(q), dev_i32(pos)
    ws = gd.dec_gqa_decode_attn(qd, Kd, Vd, pd, o)
    o2 = torch.empty_like(o)
    gd.dec_gqa_decode_attn(qd, Kd, Vd, pd, o2, ws=ws)
    assert torch.equal(o, o2)  # deterministic, and the counters were left at zero
    for b in range(B):
        assert rel_err(o[b].cpu().numpy(), oracle.attention(q[b], Kb[b], Vb[b], int(pos[b]) + 1)) < 1e-4


def test_attention_gqa_mapping_6q_3kv():
    # KV head g holds the constant value g+1 in V: o_h names the group of head h
    B, Hq, Hkv, D, S_max, S = 1, 6, 3, 128, 64, 40
    Kb = synth.normal_bf16(9, "K", (B, Hkv, S_max, D))
    Vf = np.zeros((B, Hkv, S_max, D), np.float32)
    for g in range(Hkv):
        Vf[:, g] = g + 1
    Vb = (Vf.view(np.uint32) >> 16).astype(np.uint16)
    q = act(10, "q", (B, Hq, D))
    o = torch.empty((B, Hq, D), dtype=torch.float32, device="cuda")
    gd.dec_gqa_decode_attn(dev_f32(q), dev_bf16(Kb), dev_bf16(Vb), dev_i32([S - 1]), o)
    groups = [int(round(float(o[0, h, 0]))) - 1 for h in range(Hq)]
    assert groups == [0, 0, 1, 1, 2, 2]
    np.testing.assert_allclose(o[0].cpu().numpy(), oracle.attention(q[0], Kb[0], Vb[0], S), rtol=1e-6)


def test_attention_position_outside_cache_sets_error():
    B, Hq, Hkv, D, S_max = 1, 4, 2, 64, 8
    Kb, Vb, q, o = _attn_case(B, Hq, Hkv, D, S_max, 0)
    gd.dec_gqa_decode_attn(dev_f32(q), dev_bf16(Kb), dev_bf16(Vb), dev_i32([S_max]), o)
    assert gd.device_error(clear=True) & 4


# ----------------------------------------------------------------------------- GLU and down

@pytest.mark.parametrize("shape", ["tiny", "4b", "gqa12x3"])
@pytest.mark.parametrize("B", [1, 2, 5, 8, 16])
def test_glu_gemv(shape, B):
    s = SHAPES[shape]
    H, I = s["H"], s["I"]
    Wg = synth.normal_bf16(1, "wg", (I, H), 0, 0.02)
    Wu = synth.normal_bf16(1, "wu", (I, H), 0, 0.02)
    y = act(2, "y", (B, H))
    h = torch.empty((B, I), dtype=torch.float32, device="cuda")
    gd.dec_glu_gemv(dev_f32(y), dev_bf16(Wg), dev_bf16(Wu), h)
    ref = oracle.glu(Wg, Wu, y)
    assert rel_err(h.cpu().numpy(), ref) < 1e-4


@pytest.mark.parametrize("N_in,N_out", [(704, 256), (256, 256), (4096, 2560), (9728, 2560), (8960, 1536), (1536, 1536),
                                        (8, 3), (1032, 77)])
@pytest.mark.parametrize("B", [1, 3, 8, 16])
def test_down_gemv_residual(N_in, N_out, B):
    W = synth.normal_bf16(3, "w", (N_out, N_in), 0, 0.02)
    x = act(4, "x", (B, N_in))
    r0 = act(5, "r", (B, N_out))
    r = dev_f32(r0)
    gd.dec_down_gemv(dev_f32(x), dev_bf16(W), r)
    ref = r0 + oracle.linear(W, x)
    assert rel_err(r.cpu().numpy(), ref) < 1e-4


# ----------------------------------------------------------------------------- LM head + argmax

@pytest.mark.parametrize("shape", ["tiny", "4b"])
@pytest.mark.parametrize("B", [1, 4])
def test_lmhead_argmax(shape, B):
    s = SHAPES[shape]
    H, V = s["H"], s["V"]
    W = synth.normal_bf16(6, "lm", (V, H), 0, 0.02)
    g = synth.normal_bf16(6, "gf", (H,), 1.0, 0.02)
    r = act(7, "r", (B, H)) * 2.0
    tok = torch.empty(B, dtype=torch.int32, device="cuda")
    logits = torch.empty((B, V), dtype=torch.float32, device="cuda")
    gd.dec_lmhead_argmax(dev_f32(r), dev_bf16(g), 1e-6, dev_bf16(W), tok, logits)
    tk = tok.cpu().numpy()
    lg = logits.cpu().numpy()
    for b in range(B):
        t_ref, l_ref = oracle.head(r[b], g, W, 1e-6)
        assert rel_err(lg[b], l_ref) < 1e-4
        assert tk[b] == int(np.argmax(lg[b]))  # its own logits, first maximum
        if oracle.top2_margin(l_ref) > MARGIN:
            assert tk[b] == t_ref


def test_lmhead_ties_pick_lowest_index():
    H, V = 256, 3000
    W = synth.normal_bf16(8, "lm", (V, H), 0, 0.02)
    g = synth.normal_bf16(8, "gf", (H,), 1.0, 0.02)
    r = act(9, "r", (1, H))
    # find the winner, then plant copies of its row earlier and later in the vocabulary
    tok = torch.empty(1, dtype=torch.int32, device="cuda")
    gd.dec_lmhead_argmax(dev_f32(r), dev_bf16(g), 1e-6, dev_bf16(W), tok)
    w = int(tok.item())
    for first in (0, 1234, V - 1):
        W2 = W.copy()
        W2[first] = W[w]
        W2[V - 1 if first != V - 1 else 0] = W[w]
        gd.dec_lmhead_argmax(dev_f32(r), dev_bf16(g), 1e-6, dev_bf16(W2), tok)
        assert int(tok.item()) == min(first, w, V - 1 if first != V - 1 else 0)


@pytest.mark.parametrize("B,Hq,Hkv,D,pos", [
    (3, 4, 2, 64, [40, 17, 64]),          # fewer tiles than SMs: one tile per CTA, the 2-tile item split
    (5, 12, 3, 128, [8191, 0, 76, 2999, 4095]),
    (16, 12, 3, 128, [511] * 16),
    (4, 32, 2, 128, [300, 1, 5000, 64]),  # 16-head groups
    (3, 8, 1, 128, [20000, 5, 5]),        # one row cut across ~150 CTAs (their partials merged), 8-head groups
])
def test_attention_balanced_schedule_rows(B, Hq, Hkv, D, pos):
    """b > 2 with more split work items than one wave (64 splits requested)
    takes the balanced schedule (one CTA per SM over the rows' tiles laid end
    to end; items cut between CTAs merge their partials): every row against
    the oracle, and twice the same bits."""
    S_max = max(pos) + 8
    Kb, Vb, q, o = _attn_case(B, Hq, Hkv, D, S_max, pos, seed=11)
    Kd, Vd, qd, pd = dev_bf16(Kb), dev_bf16(Vb), dev_f32(q), dev_i32(pos)
    ws = gd.dec_gqa_decode_attn(qd, Kd, Vd, pd, o, num_splits=64)
    o2 = torch.empty_like(o)
    gd.dec_gqa_decode_attn(qd, Kd, Vd, pd, o2, ws=ws, num_splits=64)
    assert torch.equal(o, o2)
    for b in range(B):
        assert rel_err(o[b].cpu().numpy(), oracle.attention(q[b], Kb[b], Vb[b], pos[b] + 1)) < 1e-4, b


def test_attention_balanced_schedule_position_outside_cache():
    """A row whose position lies outside the cache contributes no tiles to the
    balanced schedule: the error bit is set, nothing is read for it, and the
    other rows are still right."""
    B, Hq, Hkv, D, S_max = 4, 16, 4, 128, 2048
    pos = [2047, S_max, 900, 0]
    Kb, Vb, q, o = _attn_case(B, Hq, Hkv, D, S_max, [2047, 0, 900, 0], seed=12)
    o.zero_()
    gd.dec_gqa_decode_attn(dev_f32(q), dev_bf16(Kb), dev_bf16(Vb), dev_i32(pos), o, num_splits=64)
    assert gd.device_error(clear=True) & 4
    for b in (0, 2, 3):
        assert rel_err(o[b].cpu().numpy(), oracle.attention(q[b], Kb[b], Vb[b], pos[b] + 1)) < 1e-4, b
