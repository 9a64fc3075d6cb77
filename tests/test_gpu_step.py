"""Whole-step parity: dec_step against the fp64 oracle's step on the one-layer
workloads, the fused step against the composition of the single-op calls
(bitwise), greedy tokens against the oracle under teacher forcing, and the
native decode loop's EOS / padding / graph-replay behaviour."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import (MARGIN, TOL, HostModel, assert_close, dev_bf16, dev_f32, dev_i32, host_bits, make_caches,
                     rel_err)

pytestmark = pytest.mark.gpu

gd = pytest.importorskip("greedy_decode_step_gb300")


@pytest.fixture(autouse=True)
def _clean_error_word():
    gd.lib()
    gd.device_error(clear=True)
    yield
    assert gd.device_error(clear=True) == 0


class Pair:
    """A GPU state and an oracle model over the same seeded host buffers."""

    def __init__(self, m, batch, kv_len, S_max, seed=0, embed=True, head=True):
        self.m, self.B, self.S_max = m, batch, S_max
        self.hm = HostModel(m, seed, embed=embed, head=head)
        K, V = make_caches(m, seed, batch, S_max, kv_len)
        self.model = self.hm.to_gpu()
        self.state = gd.State(self.model, batch, S_max, k_cache=[dev_bf16(k) for k in K],
                              v_cache=[dev_bf16(v) for v in V]).init()
        self.state.pos.copy_(dev_i32(kv_len))
        self.orc = oracle.Model(m, self.hm.layers, self.hm.embed, self.hm.final_norm, self.hm.lm_head,
                                [k.copy() for k in K], [v.copy() for v in V])


# ----------------------------------------------------------------------------- one-layer workloads

def test_step_tiny_workload_matches_oracle():
    """One layer + LM head, H=256, 4/2 heads, D=64, 128-token N(0,1) cache,
    residual input N(0,1), one step at position 128 (seed 0)."""
    w = synth.workload("tiny")
    p = Pair(w.model, 1, [128], 160, embed=False)
    x = synth.make_residual(0, 1, w.model.hidden)
    p.state.residual.copy_(dev_f32(x))
    gd.dec_step(p.model, p.state)
    torch.cuda.synchronize()
    tok, logits, r = p.orc.step(0, 128, x_in=x[0])
    assert_close(p.state.residual[0].cpu().numpy(), r, TOL, "final residual")
    assert rel_err(p.state.residual[0].cpu().numpy(), r) < 1e-4
    if oracle.top2_margin(logits) > MARGIN:
        assert int(p.state.token[0]) == tok
    assert int(p.state.pos[0]) == 129
    kg = synth.bf16_to_f32(host_bits(p.state.k_cache[0])[0, :, 128])
    ko = synth.bf16_to_f32(p.orc.kcache[0][0, :, 128])
    assert_close(kg, ko, TOL, "stored key")


def test_step_one_4b_layer_matches_oracle():
    """One 4B-class layer (H=2560, 32/8 heads, D=128, I=9728), 4096-token
    N(0,1) cache, one step at position 4096, no LM head."""
    w = synth.workload("layer4b")
    p = Pair(w.model, 1, [4096], 4100, embed=False, head=False)
    x = synth.make_residual(0, 1, w.model.hidden)
    p.state.residual.copy_(dev_f32(x))
    gd.dec_step(p.model, p.state)
    torch.cuda.synchronize()
    _, _, r = p.orc.step(0, 4096, x_in=x[0])
    e = assert_close(p.state.residual[0].cpu().numpy(), r, TOL, "residual after the layer")
    assert e < 1e-4
    assert int(p.state.pos[0]) == 4097
    for cache, ref in ((p.state.k_cache[0], p.orc.kcache[0]), (p.state.v_cache[0], p.orc.vcache[0])):
        got = host_bits(cache)[0]
        assert np.array_equal(got[:, :4096], ref[0][:, :4096])
        assert_close(synth.bf16_to_f32(got[:, 4096]), synth.bf16_to_f32(ref[0][:, 4096]), TOL, "new slot")


# ----------------------------------------------------------------------------- fused == composed

def _compose(p: Pair, r, K, V, pos, tokens=None):
    """The same step from the single-op entry points."""
    m, B = p.m, p.B
    H, Hq, Hkv, D, I = m.hidden, m.n_heads, m.n_kv_heads, m.head_dim, m.intermediate
    dev = "cuda"
    y = torch.empty((B, H), dtype=torch.float32, device=dev)
    q = torch.empty((B, Hq * D), dtype=torch.float32, device=dev)
    o = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    h = torch.empty((B, I), dtype=torch.float32, device=dev)
    if tokens is not None:
        r.copy_(p.model.embed[tokens.long()].float())
    for l, lw in enumerate(p.model.layers):
        gd.dec_add_rmsnorm(None, r, lw["attn_norm"], y, m.rms_eps)
        gd.dec_qkv_gemv_rope(y, lw["wq"], lw["wk"], lw["wv"], pos, m.rope_theta, q, K[l], V[l])
        gd.dec_gqa_decode_attn(q.view(B, Hq, D), K[l], V[l], pos, o)
        gd.dec_down_gemv(o.view(B, Hq * D), lw["wo"], r)
        gd.dec_add_rmsnorm(None, r, lw["mlp_norm"], y, m.rms_eps)
        gd.dec_glu_gemv(y, lw["wg"], lw["wu"], h)
        gd.dec_down_gemv(h, lw["wd"], r)
    tok = torch.empty(B, dtype=torch.int32, device=dev)
    gd.dec_lmhead_argmax(r, p.model.final_norm, m.rms_eps, p.model.lm_head, tok)
    return tok


def _fused_vs_composed(case):
    if case == "tiny2_b2":
        m = synth.workload("tiny", n_layers=2).model
        B, kv = 2, [128, 60]
    elif case == "tiny2_b3":
        m = synth.workload("tiny", n_layers=2).model
        B, kv = 3, [128, 5, 60]
    elif case == "4b1":
        m = synth.workload("layer4b", vocab=4096).model
        B, kv = 1, [700]
    else:
        m = synth.workload("gqa12x3", n_layers=1, vocab=2048).model
        B, kv = 5, [8192, 1, 77, 3000, 4096]
    S_max = max(kv) + 8
    p = Pair(m, B, kv, S_max)
    tokens = synth.make_tokens(1, "t", (B,), m.vocab)
    p.state.token.copy_(dev_i32(tokens))
    K2 = [k.clone() for k in p.state.k_cache]
    V2 = [v.clone() for v in p.state.v_cache]
    pos2 = p.state.pos.clone()
    r2 = torch.empty_like(p.state.residual)
    gd.dec_step(p.model, p.state)
    tok2 = _compose(p, r2, K2, V2, pos2, tokens=dev_i32(tokens))
    torch.cuda.synchronize()
    return p, m, B, kv, r2, tok2, K2, V2, pos2


@pytest.mark.parametrize("case", ["tiny2_b2", "4b1"])
def test_fused_step_equals_composed_calls_bitwise(case):
    """b <= 2: the persistent step kernel computes exactly (bit for bit) what
    the single-op entry points compute one after the other."""
    p, m, B, kv, r2, tok2, K2, V2, pos2 = _fused_vs_composed(case)
    assert p.model is not None and gd.dec_step_launches(p.model, p.state) == 1
    assert torch.equal(p.state.residual, r2)
    assert torch.equal(p.state.token, tok2)
    for a, b in zip(p.state.k_cache + p.state.v_cache, K2 + V2):
        assert torch.equal(a, b)
    assert torch.equal(p.state.pos, pos2 + 1)


@pytest.mark.parametrize("case", ["tiny2_b3", "gqa12x3_b5"])
def test_gemm_step_matches_composed_calls(case):
    """b > 2: the step's weight GEMVs run as tensor-core GEMMs over the batch
    (activations split into hi/lo bf16 parts); it agrees with the single-op
    entry points within the tolerance, token for token where the logit
    margin is clear, and touches the same cache slots."""
    p, m, B, kv, r2, tok2, K2, V2, pos2 = _fused_vs_composed(case)
    assert_close(p.state.residual.cpu().numpy(), r2.cpu().numpy(), TOL, "residual")
    for l in range(m.n_layers):
        for a, b, what in ((p.state.k_cache[l], K2[l], "K"), (p.state.v_cache[l], V2[l], "V")):
            ga, gb = host_bits(a), host_bits(b)
            for row in range(B):
                pp = kv[row]
                assert np.array_equal(np.delete(ga[row], pp, axis=1), np.delete(gb[row], pp, axis=1)), what
                assert_close(synth.bf16_to_f64(ga[row][:, pp]), synth.bf16_to_f64(gb[row][:, pp]), TOL, what)
    logits = torch.empty((B, m.vocab), dtype=torch.float32, device="cuda")
    t3 = torch.empty(B, dtype=torch.int32, device="cuda")
    gd.dec_lmhead_argmax(r2, p.model.final_norm, m.rms_eps, p.model.lm_head, t3, logits)
    lg = logits.cpu().numpy()
    got, ref = p.state.token.cpu().numpy(), tok2.cpu().numpy()
    for row in range(B):
        if oracle.top2_margin(lg[row]) > MARGIN:
            assert got[row] == ref[row], row
    assert torch.equal(p.state.pos, pos2 + 1)


# ----------------------------------------------------------------------------- tokens under teacher forcing

def _oracle_free_run(p: Pair, prompt, n_steps):
    """The oracle's own greedy run: tokens, margins and final residuals per decode step."""
    B, P = prompt.shape
    toks, margins, resid = np.zeros((B, n_steps), np.int64), np.zeros((B, n_steps)), []
    for b in range(B):
        rb = []
        for i in range(P - 1):
            p.orc.step(b, i, token=int(prompt[b, i]))
        t = int(prompt[b, P - 1])
        for s in range(n_steps):
            t_next, logits, r = p.orc.step(b, P - 1 + s, token=t)
            toks[b, s], margins[b, s] = t_next, oracle.top2_margin(logits)
            rb.append(r)
            t = t_next
        resid.append(rb)
    return toks, margins, resid


@pytest.mark.parametrize("case", ["tiny3_b2", "4b_4layers"])
def test_teacher_forced_tokens_match_oracle(case):
    if case == "tiny3_b2":
        m = synth.workload("tiny", n_layers=3).model
        B, P, n = 2, 7, 10
    else:
        m = synth.workload("dense4b", n_layers=4).model
        B, P, n = 1, 6, 6
    p = Pair(m, B, [0] * B, P + n + 4)
    prompt = synth.make_tokens(3, "prompt", (B, P), m.vocab)
    toks, margins, resid = _oracle_free_run(p, prompt, n)
    gd.dec_prefill(p.model, p.state, dev_i32(prompt))
    checked = 0
    for s in range(n):
        gd.dec_step(p.model, p.state)
        got = p.state.token.cpu().numpy()
        for b in range(B):
            # the prompt pass runs its GEMMs on hi/lo bf16 parts of the fp32
            # activations and stores K/V as bf16, so its cache differs from
            # the oracle's by roundings of that order
            assert_close(p.state.residual[b].cpu().numpy(), resid[b][s], TOL, f"residual step {s} row {b}")
            if margins[b, s] > MARGIN:
                assert got[b] == toks[b, s], f"step {s} row {b}: gpu {got[b]} oracle {toks[b, s]}"
                checked += 1
        p.state.token.copy_(dev_i32(toks[:, s]))  # teacher forcing with the oracle's tokens
    assert checked >= (B * n) // 2


# ----------------------------------------------------------------------------- decode loop

def _fresh(m, B, S_max, seed=0):
    return Pair(m, B, [0] * B, S_max, seed=seed)


def test_decode_loop_graph_equals_eager_steps_and_is_deterministic():
    m = synth.workload("tiny", n_layers=2).model
    B, P, n = 3, 5, 40
    prompt = synth.make_tokens(4, "prompt", (B, P), m.vocab)
    outs = []
    for _ in range(2):
        p = _fresh(m, B, P + n + 1)
        out = torch.full((B, n), -7, dtype=torch.int32, device="cuda")
        done = gd.dec_generate(p.model, p.state, dev_i32(prompt), n, -1, out)
        assert done == n
        outs.append(out.cpu().numpy())
    assert np.array_equal(outs[0], outs[1])
    p = _fresh(m, B, P + n + 1)
    gd.dec_prefill(p.model, p.state, dev_i32(prompt))
    eager = []
    for _ in range(n):
        gd.dec_step(p.model, p.state)
        eager.append(p.state.token.cpu().numpy().copy())
    assert np.array_equal(np.stack(eager, 1), outs[0])
    assert np.all(p.state.pos.cpu().numpy() == P - 1 + n)


def test_eos_stops_every_16_steps_and_pads_on_device():
    m = synth.workload("tiny", n_layers=1).model
    B, P, n = 2, 4, 64
    prompt = synth.make_tokens(5, "prompt", (B, P), m.vocab)
    p = _fresh(m, B, P + n + 1)
    ref = torch.empty((B, n), dtype=torch.int32, device="cuda")
    gd.dec_generate(p.model, p.state, dev_i32(prompt), n, -1, ref)
    ref = ref.cpu().numpy()
    # pick as end token one that row 0 emits at step k0 >= 1 and see what happens
    eos = int(ref[0, 3])
    first = [int(np.argmax(ref[b] == eos)) if np.any(ref[b] == eos) else None for b in range(B)]
    p = _fresh(m, B, P + n + 1)
    out = torch.full((B, n), -7, dtype=torch.int32, device="cuda")
    done = gd.dec_generate(p.model, p.state, dev_i32(prompt), n, eos, out)
    out = out.cpu().numpy()
    if all(f is not None for f in first):
        last = max(first)
        assert done == min(n, 16 * ((last + 1 + 15) // 16))
    else:
        assert done == n
    for b in range(B):
        f = first[b]
        if f is None:
            assert np.array_equal(out[b], ref[b])
        else:
            assert np.array_equal(out[b, :f + 1], ref[b, :f + 1])
            assert np.all(out[b, f + 1:] == eos)


def test_decode_rejects_bad_arguments():
    m = synth.workload("tiny").model
    p = _fresh(m, 1, 32)
    with pytest.raises(gd.DecError, match="eos_id"):
        gd.dec_decode(p.model, p.state, 4, m.vocab, None)
    with pytest.raises(gd.DecError, match="n_steps"):
        gd.dec_decode(p.model, p.state, -1, 0, None)
    assert gd.dec_decode(p.model, p.state, 0, 0, None) == 0


def test_step_launch_count():
    """One launch per step while the persistent kernel applies (b <= 2); above
    that the step's own kernels: 1 embedding gather; per layer 4 (two norms,
    RoPE + cache store, attention) around 4 tensor-core GEMMs (split-K
    partials are added inside the GEMM, the attention writes the o_proj
    operand, the gate/up GEMM applies SiLU * up in its epilogue); then the
    final norm, the LM-head GEMM, the row argmax and the bookkeeping."""
    m = synth.workload("tiny", n_layers=2).model
    for B, want in ((1, {1}), (2, {1}), (3, {1 + 2 * (4 + 4) + 4})):
        p = _fresh(m, B, 64)
        assert gd.dec_step_launches(p.model, p.state) in want


@pytest.mark.parametrize("case", ["tiny2_b2_chunks", "gqa12x3_b3"])
def test_batched_prompt_pass_matches_oracle_cache(case):
    """The prompt pass (positions 0..P-2 as rows of GEMMs, in chunks when the
    prompt is longer than a chunk) leaves every layer's K/V cache entries of
    the prompt positions within the tolerance of the oracle's teacher-forced
    steps, sets token = prompt[:, P-1], advances pos by P-1, and writes no
    other cache slot."""
    if case == "tiny2_b2_chunks":
        m = synth.workload("tiny", n_layers=2).model
        B, kv, P = 2, [5, 40], 300          # 512 rows per chunk: 256 positions per chunk at b=2
    else:
        m = synth.workload("gqa12x3", n_layers=2, vocab=2048).model
        B, kv, P = 3, [100, 0, 33], 24
    S_max = max(kv) + P + 4
    p = Pair(m, B, kv, S_max)
    prompt = synth.make_tokens(11, "prompt", (B, P), m.vocab)
    before_k = [host_bits(k).copy() for k in p.state.k_cache]
    gd.dec_prefill(p.model, p.state, dev_i32(prompt))
    torch.cuda.synchronize()
    for b in range(B):
        for i in range(P - 1):
            p.orc.step(b, kv[b] + i, token=int(prompt[b, i]))
    assert np.array_equal(p.state.token.cpu().numpy(), prompt[:, P - 1])
    assert np.array_equal(p.state.pos.cpu().numpy(), np.array(kv) + P - 1)
    for l in range(m.n_layers):
        kg, vg = host_bits(p.state.k_cache[l]), host_bits(p.state.v_cache[l])
        for b in range(B):
            sl = slice(kv[b], kv[b] + P - 1)
            assert_close(synth.bf16_to_f64(kg[b][:, sl]), synth.bf16_to_f64(p.orc.kcache[l][b][:, sl]), TOL,
                         f"K layer {l} row {b}")
            assert_close(synth.bf16_to_f64(vg[b][:, sl]), synth.bf16_to_f64(p.orc.vcache[l][b][:, sl]), TOL,
                         f"V layer {l} row {b}")
            # slots before the prompt and after it are untouched
            assert np.array_equal(kg[b][:, :kv[b]], before_k[l][b][:, :kv[b]])
            assert np.array_equal(kg[b][:, kv[b] + P - 1:], before_k[l][b][:, kv[b] + P - 1:])


# ----------------------------------------------------------------------------- bounded waits

def test_step_kernel_wait_runs_out_and_the_next_step_is_clean():
    """A hold word that nothing clears (dec_state_set_wait) makes the step
    kernel's first wait for other CTAs run out after 1 ms: error bit 64 is
    set, the launch ends instead of hanging, and the decode loop reports
    DEC_EDEVICE.  With the hold removed and the inputs restored, the next
    step is bit for bit the step of a state that never failed."""
    m = synth.workload("tiny", n_layers=2).model
    p = Pair(m, 1, [128], 160)
    ref = Pair(m, 1, [128], 160)
    assert gd.dec_step_launches(p.model, p.state) == 1
    tokens = dev_i32(synth.make_tokens(3, "t", (1,), m.vocab))
    K0 = [k.clone() for k in p.state.k_cache]
    V0 = [v.clone() for v in p.state.v_cache]
    p.state.token.copy_(tokens)
    gd.dec_state_set_wait(p.model, p.state, 1_000_000, hold=True)
    gd.dec_step(p.model, p.state)
    torch.cuda.synchronize()
    assert gd.device_error(clear=True) & 64
    # the decode loop reports the error (and its steps also end)
    out = torch.empty((1, 16), dtype=torch.int32, device="cuda")
    with pytest.raises(gd.DecError) as exc:
        gd.dec_decode(p.model, p.state, 16, -1, out)
    assert exc.value.code == gd.DEC_EDEVICE
    assert gd.device_error(clear=True) & 64
    # hold removed, inputs back: the same step as a state that never failed
    gd.dec_state_set_wait(p.model, p.state, 0, hold=False)
    for a, b in zip(p.state.k_cache + p.state.v_cache, K0 + V0):
        a.copy_(b)
    p.state.pos.fill_(128)
    p.state.token.copy_(tokens)
    ref.state.token.copy_(tokens)
    gd.dec_step(p.model, p.state)
    gd.dec_step(ref.model, ref.state)
    torch.cuda.synchronize()
    assert torch.equal(p.state.residual, ref.state.residual)
    assert torch.equal(p.state.token, ref.state.token)
    assert torch.equal(p.state.pos, ref.state.pos)
    for a, b in zip(p.state.k_cache + p.state.v_cache, ref.state.k_cache + ref.state.v_cache):
        assert torch.equal(a, b)
