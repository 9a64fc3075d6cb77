"""The gated-attention layer (PR 8602, review "Two more decode-path
suggestions", item 1: per-head q/k RMSNorm with an effective gain, partial
rotate-half RoPE, attention output times sigmoid(Wgate y) before o_proj) on
the GPU against the oracle's orc_layer_ex / orc_step_ex: each part alone and
all together, one layer and whole steps, the decode loop under teacher
forcing and the batched prompt pass."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import MARGIN, TOL, HostModel, assert_close, dev_bf16, dev_f32, dev_i32, host_bits, make_caches

pytestmark = pytest.mark.gpu

gd = pytest.importorskip("greedy_decode_step_gb300")


@pytest.fixture(autouse=True)
def _clean_error_word():
    gd.lib()
    gd.device_error(clear=True)
    yield
    assert gd.device_error(clear=True) == 0


def variants(m, seed, rot_dim, parts=("q_norm", "k_norm", "wgate")):
    """Per-layer gated parts (synth recipe), keeping only `parts`."""
    out = []
    for l in range(m.n_layers):
        v = synth.make_gated_attention(seed, m, l, rot_dim)
        out.append({k: x for k, x in v.items() if k == "rot_dim" or k in parts})
    return out


class GatedPair:
    """A GPU state and an oracle model over the same seeded host buffers, with
    the same gated-attention parts on every layer."""

    def __init__(self, m, batch, kv_len, S_max, var, seed=0, embed=True, head=True):
        self.m, self.B = m, batch
        self.hm = HostModel(m, seed, embed=embed, head=head)
        K, V = make_caches(m, seed, batch, S_max, kv_len)
        gpu_layers = []
        for l, lay in enumerate(self.hm.layers):
            d = {k: dev_bf16(v) for k, v in lay.items()}
            d["rot_dim"] = var[l].get("rot_dim", 0)
            for k in ("q_norm", "k_norm", "wgate"):
                if var[l].get(k) is not None:
                    d[k] = dev_bf16(var[l][k])
            gpu_layers.append(d)
        E = dev_bf16(self.hm.embed) if self.hm.embed is not None else None
        fn = dev_bf16(self.hm.final_norm) if self.hm.final_norm is not None else None
        self.model = gd.Model(m.n_layers, m.hidden, m.n_heads, m.n_kv_heads, m.head_dim, m.intermediate, m.vocab,
                              m.rms_eps, m.rope_theta, gpu_layers, embed=E if embed else None, final_norm=fn,
                              lm_head=E if head else None)
        self.state = gd.State(self.model, batch, S_max, k_cache=[dev_bf16(k) for k in K],
                              v_cache=[dev_bf16(v) for v in V]).init()
        self.state.pos.copy_(dev_i32(kv_len))
        self.orc = oracle.Model(m, self.hm.layers, self.hm.embed, self.hm.final_norm, self.hm.lm_head,
                                [k.copy() for k in K], [v.copy() for v in V], variants=var)


@pytest.mark.parametrize("rot_dim,parts", [
    (32, ()),                                 # partial rotary alone
    (0, ("q_norm",)),                         # query head norm alone
    (0, ("k_norm",)),                         # key head norm alone
    (0, ("wgate",)),                          # output gate alone
    (32, ("q_norm", "k_norm", "wgate")),      # all together
    (2, ("q_norm", "k_norm", "wgate")),       # the narrowest rotary
])
def test_gated_tiny_layer_matches_oracle(rot_dim, parts):
    """One gated layer + LM head (H=256, 4/2 heads, D=64), 128-token N(0,1)
    cache, residual input N(0,1), one step at position 128."""
    m = synth.workload("tiny").model
    p = GatedPair(m, 1, [128], 160, variants(m, 0, rot_dim, parts), embed=False)
    x = synth.make_residual(0, 1, m.hidden)
    p.state.residual.copy_(dev_f32(x))
    gd.dec_step(p.model, p.state)
    torch.cuda.synchronize()
    tok, logits, r = p.orc.step(0, 128, x_in=x[0])
    assert_close(p.state.residual[0].cpu().numpy(), r, TOL, "final residual")
    if oracle.top2_margin(logits) > MARGIN:
        assert int(p.state.token[0]) == tok
    kg = synth.bf16_to_f32(host_bits(p.state.k_cache[0])[0, :, 128])
    ko = synth.bf16_to_f32(p.orc.kcache[0][0, :, 128])
    assert_close(kg, ko, TOL, "stored key (normed, partially rotated)")


def test_gated_4b_layer_matches_oracle():
    """One gated 4B-class layer (H=2560, 32/8 heads, D=128, rotary over 64 of
    128 dims), 4096-token cache, one step at position 4096."""
    m = synth.workload("layer4b").model
    p = GatedPair(m, 1, [4096], 4100, variants(m, 0, 64), embed=False, head=False)
    x = synth.make_residual(0, 1, m.hidden)
    p.state.residual.copy_(dev_f32(x))
    gd.dec_step(p.model, p.state)
    torch.cuda.synchronize()
    _, _, r = p.orc.step(0, 4096, x_in=x[0])
    assert_close(p.state.residual[0].cpu().numpy(), r, TOL, "residual after the gated layer")
    for cache, ref in ((p.state.k_cache[0], p.orc.kcache[0]), (p.state.v_cache[0], p.orc.vcache[0])):
        got = host_bits(cache)[0]
        assert np.array_equal(got[:, :4096], ref[0][:, :4096])
        assert_close(synth.bf16_to_f32(got[:, 4096]), synth.bf16_to_f32(ref[0][:, 4096]), TOL, "new slot")


@pytest.mark.parametrize("B", [1, 3])
def test_gated_decode_teacher_forced(B):
    """Two gated layers (H=256, 4/2 heads, D=64, rotary over 32 dims) with an
    embedding and a tied LM head: four decode steps through dec_decode from
    ragged cache lengths, each step's tokens fed back on both sides; tokens
    agree wherever the oracle's top-2 margin exceeds 1e-2 and the final
    residual stays within tolerance."""
    m = synth.ModelShape(2, 256, 4, 2, 64, 704, 1024, gain_std=0.1)
    kv = [40, 17, 63][:B]
    p = GatedPair(m, B, kv, 80, variants(m, 1, 32), seed=1)
    t0 = synth.make_tokens(1, "gated.t0", (B,), m.vocab)
    p.state.token.copy_(dev_i32(t0))
    n = 4
    out = torch.empty((B, n), dtype=torch.int32, device="cuda")
    gd.dec_decode(p.model, p.state, n, -1, out)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    for b in range(B):
        tok = int(t0[b])
        for i in range(n):
            want, logits, _ = p.orc.step(b, kv[b] + i, token=tok)
            if oracle.top2_margin(logits) > MARGIN:
                assert int(got[b, i]) == want, f"row {b} step {i}"
            tok = int(got[b, i])  # teacher forcing: the GPU's token goes on
        kg = synth.bf16_to_f32(host_bits(p.state.k_cache[1])[b, :, kv[b] + n - 1])
        ko = synth.bf16_to_f32(p.orc.kcache[1][b, :, kv[b] + n - 1])
        assert_close(kg, ko, TOL, f"row {b}: last stored key of layer 1")


def test_gated_prompt_pass_fills_the_cache_like_the_oracle():
    """dec_prefill of a 24-token prompt through two gated layers (batched
    rows, tensor-core GEMMs): every stored key and value equals the oracle's
    step-by-step prompt pass within tolerance, and the state ends at the
    prompt's last token."""
    m = synth.ModelShape(2, 256, 4, 2, 64, 704, 1024, gain_std=0.1)
    B, P = 2, 24
    p = GatedPair(m, B, [0, 0], 40, variants(m, 2, 32), seed=2)
    prompt = synth.make_tokens(2, "gated.prompt", (B, P), m.vocab)
    gd.dec_prefill(p.model, p.state, dev_i32(prompt))
    torch.cuda.synchronize()
    for b in range(B):
        for i in range(P - 1):
            p.orc.step(b, i, token=int(prompt[b, i]))
    for l in range(m.n_layers):
        for cache, ref in ((p.state.k_cache[l], p.orc.kcache[l]), (p.state.v_cache[l], p.orc.vcache[l])):
            got = synth.bf16_to_f32(host_bits(cache)[:, :, :P - 1])
            want = synth.bf16_to_f32(ref[:, :, :P - 1])
            assert_close(got, want, TOL, f"layer {l} cache")
    assert p.state.pos.cpu().tolist() == [P - 1] * B
    assert p.state.token.cpu().tolist() == [int(prompt[b, P - 1]) for b in range(B)]


def test_gated_model_takes_the_batched_row_path():
    """A gated model at b=1 does not use the persistent step kernel (one
    launch): the step runs as GEMMs and the kernels around them."""
    m = synth.workload("tiny").model
    p = GatedPair(m, 1, [16], 32, variants(m, 0, 32), embed=False)
    assert gd.dec_step_launches(p.model, p.state) > 1
