"""Token selection on the GPU (dec_select_tokens) against the fp64 oracle.

Greedy choices, the order of tokens and the top-k cut are decided on float32
logits on both sides, so they must agree exactly.  The top-p cut and the draw
compare weights that the kernel sums in float32: a row must agree wherever
the oracle's distance from each decision boundary (relative to the total
weight) is at least AMBIG; nearer a boundary the GPU's token must be one that
the oracle picks for a draw or a p within that distance.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import dev_f32, dev_i32

pytestmark = pytest.mark.gpu

# Relative difference of the kernel's weights from the oracle's: float32
# (z - max) / T and expf (a few ulp, ~1e-6 at |z - max| / T ~ 10), then
# truncation to multiples of 2^-40; the kernel's sums of them are exact
# integers.  The bar keeps a margin above that.
AMBIG = 2e-5
VOCAB = 151936


@pytest.fixture(scope="module")
def gd():
    import greedy_decode_step_gb300 as gd
    gd.build()
    return gd


def run(gd, z, u=None, prev=None, **kw):
    B = z.shape[0]
    out = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    gd.dec_select_tokens(dev_f32(z), out, u=None if u is None else dev_f32(u),
                         prev_tokens=None if prev is None else dev_i32(prev), **kw)
    torch.cuda.synchronize()
    assert gd.device_error(clear=True) == 0
    return out.cpu().numpy()


def oracle_rows(z, u, prev, penalty, temperature, top_k, top_p):
    res = []
    for b in range(z.shape[0]):
        res.append(oracle.select_token(z[b], prev=None if prev is None else prev[b], penalty=penalty,
                                       temperature=temperature, top_k=top_k, top_p=top_p,
                                       u=0.0 if u is None else float(u[b])))
    return res


def nearby_tokens(zb, ub, prevb, penalty, temperature, top_k, top_p):
    """Oracle tokens for draws and p within AMBIG of the given ones."""
    out = set()
    for du in (-AMBIG, 0.0, AMBIG):
        for dp in (-AMBIG, 0.0, AMBIG):
            uu = min(max(ub + du, 0.0), np.nextafter(1.0, 0.0))
            pp = min(top_p + dp, 1.0) if top_p < 1.0 else 1.0
            out.add(oracle.select_token(zb, prev=prevb, penalty=penalty, temperature=temperature, top_k=top_k,
                                        top_p=pp, u=uu)[0])
    return out


def check_rows(got, z, u, prev, penalty, temperature, top_k, top_p, min_exact=0.5):
    ref = oracle_rows(z, u, prev, penalty, temperature, top_k, top_p)
    exact = 0
    for b, (t, mp, mu) in enumerate(ref):
        assert 0 <= got[b] < z.shape[1]
        if min(mp, mu) >= AMBIG:
            assert got[b] == t, f"row {b}: gpu {got[b]} oracle {t} (margins {mp:.2e}, {mu:.2e})"
            exact += 1
        else:
            near = nearby_tokens(z[b], float(u[b]), None if prev is None else prev[b], penalty, temperature, top_k,
                                 top_p)
            assert got[b] in near, f"row {b}: gpu {got[b]} not among {sorted(near)} near a boundary"
    assert exact >= min_exact * len(ref), f"only {exact} of {len(ref)} rows away from every boundary"


# ----------------------------------------------------------------------------- greedy

@pytest.mark.parametrize("V,fine,penalty", [(1024, True, 1.0), (VOCAB, True, 1.0), (VOCAB, False, 1.0),
                                            (VOCAB, True, 1.3), (8, False, 1.3)])
def test_greedy_is_bit_exact(gd, V, fine, penalty):
    B = 4
    z = synth.make_logits(11, f"sel.greedy.{V}", B, V, 2.0, fine)
    prev = synth.uniform_int(11, f"sel.prev.{V}", (B, 64), -3, V + 3)
    # make the penalty decide: list each row's current maximum
    prev[:, 0] = np.argmax(z, axis=1)
    got = run(gd, z, prev=prev, repetition_penalty=penalty)
    for b in range(B):
        assert got[b] == oracle.select_token(z[b], prev=prev[b], penalty=penalty)[0]


def test_greedy_ties_take_the_lowest_index_across_cluster_slices(gd):
    V = VOCAB
    z = np.full((3, V), -5.0, dtype=np.float32)
    z[0, [100_000, 20, 150_000]] = 3.0
    z[1, [151_935, 151_934]] = 1.0
    z[2, :] = -0.0
    z[2, 77] = 0.0  # +0 and -0 tie: index 0 is the first maximum
    got = run(gd, z)
    assert list(got) == [20, 151_934, 0]


# ----------------------------------------------------------------------------- sampling

CASES = [
    # V,     std, fine, T,   top_k, top_p, penalty, share of rows that must match exactly
    (1024, 2.0, True, 1.0, 0, 1.0, 1.0, 0.5),
    (1024, 2.0, True, 0.7, 50, 0.9, 1.2, 0.5),
    # flat: each of the 151,936 tokens holds ~1e-5 of the weight, so every draw
    # lies within AMBIG of a boundary; the rows are checked against their neighbours
    (VOCAB, 1.0, True, 1.0, 0, 1.0, 1.0, 0.0),
    (VOCAB, 4.0, True, 0.7, 0, 0.9, 1.0, 0.5),
    (VOCAB, 4.0, True, 0.7, 50, 0.9, 1.1, 0.5),
    (VOCAB, 3.0, False, 1.0, 40, 0.8, 1.0, 0.5),   # bf16-valued logits: large tie groups
    (VOCAB, 6.0, True, 1.5, 0, 0.5, 1.0, 0.5),
    (VOCAB, 2.0, True, 1.0, 1, 1.0, 1.0, 0.5),
    (VOCAB, 8.0, True, 0.6, 0, 0.95, 1.3, 0.5),
    (4104, 2.0, True, 1.0, 5000, 0.3, 1.0, 0.5),   # top_k >= V: no cut
    (256000, 4.0, True, 0.8, 64, 0.9, 1.0, 0.5),   # 32,000 logits per CTA
    (VOCAB, 2.0, True, 1.0, 1000, 0.9, 1.0, 0.5),  # more top-k candidates than one CTA finishes: cluster path
    (VOCAB, 4.0, True, 0.7, 512, 0.9, 1.0, 0.5),   # exactly the candidates one CTA takes
]


@pytest.mark.parametrize("case", CASES, ids=[f"V{c[0]}_T{c[3]}_k{c[4]}_p{c[5]}_pen{c[6]}_{'f' if c[2] else 'b'}"
                                              for c in CASES])
def test_sampling_matches_oracle(gd, case):
    V, std, fine, T, K, P, pen, share = case
    B = 6
    tag = f"sel.{V}.{std}.{fine}.{T}.{K}.{P}.{pen}"
    z = synth.make_logits(12, tag, B, V, std, fine)
    u = synth.make_uniforms(12, tag + ".u", B)
    prev = synth.uniform_int(12, tag + ".prev", (B, 256), 0, V - 1) if pen != 1.0 else None
    got = run(gd, z, u=u, prev=prev, repetition_penalty=pen, temperature=T, top_k=K, top_p=P)
    check_rows(got, z, u, prev, pen, T, K, float(np.float32(P)), min_exact=share)


def test_many_rows_and_a_large_vocabulary(gd):
    # 40 rows are more clusters than fit the GPU at once with full-length
    # search lists, so the kernel takes the short lists; 400,000 logits put
    # 50,000 in each CTA
    for B, V, K, P in ((40, VOCAB, 50, 0.9), (3, 400_000, 0, 0.8)):
        tag = f"sel.rows.{B}.{V}"
        z = synth.make_logits(17, tag, B, V, 4.0, True)
        u = synth.make_uniforms(17, tag + ".u", B)
        got = run(gd, z, u=u, temperature=0.8, top_k=K, top_p=P)
        check_rows(got, z, u, None, 1.0, 0.8, K, float(np.float32(P)))
        assert np.array_equal(run(gd, z), np.argmax(z, axis=1))


def test_many_draws_over_one_row(gd):
    # one row repeated with a grid of draws: every inverse-CDF interval is hit
    V, B = 64, 512
    z1 = synth.make_logits(13, "sel.grid", 1, V, 1.5, True)
    z = np.repeat(z1, B, axis=0)
    u = ((np.arange(B) + 0.5) / B).astype(np.float32)
    for K, P in ((0, 1.0), (10, 0.9), (0, 0.6)):
        got = run(gd, z, u=u, temperature=0.8, top_k=K, top_p=P)
        check_rows(got, z, u, None, 1.0, 0.8, K, float(np.float32(P)), min_exact=0.9)


def test_draw_edges_and_masked_logits(gd):
    V = 4104
    z = synth.make_logits(14, "sel.edges", 4, V, 1.0, True)
    z[2, :] = -np.inf
    z[2, 4000] = 0.5          # one finite logit: always chosen
    z[3, ::2] = -np.inf       # half the vocabulary masked
    u = np.array([0.0, np.nextafter(np.float32(1), np.float32(0)), 0.3, 0.7], dtype=np.float32)
    got = run(gd, z, u=u, temperature=1.0)
    ref = oracle_rows(z, u, None, 1.0, 1.0, 0, 1.0)
    assert got[0] == ref[0][0] == 0           # u = 0: the first token with weight
    assert got[2] == 4000
    assert got[3] % 2 == 1
    check_rows(got, z, u, None, 1.0, 1.0, 0, 1.0)


def test_small_vocabulary_uses_one_slice(gd):
    z = np.array([[0.0, 1.0, 2.0, 3.0, -1.0, 0.5, 2.5, 1.5]] * 3, dtype=np.float32)
    u = np.array([0.01, 0.5, 0.99], dtype=np.float32)
    got = run(gd, z, u=u, temperature=1.0, top_k=3)
    check_rows(got, z, u, None, 1.0, 1.0, 3, 1.0, min_exact=1.0)


def test_selection_is_reproducible(gd):
    B, V = 8, VOCAB
    z = synth.make_logits(15, "sel.repro", B, V, 3.0, True)
    u = synth.make_uniforms(15, "sel.repro.u", B)
    kw = dict(temperature=0.9, top_k=100, top_p=0.9)
    a = run(gd, z, u=u, **kw)
    b = run(gd, z, u=u, **kw)
    assert np.array_equal(a, b)


def test_greedy_selection_of_lmhead_logits_equals_its_argmax(gd):
    B, H, V = 3, 256, 1024
    W = synth.normal_bf16(16, "sel.lm", (V, H), 0.0, 0.05)
    g = synth.normal_bf16(16, "sel.gain", (H,), 1.0, 0.1)
    r = synth.make_residual(16, B, H)
    from helpers import dev_bf16
    tok = torch.empty(B, dtype=torch.int32, device="cuda")
    logits = torch.empty(B, V, dtype=torch.float32, device="cuda")
    gd.dec_lmhead_argmax(dev_f32(r), dev_bf16(g), 1e-6, dev_bf16(W), tok, logits_out=logits)
    out = torch.empty(B, dtype=torch.int32, device="cuda")
    gd.dec_select_tokens(logits, out)
    torch.cuda.synchronize()
    assert torch.equal(out, tok)


def test_top_k_cut_inside_a_large_tie_group(gd):
    """Top-k keeps every token tied at the cut: with 3 large logits and the
    rest equal, top_k = 5 keeps the whole tie group (more candidates than one
    CTA finishes, so the cluster path decides), and top_k = 3 keeps the three."""
    V, B = VOCAB, 4
    z = np.zeros((B, V), np.float32)
    z[:, [10, 70_000, 151_000]] = [3.0, 2.5, 2.0]
    u = np.array([0.1, 0.5, 0.9, 0.999], dtype=np.float32)
    for K in (5, 3):
        got = run(gd, z, u=u, temperature=1.0, top_k=K)
        # the tie group spreads the draw over ~150,000 near-equal weights: every
        # row lies near a boundary there and is checked against its neighbours
        check_rows(got, z, u, None, 1.0, 1.0, K, 1.0, min_exact=1.0 if K == 3 else 0.0)


@pytest.mark.parametrize("K", [256, 257])
def test_top_k_at_the_candidate_limit(gd, K):
    """top_k = 256 is the largest cut that the candidate path takes (each CTA
    hands at most 256 candidates to CTA 0); 257 goes to the cluster searches.
    Both agree with the oracle on the same rows."""
    V, B = VOCAB, 6
    z = synth.make_logits(18, "sel.cap", B, V, 3.0, True)
    u = synth.make_uniforms(18, "sel.cap.u", B)
    got = run(gd, z, u=u, temperature=0.9, top_k=K, top_p=0.95)
    check_rows(got, z, u, None, 1.0, 0.9, K, float(np.float32(0.95)))


def test_candidates_of_a_cta_below_another_ctas_cut(gd):
    """All large logits in the first CTA's slice: every other CTA's local
    candidates rank below the row's top_k and must drop out when CTA 0 ranks
    them.  With top-p 1 and the draw spread over the survivors, the token must
    be one of the 50 largest."""
    V, B, K = VOCAB, 4, 50
    rng_z = synth.make_logits(19, "sel.skew", B, V, 1.0, True)
    idx = synth.uniform_int(19, "sel.skew.idx", (B, 200), 0, V // 8 - 1)
    z = rng_z.copy()
    for b in range(B):
        z[b, idx[b]] += 8.0
    u = synth.make_uniforms(19, "sel.skew.u", B)
    got = run(gd, z, u=u, temperature=1.0, top_k=K)
    check_rows(got, z, u, None, 1.0, 1.0, K, 1.0)
    for b in range(B):
        top = np.argsort(-z[b], kind="stable")[:K]
        assert got[b] in set(top.tolist()) and got[b] < V // 8


def test_candidate_path_with_masked_logits(gd):
    """Half of the vocabulary at -inf with a small top-k: masked keys never
    become candidates above a finite cut, and the drawn token is finite."""
    V, B = VOCAB, 4
    z = synth.make_logits(20, "sel.mask", B, V, 2.0, True)
    z[:, 1::2] = -np.inf
    u = synth.make_uniforms(20, "sel.mask.u", B)
    got = run(gd, z, u=u, temperature=0.8, top_k=5, top_p=0.9)
    check_rows(got, z, u, None, 1.0, 0.8, 5, float(np.float32(0.9)))
    assert all(int(t) % 2 == 0 for t in got)
