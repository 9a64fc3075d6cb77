"""Pins of the oracle's token selection (repetition penalty, temperature, top-k,
top-p and the inverse-CDF draw) against hand-worked cases, brute force over
subsets and the frequencies the draw must produce.

The selection follows the sampling path of the rollout engine on the
segment-KI pull request (its generate fallback takes do_sample / temperature /
top_p; a repetition penalty is applied before the token selector), with the
processors' definitions as Hugging Face generate documents them.
"""
import itertools
import math

import numpy as np
import pytest

import oracle


def f32(a):
    return np.asarray(a, dtype=np.float32)


def frequencies(logits, n=4000, **kw):
    """Share of a uniform grid of draws u = (i + 1/2) / n mapped to each token."""
    V = len(logits)
    counts = np.zeros(V)
    for i in range(n):
        t, _, _ = oracle.select_token(f32(logits), u=(i + 0.5) / n, **kw)
        counts[t] += 1
    return counts / n


def softmax(z, T):
    m = max(z)
    e = [math.exp((float(x) - float(m)) / T) for x in z]
    s = sum(e)
    return [x / s for x in e]


# ----------------------------------------------------------------------------- greedy and penalty

def test_greedy_picks_lowest_index_of_the_maximum():
    assert oracle.select_token(f32([1, 5, 5, 2]))[0] == 1
    assert oracle.select_token(f32([7, 5, 7, 7]))[0] == 0
    assert oracle.select_token(f32([-3, -1, -2]))[0] == 1
    # -0 and +0 are one value: a tie, lowest index wins
    assert oracle.select_token(f32([-1.0, -0.0, 0.0]))[0] == 1


def test_repetition_penalty_divides_positive_and_multiplies_negative_logits():
    # 2.0 / 1.2 = 1.667 falls below 1.9
    assert oracle.select_token(f32([2.0, 1.9]), prev=[0], penalty=1.2)[0] == 1
    # -1.0 * 1.2 = -1.2 falls below -1.1
    assert oracle.select_token(f32([-1.0, -1.1]), prev=[0], penalty=1.2)[0] == 1
    # a penalty below 1 favours the listed token instead
    assert oracle.select_token(f32([1.0, 1.1]), prev=[0], penalty=0.8)[0] == 0
    # without the listed token nothing changes
    assert oracle.select_token(f32([2.0, 1.9]), prev=[1], penalty=1.2)[0] == 0


def test_repetition_penalty_counts_each_id_once_and_ignores_out_of_range_ids():
    # once: 2.0 / 1.2 = 1.667 > 1.5; three times would give 1.157 < 1.5
    assert oracle.select_token(f32([2.0, 1.5]), prev=[0, 0, 0], penalty=1.2)[0] == 0
    assert oracle.select_token(f32([2.0, 1.9]), prev=[0, 0], penalty=1.2)[0] == 1
    assert oracle.select_token(f32([2.0, 1.9]), prev=[-1, 2, 7], penalty=1.2)[0] == 0


# ----------------------------------------------------------------------------- the draw

def test_draw_frequencies_equal_the_softmax_at_the_temperature():
    rng = np.random.default_rng(5)
    z = f32(rng.standard_normal(7) * 2)
    for T in (0.5, 1.0, 1.7):
        got = frequencies(z, temperature=T)
        want = softmax(z, T)
        assert np.max(np.abs(got - want)) < 2.0 / 4000 + 1e-12, (T, got, want)


def test_draw_walks_the_vocabulary_in_index_order():
    # u = 0 lands on the first kept token by index, not the most probable one
    assert oracle.select_token(f32([0, 5, 1]), temperature=1.0, u=0.0)[0] == 0
    assert oracle.select_token(f32([0, 5, 1]), temperature=1.0, top_k=2, u=0.0)[0] == 1
    # two equal weights split [0, 1) at one half
    assert oracle.select_token(f32([3, 3]), temperature=1.0, u=0.4999)[0] == 0
    assert oracle.select_token(f32([3, 3]), temperature=1.0, u=0.5001)[0] == 1
    # the split point itself belongs to the upper token: [0, 1/2) and [1/2, 1)
    assert oracle.select_token(f32([3, 3]), temperature=1.0, u=0.5)[0] == 1


def test_temperature_divides_the_logits():
    # logits a at temperature T and 2a at 2T are the same distribution
    rng = np.random.default_rng(6)
    a = f32(rng.standard_normal(9))
    b = f32(2 * a)
    assert np.all(b == 2 * a)
    assert np.array_equal(frequencies(a, temperature=0.7), frequencies(b, temperature=1.4))
    # and at 2a with T the distribution is sharper (the temperature is not ignored)
    assert not np.array_equal(frequencies(a, temperature=0.7), frequencies(b, temperature=0.7))


# ----------------------------------------------------------------------------- top-k

def test_top_k_one_is_greedy_at_any_temperature_and_draw():
    rng = np.random.default_rng(7)
    for _ in range(20):
        z = f32(rng.standard_normal(50))
        g = int(np.argmax(z))
        for T, u in ((0.3, 0.9), (1.0, 0.1), (3.0, 0.55)):
            assert oracle.select_token(z, temperature=T, top_k=1, u=u)[0] == g


def test_top_k_keeps_every_token_tied_at_the_cut():
    z = [1, 3, 3, 2]
    # k = 1 and k = 2 keep both threes (equal weights, half each)
    for k in (1, 2):
        f = frequencies(z, temperature=1.0, top_k=k)
        assert f[0] == 0 and f[3] == 0 and f[1] == pytest.approx(0.5) and f[2] == pytest.approx(0.5)
    # k = 3 adds the two: weights 1, 1, e^-1
    f = frequencies(z, temperature=1.0, top_k=3, n=20000)
    e = math.exp(-1)
    assert f[0] == 0
    assert f[3] == pytest.approx(e / (2 + e), abs=1e-4)


# ----------------------------------------------------------------------------- top-p

def test_top_p_hand_cases_with_and_without_top_k():
    z = f32([math.log(4), math.log(3), math.log(2), math.log(1)])  # weights 4 : 3 : 2 : 1
    keep = lambda **kw: set(np.nonzero(frequencies(z, temperature=1.0, n=2000, **kw))[0].tolist())
    # p*Z = 5: the 4 sits below it (keep 3), the 4+3 = 7 does not (drop 2)
    assert keep(top_p=0.5) == {0, 1}
    # over the top-2 set (Z = 7): p*Z = 3.5 keeps only the first group
    assert keep(top_p=0.5, top_k=2) == {0}
    assert keep(top_p=0.6, top_k=2) == {0, 1}
    # p = 1 keeps everything; a tiny p keeps the maximum only
    assert keep(top_p=1.0) == {0, 1, 2, 3}
    assert keep(top_p=1e-6) == {0}


def test_top_p_drops_a_group_whose_larger_mass_equals_the_cut_exactly():
    # weights 1, 1, e^-1 (Z summed in index order); p chosen so that p*Z is
    # exactly 2, the weight above the last token: "below p*Z" fails, so it is
    # dropped, as a cumulative ascending share equal to 1 - p is removed.
    Z = (1.0 + 1.0) + math.exp(-1.0)
    p = 2.0 / Z
    while p * Z != 2.0:
        p = math.nextafter(p, 0.0 if p * Z > 2.0 else 1.0)
    f = frequencies([3, 3, 2], temperature=1.0, top_p=p, n=1000)
    assert f[2] == 0 and f[0] == pytest.approx(0.5) and f[1] == pytest.approx(0.5)


def brute_force_nucleus(z, T, p):
    """Smallest set closed upwards in the logit order whose softmax mass reaches p,
    found by enumerating every subset (distinct logits)."""
    V = len(z)
    w = softmax(z, T)
    best = None
    for r in range(1, V + 1):
        for S in itertools.combinations(range(V), r):
            inside = set(S)
            upward = all(j in inside for i in S for j in range(V) if z[j] > z[i])
            if upward and sum(w[i] for i in S) >= p:
                best = inside
                break
        if best is not None:
            break
    return best, w


def test_top_p_equals_brute_force_smallest_upper_set():
    rng = np.random.default_rng(8)
    checked = 0
    while checked < 25:
        V = int(rng.integers(2, 8))
        z = f32(rng.standard_normal(V) * 1.5)
        if len(set(z.tolist())) < V:
            continue
        T = float(rng.choice([0.6, 1.0, 1.5]))
        p = float(rng.uniform(0.05, 0.98))
        _, mp, _ = oracle.select_token(z, temperature=T, top_p=p, u=0.5)
        if mp < 1e-9:
            continue
        nucleus, w = brute_force_nucleus(z, T, p)
        f = frequencies(z, temperature=T, top_p=p, n=3000)
        assert set(np.nonzero(f)[0].tolist()) == nucleus
        M = sum(w[i] for i in nucleus)
        for i in nucleus:
            assert f[i] == pytest.approx(w[i] / M, abs=2.0 / 3000)
        checked += 1


def test_margins_measure_the_distance_to_the_boundaries():
    z = f32([math.log(4), math.log(3), math.log(2), math.log(1)])
    t, mp, mu = oracle.select_token(z, temperature=1.0, top_p=0.5, u=0.25)
    # p*Z = 5 sits 1 above the first boundary (4) and 2 below the next (7): 1/10
    assert mp == pytest.approx(0.1, rel=1e-6)
    # kept {0, 1}, M = 7; u*M = 1.75 inside token 0's [0, 4): distance 1.75 / 7
    assert t == 0 and mu == pytest.approx(0.25, rel=1e-6)
    t, mp, mu = oracle.select_token(z, u=0.3)
    assert math.isinf(mp) and math.isinf(mu) and t == 0
