"""The top-k candidate rule of the selection kernel, checked on the CPU.

The kernel skips its cluster-wide searches when top_k is small: each of the 8
slices of a row keeps only its keys at or above a bound (the top_k-th largest
of its 512 threads' largest keys), and the survivors of the top-k cut are the
candidates with fewer than top_k larger keys among all slices' candidates.
The claim is that this gives exactly the top-k rule's survivor set (v
survives iff fewer than top_k tokens of the whole row have a strictly larger
logit), ties included.  Here that rule is restated with numpy, with the
kernel's slice and thread layout (float4 blocks t, t + 512, ... of a slice
belong to thread t), and compared with the definition written out on random
rows, many of them full of ties.  No GPU is involved.
"""
import numpy as np
import pytest

CLUSTER = 8
THREADS = 512


def chunk_of(V):
    per = -(-V // CLUSTER)
    return -(-per // 64) * 64


def survivors_by_definition(z, k):
    return {v for v in range(len(z)) if int(np.sum(z > z[v])) < k}


def survivors_by_candidates(z, k):
    """The candidate rule; None when a slice's candidates exceed the 256 the
    kernel hands to CTA 0 (the kernel then runs its searches instead)."""
    V = len(z)
    chunk = chunk_of(V)
    lists = []
    for c in range(CLUSTER):
        lo = c * chunk
        n = max(0, min(chunk, V - lo))
        zs = z[lo:lo + n]
        tmax = np.full(THREADS, -np.inf)
        for t in range(THREADS):
            idx = [4 * i4 + e for i4 in range(t, n // 4, THREADS) for e in range(4)]
            if idx:
                tmax[t] = zs[idx].max()
        bound = np.sort(tmax)[::-1][k - 1]  # the k-th largest thread maximum
        cand = [lo + i for i in range(n) if zs[i] >= bound]
        if len(cand) > 256:
            return None
        lists.append(cand)
    union = [v for cand in lists for v in cand]
    keys = np.array([z[v] for v in union])
    return {v for v, kv in zip(union, keys) if int(np.sum(keys > kv)) < k}


@pytest.mark.parametrize("seed", range(12))
def test_candidate_rule_equals_the_top_k_definition(seed):
    rng = np.random.default_rng(seed)
    V = int(rng.choice([8, 64, 1024, 4104, 8192]))
    # integer logits from a small range tie in large groups; a few rows also
    # put every large value into one slice
    z = rng.integers(-6, 7, size=V).astype(np.float64)
    if seed % 3 == 0:
        z[: max(1, V // 8) : 3] += 20.0
    checked = 0
    for k in (1, 2, 3, 5, 16, 50):
        if k >= V:
            continue
        got = survivors_by_candidates(z, k)
        if got is None:
            continue
        assert got == survivors_by_definition(z, k), (V, k)
        checked += 1
    assert checked > 0 or V <= 8


def test_candidate_rule_with_distinct_values():
    """Distinct values: exactly k survivors.  A slice whose threads hold fewer
    than k keys in all gets the bound -inf (every key a candidate), so large
    k on a small vocabulary goes to the searches, as in the kernel."""
    rng = np.random.default_rng(99)
    applied = 0
    for V in (4104, 16384, 65536):
        z = rng.standard_normal(V)
        for k in (1, 7, 50, 200):
            got = survivors_by_candidates(z, k)
            if got is None:
                continue
            assert got == survivors_by_definition(z, k)
            assert len(got) == k
            applied += 1
    assert applied >= 9


def kept_by_definition(w, z, target):
    """Top-p over the whole row: v is kept iff the tokens with a larger logit
    weigh less than the target."""
    return {v for v in range(len(z)) if float(np.sum(w[z > z[v]])) < target}


@pytest.mark.parametrize("seed", range(8))
def test_speculative_top_p_check(seed):
    """Top-p without top-k runs the candidate rule as a top-kc cut: when the
    cut's survivors S already weigh the target, every kept token is in S and
    the kept set computed inside S equals the one over the whole row."""
    rng = np.random.default_rng(100 + seed)
    V = int(rng.choice([1024, 4104, 8192]))
    scale = float(rng.choice([0.5, 2.0, 6.0]))
    z = np.round(rng.standard_normal(V) * scale * 8) / 8  # ties from rounding
    w = np.exp(z - z.max())
    Z = float(np.sum(w))
    decided = 0
    for kc in (16, 64, 128):
        S = survivors_by_candidates(z, kc)
        if S is None:
            continue
        for p in (0.3, 0.9, 0.99):
            target = p * Z
            if float(np.sum(w[sorted(S)])) < target:
                continue  # the kernel would fall back to the searches
            kept = kept_by_definition(w, z, target)
            assert kept <= S
            inside = {v for v in S if float(sum(w[u] for u in S if z[u] > z[v])) < target}
            assert inside == kept
            decided += 1
    assert decided > 0 or scale < 1.0
