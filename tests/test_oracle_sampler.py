"""Pins for the oracle's fused sampler (CPU only, no GPU).

The sampler (Optimized Parler TTS, "Future work" item 2: temperature scaling,
top-k and softmax fused into one pass; the nine codebooks decoded in parallel
under the delayed pattern, architecture overview) is pinned by:
  * Philox4x32-10 against the published Random123 known-answer vectors;
  * top-k against a brute-force rank count over every value pattern on V=5;
  * k=1 giving the argmax and k=V giving every index;
  * temperature identities (T=1 and powers of two are exact);
  * the delay-pattern invariant;
  * a chi-squared test that the Gumbel-max draw follows softmax over the top-k set;
  * softmax probabilities summing to one on exactly the top-k support;
  * the Gumbel margin, by behaviour: raising another member of the top-k set
    by just more than the margin hands the draw to some member, by just less
    it changes nothing (no score is recomputed here).
"""
import itertools
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.txt")


def _kat_rows():
    rows = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        f = line.split()
        assert f[0] == "10"
        vals = [int(x, 16) for x in f[1:]]
        rows.append((vals[0:4], vals[4:6], vals[6:10]))
    return rows


@pytest.mark.parametrize("ctr,key,expect", _kat_rows())
def test_philox_known_answer_vectors(ctr, key, expect):
    assert [int(x) for x in oracle.philox4x32_10(ctr, key)] == expect


def test_uniform_is_odd_multiple_of_2_pow_minus_24_and_centered():
    us = np.array([oracle.uniform(12345, 1, 2, 3, i) for i in range(20000)])
    assert (us > 0).all() and (us < 1).all()
    m = us * 2 ** 24
    assert np.array_equal(m, np.round(m)) and (np.round(m).astype(np.int64) % 2 == 1).all()
    assert abs(us.mean() - 0.5) < 0.01
    assert abs(us.var() - 1 / 12) < 0.005
    # different seeds, rows, codebooks and steps give different streams
    base = oracle.uniform(1, 0, 0, 0, 0)
    assert len({base, oracle.uniform(2, 0, 0, 0, 0), oracle.uniform(1, 1, 0, 0, 0), oracle.uniform(1, 0, 1, 0, 0),
                oracle.uniform(1, 0, 0, 1, 0), oracle.uniform(1, 0, 0, 0, 1)}) == 6


def _brute_topk(x, k):
    """Rank-count definition: i is kept iff fewer than k entries precede it
    (greater value, or equal value at a lower index)."""
    V = len(x)
    keep = []
    for i in range(V):
        before = sum(1 for j in range(V) if x[j] > x[i] or (x[j] == x[i] and j < i))
        if before < k:
            keep.append(i)
    return keep


def test_topk_matches_brute_force_rank_count_on_all_patterns():
    vals = [-math.inf, -1.0, -0.0, 0.0, 2.0]
    V = 5
    for pat in itertools.product(vals, repeat=V):
        x = np.array(pat, np.float32)
        for k in range(1, V + 1):
            r = oracle.sample_row(x, 1.0, k, 7, 0, 0, 5, 99, want_topk=True)
            assert list(r["topk"]) == _brute_topk(list(x), k), (pat, k)


def test_k1_is_argmax_with_lowest_index_ties():
    rng = np.random.default_rng(3)
    for trial in range(200):
        x = rng.integers(-3, 3, size=16).astype(np.float32)
        r = oracle.sample_row(x, 1.0, 1, trial, 0, 0, 3, -1)
        assert r["token"] == int(np.argmax(x))          # numpy argmax returns the first maximum
        assert r["margin"] == math.inf


def test_k_equals_v_keeps_every_index():
    x = np.random.default_rng(4).normal(size=37).astype(np.float32)
    r = oracle.sample_row(x, 0.8, 37, 1, 0, 0, 3, -1, want_topk=True, want_probs=True)
    assert list(r["topk"]) == list(range(37))
    assert (r["probs"] > 0).all()


def test_temperature_identities():
    rng = np.random.default_rng(5)
    x = (rng.normal(size=(4, 9, 64)) * 3).astype(np.float32)
    seeds = np.arange(4, dtype=np.uint64) + 11
    steps = np.array([9, 12, 30, 100], np.int32)
    a = oracle.sample(x, 1.0, 10, seeds, steps, 1024)
    b = oracle.sample(x.copy(), 1.0, 10, seeds, steps, 1024)
    assert np.array_equal(a["tokens"], b["tokens"])
    # dividing by a power of two is exact, so sampling (x, T=4) == sampling (x/4, T=1) bit for bit
    c = oracle.sample(x, 4.0, 10, seeds, steps, 1024, want_probs=True)
    d = oracle.sample((x / np.float32(4)).astype(np.float32), 1.0, 10, seeds, steps, 1024, want_probs=True)
    assert np.array_equal(c["tokens"], d["tokens"]) and np.array_equal(c["probs"], d["probs"])


def test_topk_is_taken_on_temperature_scaled_floats():
    # Two adjacent float32 logits just below 2 merge under the binary32 division by T=3
    # (their spacing 2^-23 shrinks to 2^-23/3, below the quotient's spacing 2^-24).
    T = np.float32(3.0)
    pair = None
    a = np.float32(1.9)
    for _ in range(64):
        b = np.nextafter(a, np.float32(2), dtype=np.float32)
        if np.float32(a / T) == np.float32(b / T):
            pair = (a, b)
            break
        a = b
    assert pair is not None
    x = np.array([pair[0], pair[1], -5.0], np.float32)   # raw: index 1 is strictly larger
    r = oracle.sample_row(x, float(T), 1, 0, 0, 0, 5, -1)
    assert r["token"] == 0                                # scaled values tie, lower index wins
    r1 = oracle.sample_row(x, 1.0, 1, 0, 0, 0, 5, -1)
    assert r1["token"] == 1


@pytest.mark.parametrize("step", list(range(0, 12)))
def test_delay_pattern_invariant(step):
    C, V, pad = 9, 40, 7
    x = np.random.default_rng(step).normal(size=(1, C, V)).astype(np.float32)
    x[:, :, pad] = -np.inf                              # a drawn token can never equal pad_id
    r = oracle.sample(x, 1.0, 5, np.array([3], np.uint64), np.array([step], np.int32), pad, want_probs=True)
    for c in range(C):
        if step <= c:
            assert r["tokens"][0, c] == pad and (r["probs"][0, c] == 0).all()
        else:
            assert r["tokens"][0, c] != pad and abs(r["probs"][0, c].sum() - 1) < 1e-12


def test_delay_pattern_example_step5_pads_codebooks_5_to_8():
    x = np.random.default_rng(9).normal(size=(1, 9, 1088)).astype(np.float32) * 3
    x[:, :, 1024] = -np.inf
    r = oracle.sample(x, 1.0, 50, np.array([0], np.uint64), np.array([5], np.int32), 1024)
    assert [int(t == 1024) for t in r["tokens"][0]] == [0, 0, 0, 0, 0, 1, 1, 1, 1]


def test_gumbel_max_draw_follows_softmax_over_topk_chi_squared():
    scipy_stats = pytest.importorskip("scipy.stats")
    x = np.array([1.0, 0.3, -0.2, 0.9, -2.0, 0.5], np.float32)
    k, T = 4, 0.8
    r = oracle.sample_row(x, T, k, 0, 0, 0, 1, -1, want_probs=True, want_topk=True)
    K = list(r["topk"])
    p = r["probs"][K]
    N = 30000
    counts = {i: 0 for i in range(len(x))}
    for s in range(1, N + 1):
        counts[oracle.sample_row(x, T, k, 2024, 0, 0, s, -1)["token"]] += 1
    assert sum(counts[i] for i in range(len(x)) if i not in K) == 0
    obs = np.array([counts[i] for i in K], np.float64)
    exp = p * N
    chi2 = float(((obs - exp) ** 2 / exp).sum())
    assert scipy_stats.chi2.sf(chi2, df=k - 1) > 1e-6, (obs, exp, chi2)
    # and the probabilities are the softmax of the scaled values over K
    xs = (x / np.float32(T)).astype(np.float64)[K]
    np.testing.assert_allclose(p, np.exp(xs - xs.max()) / np.exp(xs - xs.max()).sum(), rtol=1e-12)


def test_probs_sum_to_one_on_topk_support():
    rng = np.random.default_rng(10)
    x = (rng.normal(size=(2, 9, 1088)) * 5).astype(np.float32)
    r = oracle.sample(x, 0.7, 250, np.array([1, 2], np.uint64), np.array([20, 20], np.int32), 1024,
                      want_probs=True, want_topk=True)
    for b in range(2):
        for c in range(9):
            pr = r["probs"][b, c]
            assert abs(pr.sum() - 1.0) < 1e-12
            assert sorted(np.nonzero(pr)[0]) == sorted(r["topk"][b, c])
    r1 = oracle.sample(x, 0.7, 1, np.array([1, 2], np.uint64), np.array([20, 20], np.int32), 1024, want_probs=True)
    assert ((r1["probs"] == 0) | (r1["probs"] == 1)).all()


def test_negative_infinity_logits():
    # every top-k member -inf: the lowest index of the set is returned
    x = np.full(8, -np.inf, np.float32)
    r = oracle.sample_row(x, 1.0, 3, 5, 0, 0, 4, -1, want_probs=True)
    assert r["token"] == 0 and r["margin"] == math.inf
    np.testing.assert_allclose(r["probs"][:3], 1 / 3)
    # -inf members of the set are never drawn while a finite member exists
    x = np.array([-np.inf, 0.0, -np.inf, -np.inf], np.float32)
    for s in range(1, 200):
        assert oracle.sample_row(x, 1.0, 4, 9, 0, 0, s, -1)["token"] == 1


def test_invalid_inputs_are_rejected():
    x = np.zeros(8, np.float32)
    for T, k in [(0.0, 3), (-1.0, 3), (1.0, 0), (1.0, 9)]:
        with pytest.raises(ValueError):
            oracle.sample_row(x, T, k, 0, 0, 0, 4, -1)
    x[3] = np.nan
    with pytest.raises(ValueError):
        oracle.sample_row(x, 1.0, 3, 0, 0, 0, 4, -1)


def _raised(x: np.float32, delta: float, above: bool) -> np.float32:
    """The float32 nearest x + delta whose exact increase over x is at least delta (above) or at most delta."""
    y = np.float32(float(x) + delta)
    step = np.float32(np.inf if above else -np.inf)
    while (float(y) - float(x) < delta) if above else (float(y) - float(x) > delta):
        y = np.nextafter(y, step, dtype=np.float32)
    return y


def _margin_row(rng, V, k, ties):
    x = (rng.normal(size=V) * 3).astype(np.float32)
    if ties:   # entries that share the value of the k-th largest: ties at the top-k boundary
        kth = np.argsort(-x, kind="stable")[k - 1]
        x[rng.choice(V, size=min(V - 1, 6), replace=False)] = x[kth]
    return x


@pytest.mark.parametrize("T", [1.0, 0.5])
@pytest.mark.parametrize("V,k", [(8, 2), (8, 5), (64, 2), (64, 50), (1088, 2), (1088, 50), (1088, 250)])
@pytest.mark.parametrize("ties", [False, True])
def test_gumbel_margin_is_the_gap_to_the_runner_up(V, k, T, ties):
    """The margin m the oracle returns is the gap between the best and the second-best perturbed score.

    Checked through the draw alone: only member i's score moves when its logit is raised (its uniform is
    indexed by vocabulary id, and a member stays a member), and by exactly the raise of x_i = logit_i / T
    (T = 1, or T = 0.5 where the division is exact).  So raising some member by more than m must hand the
    draw to it -- the runner-up -- and raising any member by less than m must leave the draw where it was.
    A margin that is too large fails the second half (the runner-up overtakes early), one that is too small
    the first (nobody overtakes)."""
    rng = np.random.default_rng(V * 1000 + k + (7 if ties else 0) + int(T * 10))
    compared = 0
    for trial in range(3 if V == 1088 else 10):
        x = _margin_row(rng, V, k, ties)
        seed, b, c, step = int(rng.integers(0, 2 ** 63)), trial, trial % 9, 20 + trial
        draw = lambda y: oracle.sample_row(y, T, k, seed, b, c, step, -1)["token"]
        r = oracle.sample_row(x, T, k, seed, b, c, step, -1, want_topk=True)
        t, m = r["token"], r["margin"]
        assert draw(x) == t
        if not (0.0 < m < math.inf):
            continue
        compared += 1
        overtaken = []
        for i in (int(j) for j in r["topk"] if j != t):
            y = x.copy()
            y[i] = _raised(x[i], T * m * (1 + 1e-6), above=True)
            got = draw(y)
            assert got in (t, i), (i, got)            # a raise of i can only hand the draw to i
            if got == i:
                overtaken.append(i)
            y[i] = _raised(x[i], T * m * (1 - 1e-6), above=False)
            assert draw(y) == t, (i, m)               # just short of the margin: no change
        assert overtaken, ("no member overtakes the draw with a raise of the margin", m)
    assert compared >= 2
