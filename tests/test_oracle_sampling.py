"""Pins of the sampling oracle against facts outside it: the generator against
a second implementation of splitmix64's published definition, the penalties
and kept sets in closed form, the greedy rules of "Metal LLM decode" (the
sampled arm: temperature <= 0 falls back to greedy, top_k = 1 reproduces the
greedy tokens), the inverse-CDF draw on a two-token distribution, and the
draw frequencies against the kept probabilities (chi-square)."""
import numpy as np
import pytest

import synth
from oracle import sampling as S


def test_generator_matches_the_input_generator_implementation():
    # synth's C tqs_draw(s, k) is mix64(s + (k + 1) * golden), written separately
    L = synth.lib()
    for seed in (0, 1, 7, 0xDEADBEEF, (1 << 64) - 1, 0x9E3779B97F4A7C15):
        for k in (0, 1, 2, 511, 4095, 1 << 20, (1 << 40) + 3):
            assert S.draw(seed, k) == L.tqs_draw(seed, k)


def test_uniform24_is_exact_in_f32_and_in_range():
    for pos in range(2000):
        u = S.uniform24(123, pos)
        assert 0.0 <= u < 1.0
        assert float(np.float32(u)) == u
        assert u * 2 ** 24 == int(u * 2 ** 24)


def test_penalties_closed_form():
    logits = np.array([2.0, -2.0, 1.0, 0.5], dtype=np.float32)
    got = S.penalised(logits, [0, 1, 2, 2, 2], repeat=2.0, presence=0.5, frequency=0.25)
    # t0 (once): 2/2 - 0.5 - 0.25; t1 (once): -2*2 - 0.5 - 0.25; t2 (3x): 1/2 - 0.5 - 0.75; t3 untouched
    assert got.tolist() == [0.25, -4.75, -0.75, 0.5]
    assert S.penalised(logits, [3, 3], 1.0, 0.0, 0.0).tolist() == logits.tolist()


def test_temperature_zero_is_greedy_on_the_raw_logits():
    rng = np.random.default_rng(0)
    for _ in range(50):
        l = rng.normal(size=300).astype(np.float32)
        hist = rng.integers(0, 300, size=20)
        assert S.sample(l, hist, 5, 0.0, top_k=3, repeat=3.0, presence=1.0, seed=9)[0] == int(np.argmax(l))
        assert S.sample(l, hist, 5, -1.0)[0] == int(np.argmax(l))


def test_top_k_one_is_greedy_including_ties_and_nan():
    rng = np.random.default_rng(1)
    for i in range(200):
        l = rng.normal(size=257).astype(np.float32)
        if i % 3 == 0:  # a planted tie for the maximum: the lower index wins
            a, b = sorted(rng.choice(257, 2, replace=False))
            l[a] = l[b] = np.float32(9.0)
        if i % 5 == 0:
            l[rng.integers(0, 257)] = np.nan
        want = S.greedy(l)
        for T in (0.3, 1.0, 2.5):
            assert S.sample(l, [], i, T, top_k=1, seed=i)[0] == want


PROBS = np.array([0.1, 0.5, 0.15, 0.25])


def kept_set(**kw):
    _, keep, _ = S.kept(np.log(PROBS).astype(np.float32), [], kw.pop("T", 1.0), **kw)
    return set(np.nonzero(keep)[0].tolist())


def test_kept_sets_closed_form():
    # descending probability order: 1 (0.5), 3 (0.25), 2 (0.15), 0 (0.1)
    assert kept_set() == {0, 1, 2, 3}
    assert kept_set(top_k=2) == {1, 3}
    assert kept_set(top_k=3) == {1, 2, 3}
    assert kept_set(top_p=0.4) == {1}                # 0.5 >= 0.4
    assert kept_set(top_p=0.6) == {1, 3}             # 0.5 < 0.6 <= 0.75
    assert kept_set(top_p=0.8) == {1, 2, 3}          # 0.75 < 0.8 <= 0.9
    assert kept_set(top_k=3, top_p=0.8) == {1, 3}    # mass of the top 3 is 0.9: 0.75 >= 0.72
    assert kept_set(min_p=0.25) == {1, 2, 3}         # p >= 0.125
    assert kept_set(min_p=0.4) == {1, 3}             # p >= 0.2
    assert kept_set(min_p=0.6) == {1}
    assert kept_set(T=0.5, top_p=0.8) == {1, 3}      # p^2 normalised: 0.725, then 0.906


def test_temperature_scales_log_probabilities():
    w, _, _ = S.kept(np.log(PROBS).astype(np.float32), [], 0.5)
    assert w[3] / w[1] == pytest.approx((0.25 / 0.5) ** 2, rel=1e-6)
    w, _, _ = S.kept(np.log(PROBS).astype(np.float32), [], 4.0)
    assert w[0] / w[1] == pytest.approx((0.1 / 0.5) ** 0.25, rel=1e-6)


def test_draw_is_the_inverse_cdf_in_index_order():
    # p = (0.25, 0.75): token 0 exactly when u < 0.25
    l = np.log(np.array([0.25, 0.75])).astype(np.float32)
    seen = 0
    for pos in range(3000):
        u = S.uniform24(11, pos)
        if abs(u - 0.25) < 1e-6:
            continue
        assert S.sample(l, [], pos, 1.0, seed=11)[0] == (0 if u < 0.25 else 1)
        seen += 1
    assert seen > 2900


@pytest.mark.parametrize("kw, support", [({}, [0, 1, 2, 3]), ({"top_k": 2}, [1, 3]),
                                         ({"T": 0.5}, [0, 1, 2, 3]), ({"min_p": 0.25}, [1, 2, 3])])
def test_draw_frequencies_follow_the_kept_probabilities(kw, support):
    kw = dict(kw)
    T = kw.pop("T", 1.0)
    p = PROBS ** (1.0 / T)
    p = np.array([p[i] if i in support else 0.0 for i in range(4)])
    p /= p.sum()
    n = 20000
    l = np.log(PROBS).astype(np.float32)
    counts = np.bincount([S.sample(l, [], pos, T, seed=3, **kw)[0] for pos in range(n)], minlength=4)
    assert all(counts[i] == 0 for i in range(4) if i not in support)
    exp = n * p[support]
    chi2 = float(((counts[support] - exp) ** 2 / exp).sum())
    assert chi2 < 18.5  # p < 0.0005 at 3 degrees of freedom


def test_nan_logits_are_never_drawn():
    l = np.log(PROBS).astype(np.float32)
    l[3] = np.nan
    assert all(S.sample(l, [], pos, 1.0, seed=5)[0] != 3 for pos in range(2000))


def test_boundaries_inside_ties_follow_the_index_order():
    # p = (0.2, 0.4, 0.2, 0.2): token 1 first, then the tied 0, 2, 3 in index order
    l = np.log(np.array([0.2, 0.4, 0.2, 0.2])).astype(np.float32)
    assert l[0] == l[2] == l[3]

    def ks(**kw):
        return set(np.nonzero(S.kept(l, [], 1.0, **kw)[1])[0].tolist())

    assert ks(top_k=2) == {1, 0}
    assert ks(top_k=3) == {1, 0, 2}
    assert ks(top_p=0.5) == {1, 0}        # 0.4 < 0.5 <= 0.6
    assert ks(top_p=0.7) == {1, 0, 2}     # 0.6 < 0.7 <= 0.8
    assert ks(top_k=3, top_p=0.9) == {1, 0, 2}


def colliding_pair(T):
    """Adjacent f32 values lo < hi (searched upward from 7) with
    f32(lo / T) == f32(hi / T)."""
    t = np.float32(T)
    lo = np.float32(7.0)
    for _ in range(1000):
        hi = np.nextafter(lo, np.float32(np.inf))
        if np.float32(lo / t) == np.float32(hi / t):
            return lo, hi
        lo = hi
    raise AssertionError("no colliding pair")


def test_top_k_one_is_greedy_where_the_temperature_merges_two_logits():
    # l_hi > l_lo but l_hi / T == l_lo / T in f32; the lower index holds l_lo,
    # so ranking on z with ties to the lower index would keep the wrong token
    T = 3.0
    lo, hi = colliding_pair(T)
    rng = np.random.default_rng(4)
    for i in range(50):
        l = rng.normal(size=300).astype(np.float32)
        a, b = sorted(rng.choice(300, 2, replace=False))
        l[a], l[b] = lo, hi
        assert S.greedy(l) == b
        assert S.sample(l, [], i, T, top_k=1, seed=i)[0] == b
        _, keep, _ = S.kept(l, [], T, top_k=2)
        assert set(np.nonzero(keep)[0].tolist()) == {a, b}
        _, keep, _ = S.kept(l, [], T, top_k=1, top_p=0.3, min_p=0.5)
        assert np.nonzero(keep)[0].tolist() == [b]


def test_the_order_applies_after_the_penalties():
    # the penalty moves token 2 below token 0; top_k = 1 is then the greedy
    # token of the penalised logits
    l = np.array([1.0, 0.5, 1.5], dtype=np.float32)
    assert S.sample(l, [2], 0, 1.0, top_k=1, repeat=2.0)[0] == 0
    assert S.sample(l, [2], 0, 1.0, top_k=1)[0] == 2


def test_an_overflowing_temperature_is_the_greedy_limit():
    # l_max / T beyond f32: every draw is the greedy token of the penalised logits
    rng = np.random.default_rng(6)
    for i in range(20):
        l = rng.normal(size=100).astype(np.float32) * 4
        hist = rng.integers(0, 100, size=5)
        want = S.greedy(S.penalised(l, hist, 1.3, 0.2, 0.0))
        for T in (1e-38, 1e-40):
            assert np.isinf(np.float32(np.max(np.abs(l)) / np.float32(T)))
            assert S.sample(l, hist, i, T, top_p=0.9, repeat=1.3, presence=0.2, seed=i)[0] == want


def test_an_overflowing_temperature_on_negative_logits_is_the_greedy_limit():
    l = np.array([-3.0, -1.0, -2.0, -1.0], dtype=np.float32)
    assert S.sample(l, [], 0, 1e-39, seed=1)[0] == 1
    assert S.sample(l, [], 0, 1e-39, top_k=2, seed=1)[0] == 1
