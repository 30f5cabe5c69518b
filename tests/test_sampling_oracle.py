"""Pins of the sampling oracle (oracle/k2_sampling.py) against what the
definitions and the mathematics fix, without a GPU.

  * Philox4x32-10: known-answer vectors of the published generator (Salmon et
    al., SC 2011, as distributed with its reference implementation).
  * exp_neg: within a few float32 ulps of exp, exactly 1 at 0, monotone.
  * the order key sorts exactly like the floats.
  * limits that reduce to the greedy argmax: a tiny temperature, top-k = 1,
    min-p = 1, a tiny top-p.
  * top-p: the kept set is the smallest most-probable set reaching top_p
    (brute force over the sorted probabilities).
  * the repetition penalty divides positive and multiplies negative logits of
    seen ids, once per distinct id.
  * the draw: frequencies over many positions follow the kept masses.
"""
import math

import numpy as np
import pytest

from oracle import k2_sampling as S

F32 = np.float32


def test_philox_known_answers():
    assert S.philox4x32_10((0, 0, 0, 0), (0, 0)) == (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)
    assert S.philox4x32_10((0xFFFFFFFF,) * 4, (0xFFFFFFFF, 0xFFFFFFFF)) == (
        0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)
    assert S.philox4x32_10((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0)) == (
        0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)


def test_exp_neg_is_exp_to_a_few_ulps():
    x = np.concatenate([-np.linspace(0, 86.9, 20001, dtype=np.float64), [-1e-7, -0.5, -1.0, -2.0]]).astype(F32)
    got = S.exp_neg(x).astype(np.float64)
    want = np.exp(x.astype(np.float64))
    ulp = np.spacing(want.astype(F32)).astype(np.float64)
    assert np.max(np.abs(got - want) / ulp) <= 4.0
    assert S.exp_neg(np.array([0.0], F32))[0] == 1.0
    assert np.all(np.diff(S.exp_neg(-np.linspace(0, 80, 5001).astype(F32))) <= 0)
    assert S.exp_neg(np.array([-87.5, -200.0, -np.inf], F32)).tolist() == [0.0, 0.0, 0.0]


def test_order_key_sorts_like_the_floats():
    rng = np.random.default_rng(5)
    z = np.concatenate([rng.standard_normal(2000).astype(F32) * F32(50), [0.0, -0.0, -np.inf, np.inf, 1e-38, -1e-38]])
    z = z.astype(F32)
    k = S.order_key(z)
    by_key = z[np.argsort(k, kind="stable")]
    assert np.all(np.diff(by_key.astype(np.float64)) >= 0)


def logits_row(V, seed, scale=2.0):
    return (np.random.default_rng(seed).standard_normal(V) * scale).astype(F32)


@pytest.mark.parametrize("seed", range(6))
def test_limits_that_are_the_greedy_argmax(seed):
    lg = logits_row(4000, seed)
    am = int(np.argmax(lg))
    for pos in range(3):
        assert S.sample_row(lg, 1e-4, seed=seed, position=pos) == am
        assert S.sample_row(lg, 1.0, top_k=1, seed=seed, position=pos) == am
        assert S.sample_row(lg, 1.0, min_p=1.0, seed=seed, position=pos) == am
        assert S.sample_row(lg, 1.0, top_p=1e-6, seed=seed, position=pos) == am


@pytest.mark.parametrize("top_p", [0.05, 0.5, 0.9, 0.99])
def test_top_p_keeps_the_smallest_set_reaching_it(top_p):
    lg = logits_row(3000, 11, scale=3.0)
    keep, mass = S.filter_row(lg, 0.8, top_p=top_p)
    m = mass.astype(np.float64)
    order = np.argsort(-m, kind="stable")
    csum = np.cumsum(m[order])
    n = int(np.searchsorted(csum, top_p * m.sum())) + 1  # the first prefix reaching top_p
    brute = np.zeros(lg.size, bool)
    brute[order[:n]] = True
    assert np.array_equal(keep, brute)
    assert m[keep].sum() >= top_p * m.sum() > m[keep].sum() - m[keep].min()


def test_top_k_and_min_p_sets():
    lg = logits_row(1000, 3)
    keep, _ = S.filter_row(lg, 1.3, top_k=37)
    assert keep.sum() == 37 and lg[keep].min() >= np.sort(lg)[-37]
    keep, mass = S.filter_row(lg, 1.3, min_p=0.05)
    w = np.exp((lg.astype(np.float64) - lg.max()) / 1.3)
    assert np.array_equal(keep, w >= 0.05) or np.sum(keep != (w >= 0.05)) <= 1  # rounding at the edge


def test_repetition_penalty_once_per_distinct_seen_id():
    lg = np.array([2.0, -2.0, 1.0, 0.5], F32)
    keep, m1 = S.filter_row(lg, 1.0, penalty=2.0, seen=[0, 1, 1, 1, 7])
    keep, m0 = S.filter_row(np.array([1.0, -4.0, 1.0, 0.5], F32), 1.0)
    assert np.array_equal(m1, m0)  # 2 -> 1, -2 -> -4, duplicates and ids outside the vocabulary ignored
    assert S.filter_row(lg, 1.0, penalty=1.0, seen=[0, 1])[1].tolist() == S.filter_row(lg, 1.0)[1].tolist()


def test_draw_frequencies_follow_the_masses():
    lg = np.array([0.0, -0.3, -1.0, -2.0, 0.7, -5.0, 0.2, -0.1], F32)
    keep, mass = S.filter_row(lg, 1.0)
    p = mass.astype(np.float64) / mass.sum()
    n = 20000
    counts = np.bincount([S.sample_row(lg, 1.0, seed=99, position=i) for i in range(n)], minlength=8)
    chi2 = float(np.sum((counts - n * p) ** 2 / (n * p)))
    assert chi2 < 30.0  # 7 degrees of freedom: p-value ~ 1e-4 at 30
    # another seed or sequence gives other draws
    a = [S.sample_row(lg, 1.0, seed=1, position=i) for i in range(50)]
    b = [S.sample_row(lg, 1.0, seed=2, position=i) for i in range(50)]
    c = [S.sample_row(lg, 1.0, seed=1, position=i, seq=1) for i in range(50)]
    assert a != b and a != c


def test_the_draw_picks_the_first_index_crossing_the_target():
    # all mass on two tokens of equal weight: u < 1/2 picks the first, else the second
    lg = np.array([-np.inf, 3.0, -np.inf, 3.0], F32)
    for pos in range(64):
        r = S.uniform24(7, pos, 0)
        want = 1 if r < (1 << 23) else 3
        assert S.sample_row(lg, 1.0, seed=7, position=pos) == want
    assert math.isclose(np.mean([S.uniform24(3, i, 0) / 2 ** 24 for i in range(4000)]), 0.5, abs_tol=0.02)
