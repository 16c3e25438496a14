"""Pins of the oracle's segmentation (brute force, invariants, planted spans).

The segmentation rule (SeKV technical summary, Methodik 1 on the German page /
方法论 1 on the Chinese page: high-surprisal tokens are span boundaries and
anchors) is pinned by a *characterisation* checked over every candidate set of
span starts, independently of the oracle's left-to-right walk.
"""
import itertools

import numpy as np
import pytest

import oracle
from synth import gen


def valid_segmentation(H, starts, m0, m1, tau, lmin, lmax):
    """True iff ``starts`` satisfies the rule, checked span by span.

    A start set is valid iff it begins at m0 and for every span [s, e)
    (e = next start, or m1 for the last span): 1 <= e - s <= lmax; no token
    t in [s + lmin, e) has H_t > tau (it would have opened a span); and if e
    is a start then it was opened legally: e - s == lmax or
    (H_e > tau and e - s >= lmin); a last span longer than lmax is illegal.
    """
    if not starts or starts[0] != m0:
        return False
    ends = list(starts[1:]) + [m1]
    for i, (s, e) in enumerate(zip(starts, ends)):
        if e - s < 1 or e - s > lmax:
            return False
        for t in range(s + lmin, e):
            if H[t] > tau and t - s < lmax:
                return False
        if i + 1 < len(starts):
            if not (e - s == lmax or (H[e] > tau and e - s >= lmin)):
                return False
    return True


@pytest.mark.parametrize("lmin,lmax", [(2, 4), (3, 5), (1, 3), (2, 2)])
def test_segment_matches_brute_force(lmin, lmax):
    rng = np.random.default_rng(5)
    n_sink, n_recent, T = 1, 1, 12
    m0, m1 = n_sink, T - n_recent
    tau = 1.0
    for _ in range(60):
        H = np.where(rng.random(T) < 0.4, 2.0, 0.5).astype(np.float32)
        starts, lens = oracle.segment(H, n_sink, n_recent, tau, lmin, lmax)
        sols = []
        mid = list(range(m0 + 1, m1))
        for k in range(len(mid) + 1):
            for comb in itertools.combinations(mid, k):
                cand = [m0] + list(comb)
                if valid_segmentation(H, cand, m0, m1, tau, lmin, lmax):
                    sols.append(cand)
        assert len(sols) == 1, sols
        assert list(starts) == sols[0]
        assert int(lens.sum()) == m1 - m0


def test_segment_invariants_large():
    rng = np.random.default_rng(11)
    T, ns, nr, tau, lmin, lmax = 20000, 4, 64, 4.0, 4, 256
    H = (rng.gamma(2.0, 1.0, T)).astype(np.float32)
    starts, lens = oracle.segment(H, ns, nr, tau, lmin, lmax)
    assert starts[0] == ns and int(lens.sum()) == T - ns - nr
    assert np.all(lens[:-1] >= lmin) and np.all(lens <= lmax)
    for s, n in zip(starts, lens):
        # no body token past the minimum length is above tau
        seg = H[s + lmin:s + n]
        assert not np.any(seg > np.float32(tau))
    for s, n, s2 in zip(starts[:-1], lens[:-1], starts[1:]):
        assert n == lmax or H[s2] > np.float32(tau)


def test_segment_strict_comparison():
    # a token exactly at tau does not open a span
    H = np.zeros(12, np.float32)
    H[6] = np.float32(4.0)
    starts, _ = oracle.segment(H, 1, 1, 4.0, 2, 100)
    assert list(starts) == [1]
    H[6] = np.nextafter(np.float32(4.0), np.float32(10))
    starts, _ = oracle.segment(H, 1, 1, 4.0, 2, 100)
    assert list(starts) == [1, 6]


def test_segment_empty_middle():
    starts, lens = oracle.segment(np.ones(10, np.float32), 5, 5, 0.5, 2, 4)
    assert len(starts) == 0 and len(lens) == 0


@pytest.mark.parametrize("tau,lmax", [(4.0, 256), (5.2, 256), (6.1, 512)])
def test_planted_spans_are_recovered(tau, lmax):
    g = gen._gen(3)
    T, ns, nr = 30000, 4, 128
    lens = gen.span_lengths(g, T - ns - nr, tau, 4, lmax)
    H = gen.planted_surprisal(g, T, ns, nr, lens, tau, 4, lmax)
    starts, got = oracle.segment(H, ns, nr, tau, 4, lmax)
    assert np.array_equal(got, lens)
