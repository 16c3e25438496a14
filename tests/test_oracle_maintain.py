"""Pins of the oracle's decode-time cache maintenance (oracle/maintain.py).

Two independent checks:

* a hand-worked sequence (tests/golden/maintenance_worked.txt) fixes the
  positions: when a span opens and closes, which rows stay at full
  resolution, and in what order;
* after every appended token (and every flush of the closed spans waiting to
  be built), the maintained cache equals the batch build of the same prefix
  with the recent window taken from the anchor of the first span not yet
  built (``closed_build``), array by array and factor by factor.  The batch side
  walks the whole prefix and builds every span from the raw K/V; the
  maintained side only ever sees one token at a time.
"""
import os

import numpy as np

import oracle
from oracle import maintain

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "maintenance_worked.txt")


def _rand_inputs(rng, B, Hkv, T, rank_cap, n_spans_cap):
    K = oracle.bf16_round(rng.standard_normal((B, Hkv, T, 128)))
    V = oracle.bf16_round(rng.standard_normal((B, Hkv, T, 128)))
    H = rng.gamma(2.0, 1.0, size=(B, T)).astype(np.float32)
    W = rng.standard_normal((Hkv, 64, 128)).astype(np.float32) / np.float32(np.sqrt(128))
    gates = rng.uniform(0.0, 1.0, size=(B, Hkv, 2, n_spans_cap, rank_cap)).astype(np.float32)
    # some spans keep every component, some none
    gates[:, :, :, ::5] = 0.9
    gates[:, :, :, 3::7] = 0.1
    return K, V, H, W, gates


def _same_cache(a, b):
    assert np.array_equal(a.body_len[0], b.body_len[0]), (a.body_len[0], b.body_len[0])
    assert np.array_equal(a.anchors[0], b.anchors[0])
    for c in range(len(a.k_full[0])):
        assert np.array_equal(a.k_full[0][c], b.k_full[0][c])
        assert np.array_equal(a.v_full[0][c], b.v_full[0][c])
        assert np.array_equal(a.s_route[0][c].reshape(-1, 64), b.s_route[0][c].reshape(-1, 64))
        assert np.array_equal(a.k_sum[0][c].reshape(-1, 128), b.k_sum[0][c].reshape(-1, 128))
        assert np.array_equal(a.v_sum[0][c].reshape(-1, 128), b.v_sum[0][c].reshape(-1, 128))
        assert len(a.factors[0][c]) == len(b.factors[0][c])
        for Fa, Fb in zip(a.factors[0][c], b.factors[0][c]):
            assert (Fa is None) == (Fb is None)
            if Fa is None:
                continue
            for f in ("UK", "sK", "gK", "VtK", "UV", "sV", "gV", "VtV"):
                assert np.array_equal(getattr(Fa, f), getattr(Fb, f)), f


def test_worked_positions():
    rows = []
    for line in open(GOLDEN, encoding="utf-8"):
        line = line.split("#")[0].strip()
        if line:
            rows.append(line.split())
    H = np.array([0, 0.5, 3.0, 1.0, 2.5, 0.1, 0.2, 0.3, 0.5, 0.0, 2.0, 2.0001, 0.4, 0.6],
                 np.float32)
    n = len(H)
    # token t's key and value hold t in dimension 0 (exact in bf16), so a row
    # names its token
    K = np.zeros((1, 1, n, 128))
    K[0, 0, :, 0] = np.arange(n)
    K[0, 0, :, 1] = 1.0
    V = K.copy()
    W = np.zeros((1, 64, 128), np.float32)
    W[0, np.arange(64), np.arange(64)] = 1.0
    gates = np.ones((1, 1, 2, 8, 2), np.float32)
    kw = dict(n_sink=1, n_recent=2, tau=2.0, len_min=2, len_max=4, rank_cap=2)
    st = maintain.init_state(K[:, :, :3], V[:, :, :3], H[None, :3], W, gates, **kw)

    def check(rec):
        T, s_open, anchors, body, toks = rec[0], rec[1], rec[2], rec[3], rec[4:]
        assert st.T[0] == int(T)
        assert st.s_open[0] == (None if s_open == "none" else int(s_open))
        want_a = [] if anchors == "-" else [int(x) for x in anchors.split(",")]
        want_b = [] if body == "-" else [int(x) for x in body.split(",")]
        assert list(st.caches[0].anchors[0]) == want_a
        assert list(st.caches[0].body_len[0]) == want_b
        assert list(st.caches[0].k_full[0][0][:, 0].astype(int)) == [int(x) for x in toks]
        assert list(st.caches[0].v_full[0][0][:, 0].astype(int)) == [int(x) for x in toks]
        assert len(st.tail_H[0]) == st.n_tail(0)

    check(rows[0])
    for rec in rows[1:]:
        T = int(rec[0])
        maintain.append_token(st, K[:, :, T - 1], V[:, :, T - 1], H[None, T - 1], W, gates)
        check(rec)


def _run_equal_to_closed_build(seed, B, Hkv, T0, T1, **kw):
    rng = np.random.default_rng(seed)
    K, V, H, W, gates = _rand_inputs(rng, B, Hkv, T1, kw["rank_cap"], 512)
    st = maintain.init_state(K[:, :, :T0], V[:, :, :T0], H[:, :T0], W, gates, **kw)
    closes = 0
    for T in range(T0 + 1, T1 + 1):
        before = [st.caches[b].n_spans(0) for b in range(B)]
        maintain.append_token(st, K[:, :, T - 1], V[:, :, T - 1], H[:, T - 1], W, gates)
        closes += sum(st.caches[b].n_spans(0) - before[b] for b in range(B))
        ref = maintain.closed_build(K[:, :, :T], V[:, :, :T], H[:, :T], W, gates, **kw)
        for b in range(B):
            _same_cache(st.caches[b], ref[b])
            assert st.s_open[b] == maintain.open_anchor(H[b, :T], kw["n_sink"], kw["n_recent"],
                                                        kw["tau"], kw["len_min"], kw["len_max"])
    return closes


def test_maintained_equals_closed_build_every_step():
    # forced boundaries (len_max 7) and surprisal boundaries; spans of one
    # token (empty bodies) occur with len_min 1
    kw = dict(n_sink=2, n_recent=5, tau=2.2, len_min=1, len_max=7, rank_cap=4)
    closes = _run_equal_to_closed_build(11, B=2, Hkv=2, T0=20, T1=80, **kw)
    assert closes >= 15


def test_maintenance_from_an_empty_middle_region():
    kw = dict(n_sink=3, n_recent=6, tau=2.8, len_min=3, len_max=12, rank_cap=3)
    closes = _run_equal_to_closed_build(12, B=1, Hkv=1, T0=9, T1=60, **kw)
    assert closes >= 3


def test_deferred_builds_equal_the_batch_build_with_a_longer_tail():
    """Closed spans wait in the tail until a flush: after every append the
    cache equals the batch build whose full-resolution tail starts at the
    first span not yet built; flushes at irregular intervals build them all."""
    kw = dict(n_sink=2, n_recent=5, tau=2.2, len_min=1, len_max=7, rank_cap=4)
    rng = np.random.default_rng(13)
    B, Hkv, T0, T1 = 2, 2, 20, 90
    K, V, H, W, gates = _rand_inputs(rng, B, Hkv, T1, kw["rank_cap"], 512)
    st = maintain.init_state(K[:, :, :T0], V[:, :, :T0], H[:, :T0], W, gates, **kw)
    flush_at = set(int(x) for x in rng.choice(np.arange(T0 + 1, T1 + 1), 9, replace=False))
    most_pending = 0
    for T in range(T0 + 1, T1 + 1):
        maintain.append_token(st, K[:, :, T - 1], V[:, :, T - 1], H[:, T - 1], build=False)
        most_pending = max(most_pending, max(len(p) for p in st.pending))
        if T in flush_at:
            maintain.flush(st, W, gates)
            assert all(not p for p in st.pending)
        built = [st.caches[b].n_spans(0) for b in range(B)]
        ref = maintain.closed_build(K[:, :, :T], V[:, :, :T], H[:, :T], W, gates, n_built=built, **kw)
        for b in range(B):
            _same_cache(st.caches[b], ref[b])
    assert most_pending >= 3
