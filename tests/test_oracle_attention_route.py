"""Pins of the oracle's routing and mixed-resolution attention.

Mixed-resolution attention and zoom-in routing: SeKV technical summary,
Methodik 3 (German page) / 方法论 3 (Chinese page).  The attention is pinned
against torch's scaled_dot_product_attention in float64 (a library routine)
in the cases where the method must reduce to exact attention.
"""
import math

import numpy as np
import pytest
import torch
from scipy.special import logsumexp

import oracle
from oracle import LayerCache, SpanFactors

SCALE = 1.0 / math.sqrt(128)


def sdpa(q, K, V):
    """Exact attention of q [Hq][128] over K, V [n][128] via torch (fp64)."""
    qt = torch.tensor(q, dtype=torch.float64)[None, :, None, :]
    Kt = torch.tensor(K, dtype=torch.float64)[None, None].expand(1, qt.shape[1], -1, -1)
    Vt = torch.tensor(V, dtype=torch.float64)[None, None].expand(1, qt.shape[1], -1, -1)
    o = torch.nn.functional.scaled_dot_product_attention(qt, Kt, Vt, scale=SCALE)
    return o[0, :, 0].numpy()


def manual_cache(tokK, tokV, H, n_sink, n_recent, tau, lmin, lmax, *, kind="svd",
                 rank_cap=512):
    """One-sequence, one-KV-head cache built from tokens without bf16 rounding."""
    starts, lens = oracle.segment(H, n_sink, n_recent, tau, lmin, lmax)
    T = tokK.shape[0]
    full = np.concatenate([np.arange(n_sink), starts, np.arange(T - n_recent, T)])
    ks, vs, fac = [], [], []
    for s, n in zip(starts, lens):
        Kb, Vb = tokK[s + 1:s + n], tokV[s + 1:s + n]
        if len(Kb) == 0:
            ks.append(np.zeros(128)); vs.append(np.zeros(128)); fac.append(None)
            continue
        km, vm = oracle.attention_summary(Kb, Vb)
        ks.append(km); vs.append(vm)
        fk = oracle.span_svd(Kb, np.ones(rank_cap), rank_cap)
        fv = oracle.span_svd(Vb, np.ones(rank_cap), rank_cap)
        fac.append(SpanFactors(fk.U, fk.sigma, fk.gate, fk.Vt, fv.U, fv.sigma, fv.gate, fv.Vt))
    return LayerCache(n_sink=n_sink, n_recent=n_recent, body_len=[lens - 1],
                      k_full=[[tokK[full]]], v_full=[[tokV[full]]],
                      s_route=[[np.zeros((len(starts), 64))]], k_sum=[[np.array(ks)]],
                      v_sum=[[np.array(vs)]], factors=[[fac]], anchors=[starts]), starts, lens


def _tokens(rng, T):
    return rng.standard_normal((T, 128)), rng.standard_normal((T, 128))


def test_all_expanded_full_rank_equals_full_attention():
    rng = np.random.default_rng(0)
    T = 600
    K, V = _tokens(rng, T)
    H = rng.gamma(2.0, 1.0, T).astype(np.float32)
    cache, starts, lens = manual_cache(K, V, H, 4, 16, 3.0, 4, 64)
    q = rng.standard_normal((1, 4, 128))
    E = [[np.flatnonzero(lens - 1 > 0)]]
    o, lse = oracle.decode_attention(q, cache, E, SCALE)
    assert np.allclose(o[0], sdpa(q[0], K, V), atol=1e-12, rtol=0)
    o2, lse2 = oracle.full_attention(q, K[None, None], V[None, None], SCALE)
    assert np.allclose(lse[0], lse2[0], atol=1e-10)
    assert np.allclose(lse[0], logsumexp((K @ q[0].T).T * SCALE, axis=1), atol=1e-10)


def test_identical_keys_summary_equals_exact():
    rng = np.random.default_rng(1)
    T = 300
    K, V = _tokens(rng, T)
    H = rng.gamma(2.0, 1.0, T).astype(np.float32)
    starts, lens = oracle.segment(H, 4, 16, 3.0, 4, 64)
    for s, n in zip(starts, lens):       # every span body: identical keys
        K[s + 1:s + n] = rng.standard_normal(128)
    cache, _, _ = manual_cache(K, V, H, 4, 16, 3.0, 4, 64)
    q = rng.standard_normal((1, 4, 128))
    o, _ = oracle.decode_attention(q, cache, [[np.zeros(0, np.int64)]], SCALE)
    assert np.allclose(o[0], sdpa(q[0], K, V), atol=1e-12)
    # mixed: half the spans expanded at full rank
    E = [[np.flatnonzero(lens - 1 > 0)[::2]]]
    o2, _ = oracle.decode_attention(q, cache, E, SCALE)
    assert np.allclose(o2[0], sdpa(q[0], K, V), atol=1e-12)


def test_single_token_bodies_reduce_to_tokens():
    rng = np.random.default_rng(2)
    T = 120
    K, V = _tokens(rng, T)
    H = np.full(T, 5.0, np.float32)     # every token is a boundary once len >= 2
    cache, starts, lens = manual_cache(K, V, H, 2, 8, 3.0, 2, 64)
    assert np.all(lens[:-1] == 2)
    q = rng.standard_normal((1, 3, 128))
    o, _ = oracle.decode_attention(q, cache, [[np.zeros(0, np.int64)]], SCALE)
    assert np.allclose(o[0], sdpa(q[0], K, V), atol=1e-12)


def test_no_spans_is_textbook_attention():
    rng = np.random.default_rng(3)
    T = 40
    K, V = _tokens(rng, T)
    cache, starts, lens = manual_cache(K, V, np.zeros(T, np.float32), 20, 20, 1.0, 2, 4)
    assert len(starts) == 0
    q = rng.standard_normal((1, 2, 128))
    o, lse = oracle.decode_attention(q, cache, [[np.zeros(0, np.int64)]], SCALE)
    assert np.allclose(o[0], sdpa(q[0], K, V), atol=1e-12)


def test_size_correction_is_log_count():
    # one unexpanded span of body b with summary key k and value v acts like b
    # copies of (k, v): weight ratio to a full-res token with the same key is b
    k = np.zeros(128); v1 = np.zeros(128); v1[0] = 1.0; v2 = np.zeros(128); v2[1] = 1.0
    for b in (1, 2, 5, 17):
        cache = LayerCache(n_sink=1, n_recent=0, body_len=[np.array([b])],
                           k_full=[[np.stack([k, k])]], v_full=[[np.stack([v1, v1])]],
                           s_route=[[np.zeros((1, 64))]], k_sum=[[k[None]]],
                           v_sum=[[v2[None]]], factors=[[[None]]])
        o, _ = oracle.decode_attention(np.ones((1, 1, 128)), cache, [[np.zeros(0, np.int64)]], SCALE)
        assert np.isclose(o[0, 0, 1] / o[0, 0, 0], b / 2.0)


def test_span_order_invariance_and_shift():
    rng = np.random.default_rng(4)
    T = 400
    K, V = _tokens(rng, T)
    H = rng.gamma(2.0, 1.0, T).astype(np.float32)
    cache, starts, lens = manual_cache(K, V, H, 4, 16, 3.0, 4, 64)
    q = rng.standard_normal((1, 2, 128))
    E = [[np.flatnonzero(lens - 1 > 0)[1::3]]]
    o, lse = oracle.decode_attention(q, cache, E, SCALE)
    n = len(starts)
    p = rng.permutation(n)
    inv = np.argsort(p)
    ns = 4
    perm_full = np.concatenate([np.arange(ns), ns + p, np.arange(ns + n, ns + n + 16)])
    c2 = LayerCache(n_sink=4, n_recent=16, body_len=[cache.body_len[0][p]],
                    k_full=[[cache.k_full[0][0][perm_full]]], v_full=[[cache.v_full[0][0][perm_full]]],
                    s_route=[[cache.s_route[0][0][p]]], k_sum=[[cache.k_sum[0][0][p]]],
                    v_sum=[[cache.v_sum[0][0][p]]], factors=[[[cache.factors[0][0][i] for i in p]]])
    E2 = [[np.sort(inv[E[0][0]])]]
    o2, lse2 = oracle.decode_attention(q, c2, E2, SCALE)
    assert np.allclose(o, o2, atol=1e-12) and np.allclose(lse, lse2, atol=1e-12)
    # adding a constant to every value shifts the output by that constant
    c3 = LayerCache(n_sink=4, n_recent=16, body_len=cache.body_len, k_full=cache.k_full,
                    v_full=[[cache.v_full[0][0] + 3.0]], s_route=cache.s_route,
                    k_sum=cache.k_sum, v_sum=[[cache.v_sum[0][0] + 3.0]],
                    factors=cache.factors)
    o3, _ = oracle.decode_attention(q, c3, [[np.zeros(0, np.int64)]], SCALE)
    o0, _ = oracle.decode_attention(q, cache, [[np.zeros(0, np.int64)]], SCALE)
    assert np.allclose(o3, o0 + 3.0, atol=1e-12)


# ---------------------------------------------------------------- routing

def _route_cache(s_rows, body):
    n = len(body)
    return LayerCache(n_sink=0, n_recent=0, body_len=[np.asarray(body)],
                      k_full=[[np.zeros((n, 128))] * 2], v_full=[[np.zeros((n, 128))] * 2],
                      s_route=[[np.asarray(s_rows[0]), np.asarray(s_rows[1])]],
                      k_sum=[[None, None]], v_sum=[[None, None]], factors=[[None, None]])


def test_route_hand_worked():
    # W_r picks q[0:64] for KV head 0 and q[64:128] for KV head 1; group 2
    W = np.zeros((2, 64, 128))
    W[0, :, :64] = np.eye(64)
    W[1, :, 64:] = np.eye(64)
    q = np.zeros((1, 4, 128))
    q[0, 0, 0] = 0.6      # head 0 (KV 0): y = e0 * 0.6
    q[0, 1, 1] = 2.0      # head 1 (KV 0): y = e1 * 2
    q[0, 2, 64] = -1.0    # head 2 (KV 1): y = -e0
    q[0, 3, 65] = 0.25    # head 3 (KV 1): y = e1 / 4
    s = np.zeros((3, 64)); s[0, 0] = 1.0; s[1, 1] = 1.0; s[2, 0] = -1.0
    cache = _route_cache([s, s], [3, 3, 3])
    theta = np.array([0.5, 1.9, 0.99, 0.3])
    E, z = oracle.route(q, W, cache, theta)
    assert np.allclose(z[0][0], [0.6, 0, -0.6]) and np.allclose(z[0][2], [-1, 0, 1])
    # KV 0: head 0 expands span 0 (0.6 > 0.5); head 1 expands span 1 (2 > 1.9)
    assert list(E[0][0]) == [0, 1]
    # KV 1: head 2 expands span 2 (1 > 0.99); head 3: 0.25 > 0.3 is false
    assert list(E[0][1]) == [2]
    # the gate is a probability: sigmoid(z) > sigmoid(theta) gives the same sets
    from scipy.special import expit
    for h in range(4):
        assert np.array_equal(expit(z[0][h]) > expit(theta[h]), z[0][h] > theta[h])


def test_route_extremes_and_empty_bodies():
    rng = np.random.default_rng(7)
    s = rng.standard_normal((2, 10, 64))
    cache = _route_cache([s[0], s[1]], [3, 0, 5, 1, 1, 0, 2, 2, 2, 2])
    q = rng.standard_normal((1, 4, 128))
    W = rng.standard_normal((2, 64, 128))
    E, _ = oracle.route(q, W, cache, np.full(4, np.inf))
    assert all(len(e) == 0 for e in E[0])
    E, _ = oracle.route(q, W, cache, np.full(4, -np.inf))
    for e in E[0]:
        assert list(e) == [0, 2, 3, 4, 6, 7, 8, 9]


def test_route_union_over_group():
    rng = np.random.default_rng(8)
    s = rng.standard_normal((2, 50, 64))
    cache = _route_cache([s[0], s[1]], [4] * 50)
    q = rng.standard_normal((1, 4, 128))
    W = rng.standard_normal((2, 64, 128))
    theta = rng.standard_normal(4) * 3
    E, _ = oracle.route(q, W, cache, theta)
    for c in range(2):
        parts = []
        for h in (2 * c, 2 * c + 1):
            th = np.full(4, np.inf); th[h] = theta[h]
            parts.append(set(oracle.route(q, W, cache, th)[0][0][c]))
        assert set(E[0][c]) == parts[0] | parts[1]
