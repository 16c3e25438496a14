"""Pins of the oracle's span SVD and summaries against closed forms.

Span representations: SeKV technical summary, Methodik 2 (German page) /
方法论 2 (Chinese page): a normalised surprisal-weighted routing summary of
projected keys, and a gated low-rank SVD basis per span.
"""
import numpy as np
import pytest

import oracle


def _M(rng, b, rank=None):
    if rank is None:
        return rng.standard_normal((b, 128))
    return rng.standard_normal((b, rank)) @ rng.standard_normal((rank, 128)) / np.sqrt(rank)


@pytest.mark.parametrize("b", [1, 2, 7, 31, 128, 200])
def test_singular_values_match_gram_eigenvalues(b):
    rng = np.random.default_rng(b)
    M = _M(rng, b)
    res = oracle.span_svd(M, np.ones(128), 128)
    # independent routine: eigenvalues of the Gram matrix on the small side
    Gm = M @ M.T if b <= 128 else M.T @ M
    ev = np.sort(np.linalg.eigvalsh(Gm))[::-1][:min(b, 128)]
    assert np.allclose(res.sigma_all ** 2, np.clip(ev, 0, None), rtol=1e-9, atol=1e-9)
    # Frobenius identity
    assert np.isclose(np.sum(res.sigma_all ** 2), np.sum(M * M), rtol=1e-12)


@pytest.mark.parametrize("b,cap", [(5, 16), (31, 16), (40, 32), (100, 64)])
def test_eckart_young_with_gates(b, cap):
    rng = np.random.default_rng(100 + b)
    M = _M(rng, b)
    R = min(cap, b)
    rho = R // 2 + 1
    g = 1.0 / (1.0 + np.exp(-2.0 * (rho - np.arange(R) - 0.5)))
    res = oracle.span_svd(M, g, cap)
    assert res.rank == min(rho, R)
    err2 = np.sum((M - oracle.reconstruct(res.U, res.sigma, res.gate, res.Vt)) ** 2)
    s = res.sigma_all
    r = res.rank
    expect = np.sum(((1 - g[:r]) * s[:r]) ** 2) + np.sum(s[r:] ** 2)
    assert np.isclose(err2, expect, rtol=1e-9)
    # with unit gates the error is the sum of the discarded sigma^2 and no
    # rank-r matrix does better (random rank-r competitors)
    res1 = oracle.span_svd(M, np.ones(cap), cap)
    best = np.sum((M - oracle.reconstruct(res1.U, res1.sigma, res1.gate, res1.Vt)) ** 2)
    assert np.isclose(best, np.sum(s[R:] ** 2), rtol=1e-9, atol=1e-9)
    for _ in range(5):
        A = rng.standard_normal((b, R))
        Bm = np.linalg.lstsq(A, M, rcond=None)[0]
        assert np.sum((M - A @ Bm) ** 2) >= best - 1e-9


def test_full_rank_reconstructs_exactly_and_orthonormal():
    rng = np.random.default_rng(3)
    M = _M(rng, 20)
    res = oracle.span_svd(M, np.ones(20), 64)
    assert res.rank == 20
    assert np.allclose(oracle.reconstruct(res.U, res.sigma, res.gate, res.Vt), M, atol=1e-12)
    assert np.allclose(res.U.T @ res.U, np.eye(20), atol=1e-12)
    assert np.allclose(res.Vt @ res.Vt.T, np.eye(20), atol=1e-12)


def test_rank_is_longest_prefix_above_half():
    rng = np.random.default_rng(4)
    M = _M(rng, 10)
    assert oracle.span_svd(M, [0.9, 0.8, 0.4, 0.9, 0.9], 5).rank == 2
    assert oracle.span_svd(M, [0.5, 0.9], 5).rank == 0
    assert oracle.span_svd(M, np.full(16, 0.51), 16).rank == 10  # capped by b


def test_sign_canonical():
    rng = np.random.default_rng(6)
    M = _M(rng, 12)
    res = oracle.span_svd(M, np.ones(12), 12)
    for j in range(res.rank):
        row = res.Vt[j]
        assert row[int(np.argmax(np.abs(row)))] > 0
    # flipping M's sign flips U but keeps Vt canonical
    res2 = oracle.span_svd(-M, np.ones(12), 12)
    assert np.allclose(res2.Vt, res.Vt, atol=1e-10)
    assert np.allclose(res2.U, -res.U, atol=1e-10)


def test_low_rank_block_is_captured():
    rng = np.random.default_rng(8)
    M = _M(rng, 30, rank=8)
    res = oracle.span_svd(M, np.ones(16), 16)
    assert np.all(res.sigma_all[8:] < 1e-10)
    assert np.allclose(oracle.reconstruct(res.U[:, :8], res.sigma[:8], res.gate[:8], res.Vt[:8]),
                       M, atol=1e-10)


def test_routing_summary_single_token_and_invariances():
    rng = np.random.default_rng(9)
    W = rng.standard_normal((64, 128)) / np.sqrt(128)
    k = rng.standard_normal((1, 128))
    s = oracle.routing_summary(k, [2.5], W)
    u = W @ k[0]
    assert np.allclose(s, u / np.linalg.norm(u), atol=1e-14)
    K = rng.standard_normal((9, 128))
    H = rng.gamma(2.0, 1.0, 9)
    s1 = oracle.routing_summary(K, H, W)
    assert np.isclose(np.linalg.norm(s1), 1.0)
    assert np.allclose(oracle.routing_summary(K, 3.7 * H, W), s1, atol=1e-13)
    p = rng.permutation(9)
    assert np.allclose(oracle.routing_summary(K[p], H[p], W), s1, atol=1e-13)
    # hand-worked 2-token case in a 2-d toy routing space embedded in W
    W2 = np.zeros((64, 128)); W2[0, 0] = 1.0; W2[1, 1] = 1.0
    K2 = np.zeros((2, 128)); K2[0, 0] = 1.0; K2[1, 1] = 1.0
    s2 = oracle.routing_summary(K2, [3.0, 4.0], W2)
    assert np.allclose(s2[:2], [0.6, 0.8]) and np.allclose(s2[2:], 0)
    assert oracle.routing_summary(np.zeros((0, 128)), [], W) is None


def test_attention_summary_means_and_bf16():
    K = np.array([[1.0] * 128, [2.0] * 128, [4.0] * 128])
    km, vm = oracle.attention_summary(K, -K)
    assert np.allclose(km, 7.0 / 3.0) and np.allclose(vm, -7.0 / 3.0)
    # 7/3 = 2.333... ; bf16 has 8 significant bits: 2.333 -> 2.328125 (0x4015)
    assert oracle.bf16_round(np.float64(7.0 / 3.0)) == 2.328125
    # ties to even: 1 + 2^-8 is halfway between 1 and 1 + 2^-7 -> 1
    assert oracle.bf16_round(np.float64(1.0 + 2 ** -8)) == 1.0
    assert oracle.bf16_round(np.float64(1.0 + 3 * 2 ** -8)) == 1.0 + 2 ** -6
