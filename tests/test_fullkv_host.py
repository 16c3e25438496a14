"""Host-side checks of the full-KV comparator configuration.

The comparator runs the decode step over a cache with no spans and every
context token a full-resolution row.  The mixed-resolution attention of the
SeKV technical summary (Methodik 3, German page / 方法论 3, Chinese page) then
has only full-resolution entries; these tests pin that this configuration is
textbook softmax attention on the oracle side, and check the seeded
generator that builds it.
"""
import numpy as np
import torch
from scipy.special import logsumexp

import oracle
import synth
from synth import gen

SCALE = 1.0 / np.sqrt(128.0)


def _no_span_cache(K, V):
    """oracle.LayerCache of one sequence whose tokens are all recent rows."""
    Hkv, T, _ = K.shape
    empty = lambda n: np.zeros((0, n))
    return oracle.LayerCache(
        n_sink=0, n_recent=T, body_len=[np.zeros(0, np.int64)],
        k_full=[[K[c] for c in range(Hkv)]], v_full=[[V[c] for c in range(Hkv)]],
        s_route=[[empty(64) for _ in range(Hkv)]], k_sum=[[empty(128) for _ in range(Hkv)]],
        v_sum=[[empty(128) for _ in range(Hkv)]], factors=[[[] for _ in range(Hkv)]])


def test_no_span_decode_is_textbook_attention():
    rng = np.random.default_rng(11)
    Hkv, G, T = 2, 3, 257
    K = rng.standard_normal((Hkv, T, 128))
    V = rng.standard_normal((Hkv, T, 128))
    q = rng.standard_normal((1, Hkv * G, 128))
    cache = _no_span_cache(K, V)
    o, lse = oracle.decode_attention(q, cache, [[np.zeros(0, np.int64)] * Hkv], SCALE)
    o2, lse2 = oracle.full_attention(q, K[None], V[None], SCALE)
    for h in range(Hkv * G):
        c = h // G
        logits = K[c] @ q[0, h] * SCALE
        p = np.exp(logits - logsumexp(logits))
        assert np.allclose(o[0, h], p @ V[c], atol=1e-12, rtol=0)
        assert abs(lse[0, h] - logsumexp(logits)) < 1e-10
    assert np.allclose(o, o2, atol=1e-12, rtol=0)
    assert np.allclose(lse, lse2, atol=1e-12, rtol=0)


def test_full_kv_cache_layout_and_seed():
    w = synth.get_config("llama3_8b_32k", batch=2)
    T = 300
    d = gen.full_kv_cache(w, 1, T)
    B, Hkv, ms = w.batch, w.n_kv_heads, d["max_spans"]
    assert d["k_full"].shape == (B, Hkv, ms + T, 128) and d["k_full"].dtype == torch.bfloat16
    assert d["v_full"].shape == d["k_full"].shape
    # rows past the T tokens are zero, the tokens themselves are not
    assert torch.count_nonzero(d["k_full"][:, :, T:]) == 0
    assert torch.count_nonzero(d["v_full"][:, :, T:]) == 0
    assert bool((d["k_full"][:, :, :T].float().abs().sum(-1) > 0).all())
    assert int(d["n_spans"].abs().sum()) == 0 and int(d["body_len"].abs().sum()) == 0
    assert d["s_route"].shape == (B, Hkv, ms, 64) and d["rec_off"].dtype == torch.int64
    assert ms % 64 == 0
    # seeded: the same layer twice is identical, another layer differs
    d2 = gen.full_kv_cache(w, 1, T)
    assert torch.equal(d["k_full"], d2["k_full"]) and torch.equal(d["v_full"], d2["v_full"])
    d3 = gen.full_kv_cache(w, 2, T)
    assert not torch.equal(d["k_full"], d3["k_full"])
    # unit-variance rows, as the full-resolution rows of the span cache
    x = d["k_full"][:, :, :T].float()
    assert abs(float(x.mean())) < 0.02 and abs(float(x.std()) - 1.0) < 0.02
