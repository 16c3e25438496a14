"""GPU parity of the decode step over a full-KV cache against textbook
softmax attention.

The pages report SeKV as often faster than full-KV attention (SeKV technical
summary, Ergebnisse (German page) / 实验 (Chinese page)).  The comparator is
the same decode step over a cache with no spans and every context token a
full-resolution row (n_sink = 0, n_recent = T).  The mixed-resolution
attention of Methodik 3 / 方法论 3 then has only full-resolution entries, so
its result is plain softmax attention over all T tokens:
``oracle.full_attention``.  Tolerances as for the decode step (max-abs 1e-2,
relative-L2 5e-3; lse within 1e-3).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from synth import gen

from cases import SCALE, compare_out

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sk():
    from decode_attention_span_gb300 import build
    build.build()
    import decode_attention_span_gb300 as sk
    return sk


def run_fullkv(sk, w, T):
    """One decode step of layer 0 over a T-token full-KV cache; returns the
    GPU's (o, lse) and the numpy K, V, q it was given."""
    d = gen.full_kv_cache(w, 0, T, device="cuda")
    cfg = sk.Config(w.batch, w.n_q_heads, w.n_kv_heads, 0, T, d["max_spans"], w.rank_cap,
                    w.len_min, w.len_max, w.tau)
    cache = sk.LayerCache({k: v for k, v in d.items() if isinstance(v, torch.Tensor)})
    g = gen._gen(w.seed * 7919 + 3, "cuda")
    q = gen.query(g, w.batch, w.n_q_heads, "cuda")
    W = gen.routing_weights(g, w.n_kv_heads, "cuda").contiguous()
    theta = torch.zeros(w.n_q_heads, device="cuda")
    ws = sk.Workspace(cfg)
    out, lse, _, _ = sk.decode_step(cfg, cache, q, W, theta, SCALE, ws)
    torch.cuda.synchronize()
    assert ws.status() == (0, 0)
    K = d["k_full"][:, :, :T].float().cpu().numpy()
    V = d["v_full"][:, :, :T].float().cpu().numpy()
    return out.cpu().numpy(), lse.cpu().numpy(), K, V, q.float().cpu().numpy()


@pytest.mark.parametrize("name,T,batch", [
    ("llama3_8b_32k", 4096 + 37, 1),   # ragged over 32-row pages and over CTAs
    ("qwen2_7b_stress", 2000, 2),      # group of 7, two sequences
    ("llama3_8b_32k", 1, 1),           # one token: o = v_0 exactly
])
def test_fullkv_decode_matches_full_attention(sk, name, T, batch):
    w = synth.get_config(name, batch=batch)
    o, lse, K, V, q = run_fullkv(sk, w, T)
    o_ref, lse_ref = oracle.full_attention(q, K, V, SCALE)
    compare_out(o, o_ref, f"full-KV {name} T={T}")
    assert np.allclose(lse, lse_ref, atol=1e-3)


def test_fullkv_decode_128k(sk):
    """The comparator's benchmark size (128K tokens, Llama-3-8B heads), every
    head checked one KV head at a time."""
    w = synth.get_config("llama3_8b_128k")
    T = 131072
    o, lse, K, V, q = run_fullkv(sk, w, T)
    G = w.n_q_heads // w.n_kv_heads
    for c in range(w.n_kv_heads):
        hs = slice(c * G, (c + 1) * G)
        o_ref, lse_ref = oracle.full_attention(q[:, hs], K[:, c:c + 1], V[:, c:c + 1], SCALE)
        compare_out(o[:, hs], o_ref, f"full-KV 128K KV head {c}")
        assert np.allclose(lse[:, hs], lse_ref, atol=1e-3)
