"""GPU parity of the multi-query decode step (sekv_decode_step_multi): n_q
query tokens per sequence over the same cache (in blocks of 8 / hpg tokens,
one launch each), each checked against the oracle's own routing and
mixed-resolution attention for that query alone."""
import numpy as np
import pytest
import torch

import oracle
from oracle import layout
import synth
from synth import gen

from cases import SCALE, compare_out, thresholds

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sk():
    from decode_attention_span_gb300 import build
    build.build()
    import decode_attention_span_gb300 as sk
    return sk


@pytest.mark.parametrize("name,over,n_q", [
    ("llama3_8b_32k", dict(ctx=8192), 2),                              # 4 heads x 2 tokens
    ("llama3_8b_32k", dict(ctx=8192, n_q_heads=16, batch=2), 4),       # 2 heads x 4 tokens
    ("qwen2_7b_stress", dict(ctx=8192, batch=2, n_q_heads=8), 4),      # ranks to 64
    ("llama3_8b_32k", dict(ctx=8192, n_q_heads=8), 8),                 # 1 head x 8 tokens
    ("llama3_8b_32k", dict(ctx=8192), 1),                              # = sekv_decode_step
    ("llama3_8b_32k", dict(ctx=8192), 5),                              # blocks of 2, 2, 1 tokens
    ("qwen2_7b_stress", dict(ctx=8192, batch=2, n_q_heads=8), 6),      # blocks of 4, 2
    ("qwen2_7b_stress", dict(ctx=8192, batch=1), 3),                   # 7 heads: one token a block
])
def test_multi_query_matches_oracle_per_query(sk, name, over, n_q):
    w = synth.get_config(name, **over)
    d = gen.decode_cache(w, 0, device="cpu")
    cache = layout.unpack_layer(gen.abi_to_numpy(d), w.n_sink, w.n_recent)
    g = gen._gen(w.seed * 131 + 7)
    q = gen.query(g, w.batch * n_q, w.n_q_heads).reshape(w.batch, n_q, w.n_q_heads, 128)
    W = gen.routing_weights(g, w.n_kv_heads)
    qn, Wn = q.float().numpy(), W.numpy()
    z = []
    for i in range(n_q):
        z += oracle.route_logits(qn[:, i], Wn, cache)
    # thresholds picked over every token's logits (each head expands about
    # the workload's fraction of spans per token; tokens differ)
    theta = thresholds(z, w.n_q_heads, w.expand_frac, w.group)
    E, o_ref, lse_ref = [], [], []
    for i in range(n_q):
        Ei, _ = oracle.route(qn[:, i], Wn, cache, theta)
        oi, li = oracle.decode_attention(qn[:, i], cache, Ei, SCALE)
        E.append(Ei)
        o_ref.append(oi)
        lse_ref.append(li)
    cfg = sk.Config(w.batch, w.n_q_heads, w.n_kv_heads, w.n_sink, w.n_recent, d["max_spans"],
                    w.rank_cap, w.len_min, w.len_max, w.tau)
    gc = sk.LayerCache({k: v.cuda() for k, v in d.items() if isinstance(v, torch.Tensor)})
    ws = sk.Workspace(cfg)
    o, lse, lst, cnt = sk.decode_step_multi(cfg, gc, q.cuda(), W.cuda(),
                                            torch.from_numpy(theta).cuda(), SCALE, ws,
                                            want_list=True)
    torch.cuda.synchronize()
    assert ws.status() == (0, 0)
    # one launch per block of 8 / hpg tokens; each block's list is the union
    # over its own tokens
    hpg = w.n_q_heads // w.n_kv_heads
    tpb = 8 // hpg
    nb = sk.query_blocks(cfg, n_q)
    assert nb == -(-n_q // tpb)
    ng = w.batch * w.n_kv_heads
    cnt = cnt.cpu().numpy().reshape(nb, ng)
    lst = lst.cpu().numpy().reshape(nb, ng, -1)
    differ = 0
    for k in range(nb):
        toks = range(k * tpb, min(n_q, (k + 1) * tpb))
        for b in range(w.batch):
            for c in range(w.n_kv_heads):
                union = sorted(set().union(*[set(int(x) for x in E[i][b][c]) for i in toks]))
                gi = b * w.n_kv_heads + c
                assert list(lst[k, gi, :cnt[k, gi]]) == union, (k, b, c)
    for b in range(w.batch):
        for c in range(w.n_kv_heads):
            sets = [tuple(E[i][b][c]) for i in range(n_q)]
            differ += len(set(sets)) > 1
    if n_q > 1:
        assert differ > 0, "the tokens' expansion sets should differ somewhere"
    o = o.cpu().numpy()
    lse = lse.cpu().numpy()
    for i in range(n_q):
        compare_out(o[:, i], o_ref[i], f"query token {i}")
        assert np.allclose(lse[:, i], lse_ref[i], atol=2e-3), i
