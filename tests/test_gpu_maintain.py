"""GPU parity of decode-time cache maintenance (sekv_maint_init,
sekv_append_token, sekv_maint_flush) against the oracle's reading
(oracle/maintain.py): after the appends and flushes, the maintained cache
equals the batch build of the same prefix with the recent window taken from
the anchor of each sequence's first span not yet built; and a decode step
over the maintained cache equals the oracle's decode over that build."""
import numpy as np
import pytest
import torch

import oracle
from oracle import layout, maintain
import synth
from synth import gen

from test_gpu_build import TOL_RECON, TOL_S_ROUTE, TOL_SIGMA, ulp_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sk():
    from decode_attention_span_gb300 import build
    build.build()
    import decode_attention_span_gb300 as sk
    return sk


def merged(caches):
    """One LayerCache over the batch from per-sequence batch-1 caches."""
    out = oracle.LayerCache(n_sink=caches[0].n_sink, n_recent=caches[0].n_recent, body_len=[],
                            k_full=[], v_full=[], s_route=[], k_sum=[], v_sum=[], factors=[])
    for c in caches:
        for f in ("body_len", "k_full", "v_full", "s_route", "k_sum", "v_sum", "factors"):
            getattr(out, f).append(getattr(c, f)[0])
    return out


def compare(got, ref, Hkv):
    worst = dict(s=0.0, ulps=0.0, sigma=0.0, recon=0.0, spans=0)
    for b in range(len(ref.body_len)):
        assert np.array_equal(got.body_len[b], ref.body_len[b]), f"spans of sequence {b}"
        for c in range(Hkv):
            assert np.array_equal(got.k_full[b][c], ref.k_full[b][c]), (b, c)
            assert np.array_equal(got.v_full[b][c], ref.v_full[b][c]), (b, c)
            ns = len(ref.body_len[b])
            sr = np.asarray(ref.s_route[b][c]).reshape(-1, 64)[:ns]
            worst["s"] = max(worst["s"], float(np.abs(got.s_route[b][c] - sr).max(initial=0)))
            for X, Y in ((got.k_sum[b][c], ref.k_sum[b][c]), (got.v_sum[b][c], ref.v_sum[b][c])):
                Y = np.asarray(Y).reshape(-1, 128)[:ns]
                worst["ulps"] = max(worst["ulps"], float((np.abs(X - Y) / ulp_bf16(Y)).max(initial=0)))
            for Fg, Fr in zip(got.factors[b][c], ref.factors[b][c]):
                assert (Fg is None) == (Fr is None)
                if Fr is None:
                    continue
                worst["spans"] += 1
                for side in ("K", "V"):
                    sg, sr_ = getattr(Fg, "s" + side), getattr(Fr, "s" + side)
                    assert sg.shape == sr_.shape, "ranks differ"
                    if len(sr_) == 0:
                        continue
                    worst["sigma"] = max(worst["sigma"], float(np.max(np.abs(sg - sr_) / sr_)))
                    Rg = oracle.reconstruct(getattr(Fg, "U" + side), sg, getattr(Fg, "g" + side),
                                            getattr(Fg, "Vt" + side))
                    Rr = oracle.reconstruct(getattr(Fr, "U" + side), sr_, getattr(Fr, "g" + side),
                                            getattr(Fr, "Vt" + side))
                    worst["recon"] = max(worst["recon"],
                                         float(np.linalg.norm(Rg - Rr) / np.linalg.norm(Rr)))
    assert worst["s"] <= TOL_S_ROUTE, worst
    assert worst["ulps"] <= 1.0, worst
    assert worst["sigma"] <= TOL_SIGMA, worst
    assert worst["recon"] <= TOL_RECON, worst
    return worst


@pytest.mark.parametrize("over,T0,n_app,every", [
    # 2 sequences, 2 KV heads; bodies up to 63 tokens, ranks up to 32; every
    # closed span built at once
    (dict(ctx=2600, n_kv_heads=2, n_q_heads=8, batch=2, len_max=64), 2200, 400, 1),
    # the same with builds batched: a flush every 37 appends, the last
    # appends left waiting (the decode reads them at full resolution)
    (dict(ctx=2600, n_kv_heads=2, n_q_heads=8, batch=2, len_max=64), 2200, 400, 37),
    # len_min 1 (one-token spans: empty bodies), bodies past 128 tokens (the
    # 128 x 128 side of the SVD), forced boundaries at len_max 160
    (dict(ctx=1800, n_kv_heads=1, n_q_heads=4, batch=1, tau=6.1, len_min=1, len_max=160), 1000,
     800, 5),
])
def test_append_matches_closed_build_and_decodes(sk, over, T0, n_app, every):
    w = synth.get_config("mistral_7b_build_128k", layers=1, **over)
    T1 = T0 + n_app
    assert T1 == w.ctx
    n_sp = max(len(gen.sequence_spans(w, b)) for b in range(w.batch))
    ms = (n_sp + w.len_max + 63) // 64 * 64
    inp = gen.build_inputs(w, 0, max_spans=ms)
    K, V = inp["K"].cuda(), inp["V"].cuda()
    H = torch.from_numpy(inp["H"]).cuda()
    W = inp["W_r"].cuda()
    gates = torch.from_numpy(inp["gates"]).cuda()
    cfg = sk.Config(w.batch, w.n_q_heads, w.n_kv_heads, w.n_sink, w.n_recent, ms, w.rank_cap,
                    w.len_min, w.len_max, w.tau)
    ws = sk.Workspace(cfg, which=sk.sekv.SEKV_CALL_BUILD, ctx_len=T1)
    out = sk.alloc_cache(cfg, 256 << 20)
    K0, V0 = K[:, :, :T0].contiguous(), V[:, :, :T0].contiguous()
    H0 = H[:, :T0].contiguous()
    sk.build_spans(cfg, K0, V0, H0, W, gates, out, ws)
    mt = sk.Maintainer(cfg, out, K0, V0, H0, T0, ws)
    n0 = out["n_spans"].clone()
    for i, t in enumerate(range(T0, T1)):
        mt.append(K[:, :, t].contiguous(), V[:, :, t].contiguous(), H[:, t].contiguous())
        if (i + 1) % every == 0:
            mt.flush(W, gates)
    torch.cuda.synchronize()
    assert ws.status() == (0, 0)
    assert int((out["n_spans"] - n0).min()) >= 5  # several spans built per sequence
    built = [int(x) for x in out["n_spans"].cpu()]

    kw = dict(n_sink=w.n_sink, n_recent=w.n_recent, tau=w.tau, len_min=w.len_min,
              len_max=w.len_max, rank_cap=w.rank_cap)
    Kn, Vn = inp["K"].float().numpy(), inp["V"].float().numpy()
    ref = merged(maintain.closed_build(Kn, Vn, inp["H"], inp["W_r"].numpy(), inp["gates"],
                                       n_built=built, **kw))
    arrs = gen.abi_to_numpy({**out, "n_tail": mt.n_tail})
    got = layout.unpack_layer(arrs, w.n_sink, w.n_recent)
    print(compare(got, ref, w.n_kv_heads))

    # decode over the maintained cache (n_tail rows after the anchors)
    from cases import SCALE, compare_out, thresholds
    q = inp["q"]
    z = oracle.route_logits(q.float().numpy(), inp["W_r"].numpy(), ref)
    theta = thresholds(z, w.n_q_heads, w.expand_frac, w.group)
    E, _ = oracle.route(q.float().numpy(), inp["W_r"].numpy(), ref, theta)
    o_ref, _ = oracle.decode_attention(q.float().numpy(), ref, E, SCALE)
    wsd = sk.Workspace(cfg)
    o, lse, lst, cnt = sk.decode_step(cfg, mt.layer_cache(), q.cuda(), W,
                                      torch.from_numpy(theta).cuda(), SCALE, wsd, want_list=True)
    torch.cuda.synchronize()
    assert wsd.status() == (0, 0)
    cnt = cnt.cpu().numpy()
    lst = lst.cpu().numpy().reshape(w.batch * w.n_kv_heads, -1)
    for b in range(w.batch):
        for c in range(w.n_kv_heads):
            g = b * w.n_kv_heads + c
            assert np.array_equal(lst[g, :cnt[g]], E[b][c])
    compare_out(o.cpu().numpy(), o_ref, "maintained cache")
