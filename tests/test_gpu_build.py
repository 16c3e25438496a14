"""GPU parity of the prefill cache build vs the oracle.

Segmentation and anchors (SeKV technical summary, Methodik 1 / 方法论 1) must
be bit-exact; summaries and the gated span SVD (Methodik 2 / 方法论 2) within
the tolerances below: the GPU accumulates in fp32 and rounds stored values
to bf16 like the oracle, so summary keys/values may differ by one bf16 ulp
(the fp32 and fp64 means can straddle a rounding boundary).
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import layout
import synth
from synth import gen

pytestmark = pytest.mark.gpu

TOL_S_ROUTE = 1e-5       # routing summaries, abs
TOL_SIGMA = 1e-3         # singular values, relative
TOL_RECON = 5e-3         # per-span reconstruction U diag(sigma g) Vt, relative Frobenius


@pytest.fixture(scope="module")
def sk():
    from decode_attention_span_gb300 import build
    build.build()
    import decode_attention_span_gb300 as sk
    return sk


def run_build(sk, w, inp):
    ms = inp["max_spans"]
    cfg = sk.Config(w.batch, w.n_q_heads, w.n_kv_heads, w.n_sink, w.n_recent, ms, w.rank_cap,
                    w.len_min, w.len_max, w.tau)
    ws = sk.Workspace(cfg, which=sk.sekv.SEKV_CALL_BUILD, ctx_len=w.ctx)
    out = sk.alloc_cache(cfg, 256 << 20)
    sk.build_spans(cfg, inp["K"].cuda(), inp["V"].cuda(), torch.from_numpy(inp["H"]).cuda(),
                   inp["W_r"].cuda(), torch.from_numpy(inp["gates"]).cuda(), out, ws)
    torch.cuda.synchronize()
    assert ws.status() == (0, 0)
    return cfg, out


def ulp_bf16(x):
    e = np.floor(np.log2(np.maximum(np.abs(x), 1e-30)))
    return 2.0 ** (e - 7)


def oracle_build(w, inp):
    K, V = inp["K"].float().numpy(), inp["V"].float().numpy()
    return oracle.build_layer(K, V, inp["H"], inp["W_r"].numpy(), inp["gates"],
                              n_sink=w.n_sink, n_recent=w.n_recent, tau=w.tau,
                              len_min=w.len_min, len_max=w.len_max, rank_cap=w.rank_cap)


def check_build(w, inp, out):
    ref = oracle_build(w, inp)
    got = layout.unpack_layer(gen.abi_to_numpy(out), w.n_sink, w.n_recent)
    worst = dict(sigma=0.0, recon=0.0, s=0.0, sum_ulps=0.0, spans=0)
    for b in range(w.batch):
        assert np.array_equal(got.body_len[b], ref.body_len[b]), "spans differ"
        for c in range(w.n_kv_heads):
            assert np.array_equal(got.k_full[b][c], ref.k_full[b][c])
            assert np.array_equal(got.v_full[b][c], ref.v_full[b][c])
            ds = np.abs(got.s_route[b][c] - ref.s_route[b][c]).max(initial=0)
            worst["s"] = max(worst["s"], ds)
            for X, Y in ((got.k_sum[b][c], ref.k_sum[b][c]), (got.v_sum[b][c], ref.v_sum[b][c])):
                d = np.abs(X - Y) / ulp_bf16(Y)
                worst["sum_ulps"] = max(worst["sum_ulps"], d.max(initial=0))
            for Fg, Fr in zip(got.factors[b][c], ref.factors[b][c]):
                if Fr is None:
                    assert Fg is None
                    continue
                worst["spans"] += 1
                for side in ("K", "V"):
                    sg, sr = getattr(Fg, "s" + side), getattr(Fr, "s" + side)
                    assert sg.shape == sr.shape, "ranks differ"
                    if len(sr) == 0:
                        continue
                    worst["sigma"] = max(worst["sigma"], np.max(np.abs(sg - sr) / sr))
                    Rg = oracle.reconstruct(getattr(Fg, "U" + side), sg, getattr(Fg, "g" + side),
                                            getattr(Fg, "Vt" + side))
                    Rr = oracle.reconstruct(getattr(Fr, "U" + side), sr, getattr(Fr, "g" + side),
                                            getattr(Fr, "Vt" + side))
                    worst["recon"] = max(worst["recon"],
                                         np.linalg.norm(Rg - Rr) / np.linalg.norm(Rr))
    assert worst["s"] <= TOL_S_ROUTE, worst
    assert worst["sum_ulps"] <= 1.0, worst
    assert worst["sigma"] <= TOL_SIGMA, worst
    assert worst["recon"] <= TOL_RECON, worst
    return worst


def test_build_pr1(sk):
    w = synth.get_config("pr1")
    inp = gen.build_inputs(w, 0)
    cfg, out = run_build(sk, w, inp)
    check_build(w, inp, out)


@pytest.mark.parametrize("over", [
    dict(ctx=16384, n_kv_heads=2, n_q_heads=8),                           # random gates, cap 32
    dict(ctx=16384, n_kv_heads=2, n_q_heads=8, tau=6.1, len_max=512),     # bodies > 128: M^T M
    dict(ctx=3000, n_kv_heads=2, n_q_heads=8, batch=2, rank_cap=64),      # batch 2, cap 64
])
def test_build_matches_oracle(sk, over):
    w = synth.get_config("mistral_7b_build_128k", layers=1, **over)
    inp = gen.build_inputs(w, 0)
    cfg, out = run_build(sk, w, inp)
    print(check_build(w, inp, out))


def test_build_then_decode(sk):
    """A GPU-built cache decodes like the oracle's own build of the same inputs."""
    from cases import SCALE, compare_out, thresholds
    w = synth.get_config("pr1")
    inp = gen.build_inputs(w, 0)
    cfg, out = run_build(sk, w, inp)
    ref = oracle_build(w, inp)
    q = inp["q"]
    z = oracle.route_logits(q.float().numpy(), inp["W_r"].numpy(), ref)
    theta = thresholds(z, w.n_q_heads, w.expand_frac, w.group)
    E, _ = oracle.route(q.float().numpy(), inp["W_r"].numpy(), ref, theta)
    o_ref, _ = oracle.decode_attention(q.float().numpy(), ref, E, SCALE)
    cache = sk.LayerCache(out)
    ws = sk.Workspace(cfg)
    o, lse, lst, cnt = sk.decode_step(cfg, cache, q.cuda(), inp["W_r"].cuda(),
                                      torch.from_numpy(theta).cuda(), SCALE, ws, want_list=True)
    torch.cuda.synchronize()
    cnt = cnt.cpu().numpy()
    lst = lst.cpu().numpy().reshape(w.n_kv_heads, -1)
    for c in range(w.n_kv_heads):
        assert np.array_equal(lst[c, :cnt[c]], E[0][c])
    compare_out(o.cpu().numpy(), o_ref, "built cache")
