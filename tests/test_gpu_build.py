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


def run_build(sk, w, inp, store_bytes=256 << 20):
    ms = inp["max_spans"]
    cfg = sk.Config(w.batch, w.n_q_heads, w.n_kv_heads, w.n_sink, w.n_recent, ms, w.rank_cap,
                    w.len_min, w.len_max, w.tau)
    ws = sk.Workspace(cfg, which=sk.sekv.SEKV_CALL_BUILD, ctx_len=w.ctx)
    out = sk.alloc_cache(cfg, store_bytes)
    sk.build_spans(cfg, inp["K"].cuda(), inp["V"].cuda(), torch.from_numpy(inp["H"]).cuda(),
                   inp["W_r"].cuda(), torch.from_numpy(inp["gates"]).cuda(), out, ws)
    torch.cuda.synchronize()
    assert ws.status() == (0, 0)
    out["_ws"] = ws
    return cfg, out


def ulp_bf16(x):
    e = np.floor(np.log2(np.maximum(np.abs(x), 1e-30)))
    return 2.0 ** (e - 7)


def assert_sign_convention(Vt):
    """Each stored basis row's largest-magnitude entry is positive (a tie in
    bf16 between a positive and a negative entry is allowed)."""
    Vt = np.asarray(Vt, np.float64)
    if Vt.size:
        assert np.all(Vt.max(axis=1) >= -Vt.min(axis=1)), "sign convention"


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
                    assert_sign_convention(getattr(Fg, "Vt" + side))
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
    # the operation count covers at least the Gram matrices (n(n+1)/2 dot
    # products of length m = 128 or the body, both sides of every span) and
    # is cleared by the read
    b = out["body_len"][0, :int(out["n_spans"][0])].cpu().numpy().astype(np.int64)
    n = np.minimum(b, 128)
    m = np.where(b > 128, b, 128)
    gram = int(np.sum(n * (n + 1) * m)) * w.n_kv_heads * 2
    flops = sk.build_flops(out["_ws"])
    assert flops >= gram > 0
    assert sk.build_flops(out["_ws"]) == 0


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


def test_build_128k_every_head_sampled_spans(sk):
    """One layer of the 128K prefill build at its stated shape (8 KV heads,
    131,072 tokens, about 4,100 spans per head): every span boundary, anchor
    and rank is checked; summaries, singular values and reconstructions on a
    stated sample of 40 spans per head (spread over the sequence, plus the
    longest bodies), each against the oracle's routines for that span."""
    w = synth.get_config("mistral_7b_build_128k", layers=1)
    inp = gen.build_inputs(w, 0, device="cuda")
    cfg, out = run_build(sk, w, inp, store_bytes=1 << 30)
    K, V = inp["K"], inp["V"]
    H = inp["H"][0]
    anchors, lens = oracle.segment(H, w.n_sink, w.n_recent, w.tau, w.len_min, w.len_max)
    n_sp = len(lens)
    assert int(out["n_spans"][0]) == n_sp and n_sp > 3800
    assert np.array_equal(out["body_len"][0, :n_sp].cpu().numpy(), lens - 1)
    m1 = w.ctx - w.n_recent
    full_idx = torch.as_tensor(np.concatenate([np.arange(w.n_sink), anchors,
                                               np.arange(m1, w.ctx)]), device="cuda")
    nf = len(full_idx)
    assert torch.equal(out["k_full"][0, :, :nf], K[0][:, full_idx])
    assert torch.equal(out["v_full"][0, :, :nf], V[0][:, full_idx])
    gates = inp["gates"]
    rr = out["rec_rank"][0, :, :n_sp].cpu().numpy()
    # ranks of every span from the gates (longest prefix above 0.5, at most
    # min(rank_cap, body)) -- the rule of oracle.span_svd
    for c in range(w.n_kv_heads):
        for side, rk in ((0, rr[c] & 0xFFFF), (1, rr[c] >> 16)):
            g = gates[0, c, side, :n_sp] > 0.5
            R = np.minimum(w.rank_cap, lens - 1)
            prefix = np.where(g.all(axis=1), w.rank_cap, np.argmin(g, axis=1))
            assert np.array_equal(rk, np.minimum(prefix, R) * (lens > 1)), (c, side)
    body = lens - 1
    sample = sorted(set(np.linspace(0, n_sp - 1, 32).astype(int).tolist()) |
                    set(np.argsort(-body)[:8].tolist()))
    store = out["store"]
    rec_off = out["rec_off"][0].cpu().numpy()
    s_route = out["s_route"][0].cpu().numpy()
    k_sum = out["k_sum"][0].float().cpu().numpy()
    v_sum = out["v_sum"][0].float().cpu().numpy()
    W = inp["W_r"].cpu().numpy()
    worst = dict(s=0.0, ulps=0.0, sigma=0.0, recon=0.0)
    for c in range(w.n_kv_heads):
        for k in sample:
            lo, hi = int(anchors[k]) + 1, int(anchors[k]) + int(lens[k])
            if hi <= lo:
                continue
            Kb = K[0, c, lo:hi].double().cpu().numpy()
            Vb = V[0, c, lo:hi].double().cpu().numpy()
            s_ref = oracle.routing_summary(Kb, H[lo:hi], W[c]).astype(np.float32)
            worst["s"] = max(worst["s"], float(np.abs(s_route[c, k] - s_ref).max()))
            km, vm = oracle.attention_summary(Kb, Vb)
            for got, ref in ((k_sum[c, k], oracle.bf16_round(km)), (v_sum[c, k], oracle.bf16_round(vm))):
                worst["ulps"] = max(worst["ulps"], float((np.abs(got - ref) / ulp_bf16(ref)).max()))
            size = sk.record_size(hi - lo, int(rr[c, k] & 0xFFFF), int(rr[c, k] >> 16))
            raw = store[int(rec_off[c, k]):int(rec_off[c, k]) + size].cpu().numpy()
            F = layout.unpack_record(np.concatenate([raw, np.zeros(16, np.uint8)]), 0, hi - lo)
            for side, M in (("K", Kb), ("V", Vb)):
                fr = oracle.span_svd(M, gates[0, c, 0 if side == "K" else 1, k], w.rank_cap)
                sg = getattr(F, "s" + side)
                assert len(sg) == fr.rank
                if fr.rank == 0:
                    continue
                worst["sigma"] = max(worst["sigma"], float(np.max(np.abs(sg - fr.sigma) / fr.sigma)))
                assert_sign_convention(getattr(F, "Vt" + side))
                Rg = oracle.reconstruct(getattr(F, "U" + side), sg, getattr(F, "g" + side),
                                        getattr(F, "Vt" + side))
                Rr = oracle.reconstruct(fr.U, fr.sigma, fr.gate, fr.Vt)
                worst["recon"] = max(worst["recon"], float(np.linalg.norm(Rg - Rr) / np.linalg.norm(Rr)))
    assert worst["s"] <= TOL_S_ROUTE, worst
    assert worst["ulps"] <= 1.0, worst
    assert worst["sigma"] <= TOL_SIGMA, worst
    assert worst["recon"] <= TOL_RECON, worst
