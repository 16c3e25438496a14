"""GPU parity of routing and mixed-resolution decode attention vs the oracle.

Routing and attention: SeKV technical summary, Methodik 3 (German page) /
方法论 3 (Chinese page).  Expansion sets must be bit-exact (the generator keeps
every gate logit at least 1e-3 from its threshold); attention outputs must
match within max-abs 1e-2 and relative-L2 5e-3.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import layout
import synth
from synth import gen

from cases import SCALE, compare_out, decode_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sk():
    from decode_attention_span_gb300 import build
    build.build()
    import decode_attention_span_gb300 as sk
    return sk


def to_dev(case, dev="cuda"):
    return {k: v.to(dev) for k, v in case.tensors.items() if isinstance(v, torch.Tensor)}


def sk_config(sk, case):
    w = case.wcfg
    return sk.Config(w.batch, w.n_q_heads, w.n_kv_heads, w.n_sink, w.n_recent,
                     case.tensors["max_spans"], w.rank_cap, w.len_min, w.len_max, w.tau)


def lists_equal(case, lst, cnt):
    w = case.wcfg
    ms = case.tensors["max_spans"]
    lst = lst.cpu().numpy().reshape(w.batch, w.n_kv_heads, ms)
    cnt = cnt.cpu().numpy().reshape(w.batch, w.n_kv_heads)
    for b in range(w.batch):
        for c in range(w.n_kv_heads):
            assert np.array_equal(lst[b, c, :cnt[b, c]], case.E[b][c]), (b, c)


CASES = [
    ("llama3_8b_32k", dict(ctx=8192), "frac"),
    ("llama3_8b_32k", dict(ctx=8192, batch=2, expand_frac=0.3), "frac"),
    ("qwen2_7b_stress", dict(ctx=8192, batch=2), "frac"),
    ("llama3_8b_32k", dict(ctx=4096), "none"),
    ("llama3_8b_32k", dict(ctx=4096), "all"),
    ("qwen2_7b_stress", dict(ctx=4096, batch=1), "all"),
]


@pytest.mark.parametrize("name,over,mode", CASES)
def test_decode_step_matches_oracle(sk, name, over, mode):
    case = decode_case(name, mode=mode, **over)
    cfg = sk_config(sk, case)
    cache = sk.LayerCache(to_dev(case))
    ws = sk.Workspace(cfg)
    for rep in range(2):  # the workspace must be reusable call after call
        out, lse, lst, cnt = sk.decode_step(cfg, cache, case.q.cuda(), case.W.cuda(),
                                            torch.from_numpy(case.theta).cuda(), SCALE, ws,
                                            want_list=True)
        torch.cuda.synchronize()
        assert ws.status() == (0, 0)
        lists_equal(case, lst, cnt)
        compare_out(out.cpu().numpy(), case.o, f"{name} {mode} rep {rep}")
        assert np.allclose(lse.cpu().numpy(), case.lse, atol=1e-3)


@pytest.mark.parametrize("name,over", [("llama3_8b_32k", dict(ctx=8192)),
                                       ("qwen2_7b_stress", dict(ctx=8192, batch=1))])
def test_decode_step_sharp_softmax(sk, name, over):
    """A 6x softmax scale spreads the logits over tens of log2 units, so the
    online softmax re-bases its running max often, also between the 16-token
    tiles of one expanded span: every partial sum must follow the re-base."""
    case = decode_case(name, mode="all", run_oracle=False, **over)
    sharp = 6.0 * SCALE
    o_ref, lse_ref = oracle.decode_attention(case.q.float().numpy(), case.cache, case.E, sharp)
    cfg = sk_config(sk, case)
    cache = sk.LayerCache(to_dev(case))
    ws = sk.Workspace(cfg)
    out, lse, _, _ = sk.decode_step(cfg, cache, case.q.cuda(), case.W.cuda(),
                                    torch.from_numpy(case.theta).cuda(), sharp, ws)
    torch.cuda.synchronize()
    assert ws.status() == (0, 0)
    compare_out(out.cpu().numpy(), o_ref, f"{name} sharp softmax")
    assert np.allclose(lse.cpu().numpy(), lse_ref, atol=1e-3)


@pytest.mark.parametrize("name,over,mode", CASES[:3])
def test_route_matches_oracle(sk, name, over, mode):
    case = decode_case(name, mode=mode, run_oracle=False, **over)
    cfg = sk_config(sk, case)
    cache = sk.LayerCache(to_dev(case))
    ws = sk.Workspace(cfg)
    lst, cnt, z = sk.route(cfg, cache, case.q.cuda(), case.W.cuda(),
                           torch.from_numpy(case.theta).cuda(), ws, want_z=True)
    torch.cuda.synchronize()
    lists_equal(case, lst, cnt)
    w = case.wcfg
    z = z.cpu().numpy().reshape(w.batch, w.n_q_heads, -1)
    for b in range(w.batch):
        for h in range(w.n_q_heads):
            n = len(case.z[b][h])
            assert np.abs(z[b, h, :n] - case.z[b][h]).max() < 1e-4


@pytest.mark.parametrize("name,over,mode", CASES[:3] + CASES[4:5])
def test_decode_attention_with_oracle_list(sk, name, over, mode):
    case = decode_case(name, mode=mode, **over)
    cfg = sk_config(sk, case)
    cache = sk.LayerCache(to_dev(case))
    ws = sk.Workspace(cfg)
    w = case.wcfg
    ms = case.tensors["max_spans"]
    lst = np.zeros((w.batch, w.n_kv_heads, ms), np.int32)
    cnt = np.zeros((w.batch, w.n_kv_heads), np.int32)
    for b in range(w.batch):
        for c in range(w.n_kv_heads):
            e = case.E[b][c]
            lst[b, c, :len(e)] = e
            cnt[b, c] = len(e)
    out, lse = sk.decode_attention(cfg, cache, case.q.cuda(), torch.from_numpy(lst).cuda(),
                                   torch.from_numpy(cnt).cuda(), SCALE, ws)
    torch.cuda.synchronize()
    assert ws.status() == (0, 0)
    compare_out(out.cpu().numpy(), case.o, f"{name} list")


def test_pr1_full_pipeline(sk):
    """PR1 (one layer, 4K context): oracle-built cache, GPU routing + attention."""
    w = synth.get_config("pr1")
    inp = gen.build_inputs(w, 0)
    K, V = inp["K"].float().numpy(), inp["V"].float().numpy()
    cache_o = oracle.build_layer(K, V, inp["H"], inp["W_r"].numpy(), inp["gates"],
                                 n_sink=w.n_sink, n_recent=w.n_recent, tau=w.tau,
                                 len_min=w.len_min, len_max=w.len_max, rank_cap=w.rank_cap)
    arr = layout.pack_layer(cache_o, inp["max_spans"])
    q = inp["q"]
    z = oracle.route_logits(q.float().numpy(), inp["W_r"].numpy(), cache_o)
    from cases import thresholds
    theta = thresholds(z, w.n_q_heads, w.expand_frac, w.group)
    E, _ = oracle.route(q.float().numpy(), inp["W_r"].numpy(), cache_o, theta)
    o_ref, lse_ref = oracle.decode_attention(q.float().numpy(), cache_o, E, SCALE)
    t = {k: torch.from_numpy(v) for k, v in arr.items()}
    for k in ("k_full", "v_full", "k_sum", "v_sum"):
        t[k] = t[k].view(torch.bfloat16)
    cfg = sk.Config(1, w.n_q_heads, w.n_kv_heads, w.n_sink, w.n_recent, inp["max_spans"],
                    w.rank_cap, w.len_min, w.len_max, w.tau)
    cache = sk.LayerCache({k: v.cuda() for k, v in t.items()})
    ws = sk.Workspace(cfg)
    out, lse, lst, cnt = sk.decode_step(cfg, cache, q.cuda(), inp["W_r"].cuda(),
                                        torch.from_numpy(theta).cuda(), SCALE, ws,
                                        want_list=True)
    torch.cuda.synchronize()
    assert ws.status() == (0, 0)
    cnt = cnt.cpu().numpy()
    lst = lst.cpu().numpy().reshape(w.n_kv_heads, -1)
    for c in range(w.n_kv_heads):
        assert np.array_equal(lst[c, :cnt[c]], E[0][c])
    frac = cnt.sum() / (w.n_kv_heads * len(cache_o.body_len[0]))
    assert 0.03 < frac < 0.3
    compare_out(out.cpu().numpy(), o_ref, "pr1")


def test_tiered_fetch_matches_resident(sk):
    case = decode_case("llama3_8b_32k", ctx=8192, expand_frac=0.2)
    cfg = sk_config(sk, case)
    dev = to_dev(case)
    cache = sk.LayerCache(dev)
    host = dict(dev)
    host["store"] = case.tensors["store"].pin_memory()
    cache_h = sk.LayerCache(host, store_on_host=True)
    ws = sk.Workspace(cfg)
    th = torch.from_numpy(case.theta).cuda()
    lst, cnt, _ = sk.route(cfg, cache_h, case.q.cuda(), case.W.cuda(), th, ws)
    NG = case.wcfg.batch * case.wcfg.n_kv_heads
    per_group = 8 << 20
    staging = torch.empty(NG * per_group, dtype=torch.uint8, device="cuda")
    staged_off = torch.empty(NG * case.tensors["max_spans"], dtype=torch.int64, device="cuda")
    sk.fetch_bases(cfg, cache_h, lst, cnt, staging, per_group, staged_off, ws)
    out, lse = sk.decode_attention(cfg, cache_h, case.q.cuda(), lst, cnt, SCALE, ws,
                                   staging=staging, staged_off=staged_off)
    torch.cuda.synchronize()
    assert ws.status() == (0, 0)
    compare_out(out.cpu().numpy(), case.o, "tiered")
    out2, _, _, _ = sk.decode_step(cfg, cache, case.q.cuda(), case.W.cuda(), th, SCALE, ws)
    torch.cuda.synchronize()
    assert torch.allclose(out, out2, atol=2e-3, rtol=0)


def test_bad_list_is_flagged(sk):
    case = decode_case("llama3_8b_32k", ctx=4096, run_oracle=False)
    cfg = sk_config(sk, case)
    cache = sk.LayerCache(to_dev(case))
    ws = sk.Workspace(cfg)
    ms = case.tensors["max_spans"]
    NG = case.wcfg.n_kv_heads
    lst = torch.zeros(NG * ms, dtype=torch.int32)
    lst[:3] = torch.tensor([5, 3, 9])  # not ascending
    cnt = torch.zeros(NG, dtype=torch.int32)
    cnt[0] = 3
    sk.decode_attention(cfg, cache, case.q.cuda(), lst.cuda(), cnt.cuda(), SCALE, ws)
    code, _ = ws.status()
    assert code == 1
    assert ws.status() == (0, 0)


def test_invalid_arguments_rejected_on_host(sk):
    case = decode_case("llama3_8b_32k", ctx=4096, run_oracle=False)
    cfg = sk_config(sk, case)
    cache = sk.LayerCache(to_dev(case))
    ws = sk.Workspace(cfg)
    bad = sk.Config(**{**cfg.__dict__, "head_dim": 64})
    with pytest.raises(sk.SekvError) as e:
        sk.decode_step(bad, cache, case.q.cuda(), case.W.cuda(),
                       torch.from_numpy(case.theta).cuda(), SCALE, ws)
    assert e.value.status == -5
    bad = sk.Config(**{**cfg.__dict__, "max_spans": 100})
    with pytest.raises(sk.SekvError) as e:
        sk.decode_step(bad, cache, case.q.cuda(), case.W.cuda(),
                       torch.from_numpy(case.theta).cuda(), SCALE, ws)
    assert e.value.status == -1
    small = type(ws).__new__(type(ws))
    small.buf, small.nbytes = ws.buf, 64
    with pytest.raises(sk.SekvError) as e:
        sk.decode_step(cfg, cache, case.q.cuda(), case.W.cuda(),
                       torch.from_numpy(case.theta).cuda(), SCALE, small)
    assert e.value.status == -2


def test_short_waits_time_out_and_leave_the_gpu_usable(sk):
    """With SEKV_FLAG_SHORT_WAITS every wait for a copy gives up if the copy
    has not landed at its first test: some wait runs out, the device status
    reports a timeout (code 2, never a fault), every issued copy still lands
    before the kernel exits, and the next regular call on the same
    workspace is correct."""
    case = decode_case("llama3_8b_32k", ctx=16384)
    cfg = sk_config(sk, case)
    cache = sk.LayerCache(to_dev(case))
    ws = sk.Workspace(cfg)
    short = sk.Config(**{**cfg.__dict__, "flags": sk.sekv.FLAG_SHORT_WAITS})
    th = torch.from_numpy(case.theta).cuda()
    sk.decode_step(short, cache, case.q.cuda(), case.W.cuda(), th, SCALE, ws)
    code, detail = ws.status()
    assert code == 2 and detail in (3, 4, 5, 7), (code, detail)
    assert ws.status() == (0, 0)
    out, lse, _, _ = sk.decode_step(cfg, cache, case.q.cuda(), case.W.cuda(), th, SCALE, ws)
    torch.cuda.synchronize()
    assert ws.status() == (0, 0)
    compare_out(out.cpu().numpy(), case.o, "after the timed-out call")


def test_fetch_copy_path_matches_oracle(sk):
    """The host-driven fetch (one cudaMemcpyAsync per run of adjacent
    records on a side stream, then an event the attention waits on) gives
    the oracle's attention."""
    case = decode_case("llama3_8b_32k", ctx=8192, batch=2, expand_frac=0.2)
    cfg = sk_config(sk, case)
    dev = to_dev(case)
    host = dict(dev)
    host["store"] = case.tensors["store"].pin_memory()
    cache_h = sk.LayerCache(host, store_on_host=True)
    ws = sk.Workspace(cfg)
    lst, cnt, _ = sk.route(cfg, cache_h, case.q.cuda(), case.W.cuda(),
                           torch.from_numpy(case.theta).cuda(), ws)
    lst_h = lst.cpu()
    cnt_h = cnt.cpu()
    rec_off_h = case.tensors["rec_off"].contiguous()
    NG = case.wcfg.batch * case.wcfg.n_kv_heads
    ms = case.tensors["max_spans"]
    per_group = 8 << 20
    staging = torch.empty(NG * per_group, dtype=torch.uint8, device="cuda")
    staged_off = torch.empty(NG * ms, dtype=torch.int64, device="cuda")
    staged_off_h = torch.empty(NG * ms, dtype=torch.int64).pin_memory()
    side = torch.cuda.Stream()
    done = torch.cuda.Event()
    n = sk.fetch_bases_copy(cfg, cache_h, lst_h, cnt_h, rec_off_h, staging, per_group,
                            staged_off_h, staged_off, done, side)
    assert 0 < n <= int(cnt_h.sum())
    torch.cuda.current_stream().wait_event(done)
    out, _ = sk.decode_attention(cfg, cache_h, case.q.cuda(), lst, cnt, SCALE, ws,
                                 staging=staging, staged_off=staged_off)
    torch.cuda.synchronize()
    assert ws.status() == (0, 0)
    compare_out(out.cpu().numpy(), case.o, "copy fetch")


@pytest.mark.parametrize("n_slots", [512, 8])
def test_cached_fetch_matches_oracle_hits_and_evictions(sk, n_slots):
    """Fetch through the residency cache: a first call misses everywhere, a
    second call with the same lists hits everywhere (when the pool holds
    them), a different query hits partly; with 8 slots per group most
    records evict others or go to staging.  Every call's attention is the
    oracle's."""
    cases = [decode_case("llama3_8b_32k", ctx=8192, expand_frac=0.2, seed=s) for s in (7, 8)]
    cfg = sk_config(sk, cases[0])
    dev = to_dev(cases[0])
    host = dict(dev)
    host["store"] = cases[0].tensors["store"].pin_memory()
    cache_h = sk.LayerCache(host, store_on_host=True)
    ws = sk.Workspace(cfg)
    NG = cfg.batch * cfg.n_kv_heads
    ms = cfg.max_spans
    per_group = 8 << 20
    bc = sk.BasisCache(cfg, n_slots, 20480)
    staging = torch.empty(bc.staging_bytes(cfg, per_group), dtype=torch.uint8, device="cuda")
    staged_off = torch.empty(NG * ms, dtype=torch.int64, device="cuda")
    hits = torch.zeros(NG, dtype=torch.int32, device="cuda")
    for i, case in enumerate([cases[0], cases[0], cases[1], cases[0]]):
        lst, cnt, _ = sk.route(cfg, cache_h, case.q.cuda(), case.W.cuda(),
                               torch.from_numpy(case.theta).cuda(), ws)
        sk.fetch_bases_cached(cfg, cache_h, lst, cnt, staging, per_group, bc, staged_off, ws,
                              hits=hits)
        out, _ = sk.decode_attention(cfg, cache_h, case.q.cuda(), lst, cnt, SCALE, ws,
                                     staging=staging, staged_off=staged_off)
        torch.cuda.synchronize()
        assert ws.status() == (0, 0)
        compare_out(out.cpu().numpy(), case.o, f"cached fetch call {i} ({n_slots} slots)")
        h, c = hits.cpu(), cnt.cpu()
        if i == 0:
            assert int(h.sum()) == 0
        if i == 1 and n_slots == 512:
            # everything that fits a 20 KB slot is resident from call 0
            big = 0
            for g in range(NG):
                for k in lst[g * ms:g * ms + int(c[g])].cpu().tolist():
                    rk = int(case.tensors["rec_rank"].view(-1)[g * ms + k])
                    body = int(case.tensors["body_len"].view(-1)[(g // cfg.n_kv_heads) * ms + k])
                    big += sk.record_size(body, rk & 0xFFFF, rk >> 16) > 20480
            assert int(h.sum()) == int(c.sum()) - big
        if n_slots == 8:
            assert (h <= 8).all()
