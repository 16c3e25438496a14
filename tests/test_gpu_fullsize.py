"""GPU parity of the decode step at the workloads' stated shapes.

Routing and attention: SeKV technical summary, Methodik 3 (German page) /
方法论 3 (Chinese page).  Every (sequence, KV head) group's expansion list is
compared bit for bit with the oracle's; the attention outputs of every group
(or of a stated sample of groups, for the batch-16 stress shape) are compared
element by element within max-abs 1e-2 and relative-L2 5e-3.

These shapes reach what small slices do not: many routing pages per CTA,
hundreds of expanded records per KV head, long bodies split over several
pages, and (for 2 KV heads) far more than 32 CTAs per KV head in the merge.
"""
import numpy as np
import pytest
import torch

from cases import SCALE, compare_out, sampled_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sk():
    from decode_attention_span_gb300 import build
    build.build()
    import decode_attention_span_gb300 as sk
    return sk


def run_and_compare(sk, case, what, reps=1, scale=SCALE):
    w = case.wcfg
    ms = case.tensors["max_spans"]
    cfg = sk.Config(w.batch, w.n_q_heads, w.n_kv_heads, w.n_sink, w.n_recent, ms, w.rank_cap,
                    w.len_min, w.len_max, w.tau)
    cache = sk.LayerCache({k: v.cuda() for k, v in case.tensors.items()
                           if isinstance(v, torch.Tensor)})
    ws = sk.Workspace(cfg)
    G = w.group
    for rep in range(reps):
        out, lse, lst, cnt = sk.decode_step(cfg, cache, case.q.cuda(), case.W.cuda(),
                                            torch.from_numpy(case.theta).cuda(), scale, ws,
                                            want_list=True)
        torch.cuda.synchronize()
        assert ws.status() == (0, 0)
        lst = lst.cpu().numpy().reshape(w.batch, w.n_kv_heads, ms)
        cnt = cnt.cpu().numpy().reshape(w.batch, w.n_kv_heads)
        for (b, c), E in case.E.items():
            assert cnt[b, c] == len(E), (what, b, c, int(cnt[b, c]), len(E))
            assert np.array_equal(lst[b, c, :cnt[b, c]], E), (what, b, c)
        out = out.cpu().numpy()
        lse = lse.cpu().numpy()
        for (b, c), o_ref in case.o.items():
            compare_out(out[b, c * G:(c + 1) * G], o_ref, f"{what} group ({b},{c}) rep {rep}")
            assert np.allclose(lse[b, c * G:(c + 1) * G], case.lse[(b, c)], atol=1e-3)
    return cnt


def test_headline_128k_every_head(sk):
    """One layer of the 128K Llama-3-8B shape: batch 1, 8 KV heads, about
    4,100 spans per head, about 5% of them expanded; every head checked."""
    case = sampled_case("llama3_8b_128k", layer=0)
    cnt = run_and_compare(sk, case, "128k", reps=2)
    n_sp = int(case.tensors["n_spans"][0])
    frac = cnt.sum() / (8 * n_sp)
    assert n_sp > 3500 and 0.03 < frac < 0.08


def test_32k_every_head(sk):
    case = sampled_case("llama3_8b_32k", layer=3)
    run_and_compare(sk, case, "32k")


def test_qwen_stress_batch16_64k(sk):
    """Qwen2-7B-shaped stress layer at its stated shape: batch 16 x 64K, group
    7, bodies up to 511 tokens, ranks up to 64, about 30% expanded.  Lists of
    all 64 groups are compared; outputs of 8 groups spread over the batch."""
    sample = [(0, 0), (2, 1), (5, 3), (7, 2), (9, 0), (11, 1), (13, 3), (15, 2)]
    case = sampled_case("qwen2_7b_stress", layer=0, sample=sample, device="cuda")
    cnt = run_and_compare(sk, case, "qwen")
    assert 0.2 < cnt.sum() / sum(int(n) for n in case.tensors["n_spans"].cpu()) / 4 < 0.4


def test_two_kv_heads_128k_many_ctas(sk):
    """2 KV heads at 128K: every KV head is shared by far more CTAs than the
    merge takes in one round trip, each with several routing pages."""
    case = sampled_case("llama3_8b_128k", layer=1, n_kv_heads=2, n_q_heads=8)
    run_and_compare(sk, case, "2kv 128k")


@pytest.mark.parametrize("mode", ["frac", "all"])
def test_edge_records_rank0_short_and_empty_bodies(sk, mode):
    """Records with rank 0 on the keys, on the values or on both (rank budget
    drawn from 0..32), bodies of one token, and empty bodies in the middle of
    the sequence (spans of length 1, len_min = 1)."""
    case = sampled_case("llama3_8b_32k", layer=0, mode=mode, ctx=16384, rank_lo=0, len_min=1,
                        expand_frac=0.5)
    t = case.tensors
    body = t["body_len"][0, :int(t["n_spans"][0])].cpu().numpy()
    rr = t["rec_rank"][0, :, :len(body)].cpu().numpy()
    rk, rv = rr & 0xFFFF, rr >> 16
    nonempty = body[None, :] > 0
    # the workload holds every edge this test is about
    assert (body[:-1] == 0).any() and (body == 1).any()
    assert ((rk == 0) & (rv > 0) & nonempty).any() and ((rv == 0) & (rk > 0) & nonempty).any()
    expanded_r0 = sum(int(((rk[c] == 0) | (rv[c] == 0))[case.E[(0, c)]].sum()) for c in range(8))
    assert expanded_r0 > 0
    run_and_compare(sk, case, f"edges {mode}")


def test_sharp_softmax_128k(sk):
    """A 6x logit scale at 128K: the running max re-bases often, across pages,
    records and CTAs."""
    case = sampled_case("llama3_8b_128k", layer=2, sample=[(0, 0), (0, 5)], scale=6 * SCALE)
    run_and_compare(sk, case, "sharp 128k", scale=6 * SCALE)
