"""The workspace-free decode step gives the same results as the regular one.

sekv_decode_step_noalloc serves callers that cannot allocate device memory
(for instance a plugin whose host engine owns all GPU memory, or a decode loop
that must not call cudaMalloc between tokens): it keeps its scratch in a fixed
8 MiB device array inside the library.  This file is named so that pytest
collects it last; it must pass on its own in a fresh process as well as after
the other GPU tests (the shared array then holds an earlier call's data).
"""
import ctypes

import numpy as np
import pytest
import torch

from cases import SCALE, TOL_ABS, TOL_REL, decode_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sk():
    from decode_attention_span_gb300 import build
    build.build()
    import decode_attention_span_gb300 as sk
    return sk


def _close(a, b, what):
    a = a.cpu().numpy().astype(np.float64)
    b = b.cpu().numpy().astype(np.float64)
    err = np.abs(a - b).max()
    rel = np.linalg.norm(a - b) / np.linalg.norm(b)
    assert np.all(np.isfinite(a)), what
    assert err <= TOL_ABS and rel <= TOL_REL, f"{what}: max abs {err:.3e}, rel L2 {rel:.3e}"


@pytest.mark.parametrize("name,over", [
    ("llama3_8b_32k", dict(ctx=8192)),
    ("qwen2_7b_stress", dict(ctx=8192, batch=2)),
])
def test_noalloc_matches_decode_step_twice(sk, name, over):
    case = decode_case(name, run_oracle=False, **over)
    w = case.wcfg
    cfg = sk.Config(w.batch, w.n_q_heads, w.n_kv_heads, w.n_sink, w.n_recent,
                    case.tensors["max_spans"], w.rank_cap, w.len_min, w.len_max, w.tau)
    cache = sk.LayerCache({k: v.cuda() for k, v in case.tensors.items()
                           if isinstance(v, torch.Tensor)})
    q, W = case.q.cuda(), case.W.cuda()
    theta = torch.from_numpy(case.theta).cuda()
    ws = sk.Workspace(cfg)
    ref, ref_lse, ref_lst, ref_cnt = sk.decode_step(cfg, cache, q, W, theta, SCALE, ws,
                                                    want_list=True)
    torch.cuda.synchronize()
    assert ws.status() == (0, 0)
    for call in range(2):  # the second call finds the first call's data in the array
        out, lse, lst, cnt = sk.decode_step_noalloc(cfg, cache, q, W, theta, SCALE,
                                                    want_list=True)
        torch.cuda.synchronize()
        assert sk.sekv.noalloc_status() == (0, 0)
        _close(out, ref, f"{name} call {call}")
        assert torch.allclose(lse, ref_lse, atol=1e-3)
        assert torch.equal(cnt, ref_cnt)
        for g in range(cnt.numel()):
            n = int(cnt[g])
            ms = cfg.max_spans
            assert torch.equal(lst[g * ms:g * ms + n], ref_lst[g * ms:g * ms + n])


def test_noalloc_rejects_shapes_beyond_its_array(sk):
    case = decode_case("llama3_8b_32k", ctx=4096, run_oracle=False)
    w = case.wcfg
    big = sk.Config(64, w.n_q_heads, w.n_kv_heads, w.n_sink, w.n_recent, 8192, w.rank_cap)
    need = sk.sekv.lib().sekv_workspace_size(ctypes.byref(big.c()), 2, 0)
    assert need > (8 << 20)
    cache = sk.LayerCache({k: v.cuda() for k, v in case.tensors.items()
                           if isinstance(v, torch.Tensor)})
    with pytest.raises(sk.SekvError) as e:
        sk.decode_step_noalloc(big, cache, case.q.cuda(), case.W.cuda(),
                               torch.from_numpy(case.theta).cuda(), SCALE)
    assert e.value.status == -2
