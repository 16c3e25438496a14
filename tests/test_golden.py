"""Hand-worked fixtures under tests/golden/ (each file states its derivation
and the passage of the pages it follows)."""

import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _read(name):
    vals = {}
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                key, *rest = line.split()
                vals[key] = rest
    return vals


def test_segmentation_worked_example():
    v = _read("segmentation_worked.txt")
    H = np.array([float(x) for x in v["H"]], np.float32)
    starts, lens = oracle.segment(H, int(v["n_sink"][0]), int(v["n_recent"][0]),
                                  float(v["tau"][0]), int(v["len_min"][0]),
                                  int(v["len_max"][0]))
    assert [int(x) for x in starts] == [int(x) for x in v["anchors"]]
    assert [int(x) for x in lens] == [int(x) for x in v["lengths"]]
    assert [int(x) - 1 for x in lens] == [int(x) for x in v["body_len"]]


def test_identical_keys_attention_worked_example():
    v = _read("attention_identical_keys_worked.txt")
    T = int(v["T"][0])
    K = np.full((1, 1, T, 128), float(v["key"][0]))
    Vv = np.repeat(np.arange(T, dtype=np.float64)[:, None], 128, axis=1)[None, None]
    H = np.zeros((1, T), np.float32)
    W_r = np.eye(64, 128, dtype=np.float32)[None]
    gates = np.ones((1, 1, 2, T, 16), np.float32)
    cache = oracle.build_layer(K, Vv, H, W_r, gates, n_sink=int(v["n_sink"][0]),
                               n_recent=int(v["n_recent"][0]), tau=float(v["tau"][0]),
                               len_min=int(v["len_min"][0]), len_max=int(v["len_max"][0]),
                               rank_cap=16)
    assert [int(x) for x in cache.anchors[0]] == [2, 6]
    q = np.full((1, 1, 128), float(v["query"][0]))
    o, lse = oracle.decode_attention(q, cache, [[[]]], 1.0 / np.sqrt(128.0))
    np.testing.assert_allclose(o[0, 0], float(v["o"][0]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[0, 0], float(v["lse"][0]), rtol=0, atol=1e-12)


def _read_multi(name):
    """Like _read, but keys may repeat (one list of values per line)."""
    vals = {}
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                key, *rest = line.split()
                vals.setdefault(key, []).append(rest)
    return vals


def test_build_layer_weights_and_gates_worked_example():
    """build_layer with unequal surprisal and distinct key/value gates: a
    shifted surprisal slice or swapped gate index changes the expected
    routing summaries or ranks."""
    v = _read_multi("build_layer_weights_worked.txt")
    one = lambda k: v[k][0][0]  # noqa: E731
    T, rc = int(one("T")), int(one("rank_cap"))
    K = np.zeros((1, 1, T, 128))
    Vv = np.zeros((1, 1, T, 128))
    for arr, key in ((K, "k"), (Vv, "v")):
        for t, d, x in v[key]:
            arr[0, 0, int(t), int(d)] = float(x)
    H = np.array([float(x) for x in v["H"][0]], np.float32)[None]
    gates = np.zeros((1, 1, 2, 2, rc), np.float32)
    for i, key in enumerate(("gk", "gv")):
        for k, *g in v[key]:
            gates[0, 0, i, int(k)] = [float(x) for x in g]
    W_r = np.eye(64, 128, dtype=np.float32)[None]
    cache = oracle.build_layer(K, Vv, H, W_r, gates, n_sink=int(one("n_sink")),
                               n_recent=int(one("n_recent")), tau=float(one("tau")),
                               len_min=int(one("len_min")), len_max=int(one("len_max")),
                               rank_cap=rc)
    assert [int(x) for x in cache.anchors[0]] == [int(x) for x in v["anchors"][0]]
    assert [int(x) for x in cache.body_len[0]] == [int(x) for x in v["body_len"][0]]
    for name, arr in (("s_route", cache.s_route), ("k_sum", cache.k_sum), ("v_sum", cache.v_sum)):
        want = np.zeros_like(arr[0][0])
        for k, d, x in v[name]:
            want[int(k), int(d)] = float(x)
        np.testing.assert_allclose(arr[0][0], want, rtol=0, atol=1e-7, err_msg=name)
    F = cache.factors[0][0]
    assert [f.sK.shape[0] for f in F] == [int(x) for x in v["rank_k"][0]]
    assert [f.sV.shape[0] for f in F] == [int(x) for x in v["rank_v"][0]]
    for key, attr in (("sigma_k", "sK"), ("sigma_v", "sV")):
        for k, *s in v[key]:
            np.testing.assert_allclose(getattr(F[int(k)], attr), [float(x) for x in s],
                                       rtol=1e-7, atol=0)
