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
