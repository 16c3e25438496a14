"""Byte layout fixtures and generator properties (CPU)."""
import struct

import numpy as np
import pytest

import oracle
import synth
from oracle import layout
from synth import gen


def bf(x):
    return struct.pack("<H", struct.unpack("<I", struct.pack("<f", x))[0] >> 16)


def test_record_bytes_by_hand():
    # b = 1, rK = 1, rV = 2, spelled out field by field from the C header
    UK = np.array([[0.5]]); VtK = np.zeros((1, 128)); VtK[0, 0] = 1.0
    UV = np.array([[2.0, -1.0]]); VtV = np.zeros((2, 128)); VtV[0, 1] = 1.0; VtV[1, 2] = -0.25
    F = oracle.SpanFactors(UK=UK, sK=np.array([3.0]), gK=np.array([0.75]), VtK=VtK,
                           UV=UV, sV=np.array([1.5, 0.5]), gV=np.array([1.0, 0.625]), VtV=VtV)
    want = b""
    want += struct.pack("<4i", 1, 1, 2, 0)                      # header
    want += struct.pack("<4f", 3.0, 0, 0, 0)                    # sigma_K (pad to 4)
    want += struct.pack("<4f", 0.75, 0, 0, 0)                   # g_K
    want += bf(1.0) + bf(0.0) * 127                             # Vt_K 1 x 128
    want += bf(0.5) + b"\0" * 14                                # U_K 1 x 1, pad 16
    want += bf(2.0) + bf(-1.0) + b"\0" * 12                     # U_V 1 x 2, pad 16
    want += struct.pack("<4f", 1.5, 0.5, 0, 0)                  # sigma_V
    want += struct.pack("<4f", 1.0, 0.625, 0, 0)                # g_V
    want += bf(0.0) + bf(1.0) + bf(0.0) * 126                   # Vt_V row 0
    # Vt_V row 1: chunk 0 (columns 0..7) is stored at chunk position 0 ^ 1 = 1
    want += bf(0.0) * 10 + bf(-0.25) + bf(0.0) * 117            # Vt_V row 1
    got = layout.pack_record(F)
    assert got == want
    assert len(want) == layout.record_size(1, 1, 2) == gen.record_size(1, 1, 2)
    F2 = layout.unpack_record(np.frombuffer(want, np.uint8), 0)
    for name in ("UK", "sK", "gK", "VtK", "UV", "sV", "gV", "VtV"):
        assert np.array_equal(getattr(F2, name), getattr(F, name))


def test_record_size_agrees_between_writers():
    for b in (0, 1, 2, 7, 31, 255, 511):
        for rK in (0, 1, 3, 4, 16, 33, 64):
            for rV in (0, 2, 5, 32, 64):
                assert layout.record_size(b, rK, rV) == gen.record_size(b, rK, rV)
                assert layout.record_size(b, rK, rV) % 16 == 0


def test_pack_unpack_roundtrip_built_cache():
    cfg = synth.get_config("pr1")
    inp = gen.build_inputs(cfg, 0, max_spans=None)
    K = inp["K"][:, :2].float().numpy(); V = inp["V"][:, :2].float().numpy()
    c = oracle.build_layer(K, V, inp["H"], inp["W_r"][:2].numpy(), inp["gates"][:, :2],
                           n_sink=cfg.n_sink, n_recent=cfg.n_recent, tau=cfg.tau,
                           len_min=cfg.len_min, len_max=cfg.len_max, rank_cap=cfg.rank_cap)
    arr = layout.pack_layer(c, inp["max_spans"])
    c2 = layout.unpack_layer(arr, cfg.n_sink, cfg.n_recent)
    assert np.array_equal(c2.body_len[0], c.body_len[0])
    for ci in range(2):
        assert np.array_equal(c2.k_full[0][ci], c.k_full[0][ci])
        assert np.array_equal(c2.k_sum[0][ci], c.k_sum[0][ci])
        for a, b in zip(c2.factors[0][ci], c.factors[0][ci]):
            if a is None:
                assert b is None
                continue
            assert np.array_equal(a.UK, b.UK) and np.array_equal(a.VtV, b.VtV)
            assert np.array_equal(a.sK, b.sK) and np.array_equal(a.gV, b.gV)
    # the planted spans are the oracle's spans; PR1 keeps rank min(16, b)
    assert np.array_equal(c.body_len[0] + 1, inp["lens"][0])
    for F, b in zip(c.factors[0][0], c.body_len[0]):
        if F is not None:
            assert F.sK.shape[0] == min(16, b)


def test_surprisal_margin_and_seed():
    cfg = synth.get_config("pr1")
    a = gen.build_inputs(cfg, 0)
    b = gen.build_inputs(cfg, 0)
    assert np.array_equal(a["H"], b["H"])
    assert np.all(np.abs(a["H"].astype(np.float64) - np.float32(cfg.tau)) >= 1e-3)
    assert (a["K"] == b["K"]).all()


def test_span_length_statistics():
    g = gen._gen(0)
    for tau, lmax, mean in ((5.2, 256, 32.2), (4.0, 256, 13.9)):
        L = gen.span_lengths(g, 2_000_000, tau, 4, lmax)
        assert abs(L[:-1].mean() - mean) / mean < 0.02
        assert L[:-1].min() >= 4 and L.max() <= lmax


def test_pick_threshold_margin_and_rate():
    rng = np.random.default_rng(0)
    z = rng.standard_normal(5000)
    for frac in (0.01, 0.05, 0.3):
        th = gen.pick_threshold(z, frac, 1e-3)
        assert th.dtype == np.float32
        assert np.all(np.abs(z - float(th)) >= 1e-3)
        assert abs(np.mean(z > th) - frac) < 0.01
