"""The C-ABI library loads and exports every symbol the header declares (CPU)."""
import os
import re

import pytest

import oracle.layout as olayout

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_symbols():
    text = open(os.path.join(ROOT, "include", "sekv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sekv_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def libsekv():
    from decode_attention_span_gb300 import build, sekv
    build.build()
    return sekv.lib()


def test_exports_every_declared_symbol(libsekv):
    from decode_attention_span_gb300 import sekv
    syms = header_symbols()
    assert set(syms) == set(sekv.EXPORTS), syms
    for s in syms:
        assert hasattr(libsekv, s), s


def test_record_size_matches_layout(libsekv):
    for b in (0, 1, 5, 31, 255, 511):
        for rk in (0, 1, 7, 16, 32, 64):
            for rv in (0, 3, 32, 64):
                assert libsekv.sekv_record_size(b, rk, rv) == olayout.record_size(b, rk, rv)


def test_status_strings(libsekv):
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert libsekv.sekv_status_string(code)


def test_query_blocks(libsekv):
    """Multi-query decode launches blocks of 8 / (Hq / Hkv) query tokens."""
    import decode_attention_span_gb300 as sk
    for hq, hkv in ((32, 8), (28, 4), (8, 4), (8, 8), (16, 2)):
        cfg = sk.Config(1, hq, hkv, 4, 64, 256, 32, 1, 64, 4.0)
        tpb = 8 // (hq // hkv)
        for n in (1, 2, 3, 5, 8, 17, 64):
            assert sk.query_blocks(cfg, n) == -(-n // tpb), (hq, hkv, n)
        assert sk.query_blocks(cfg, 0) == 0


def test_multi_query_limits_rejected_on_host(libsekv):
    """n_q outside 1..SEKV_MAX_QUERY_TOKENS is rejected before any device work."""
    import ctypes
    import decode_attention_span_gb300 as sk
    cfg = sk.Config(1, 32, 8, 4, 64, 256, 32, 1, 64, 4.0)
    c = cfg.c()
    cache = sk.sekv.SekvLayerCache()
    for n in (0, -1, 65):
        st = libsekv.sekv_decode_step_multi(ctypes.byref(c), ctypes.byref(cache), None, n, None,
                                            None, ctypes.c_float(1.0), None, None, None, None,
                                            None, ctypes.c_size_t(0), None)
        assert st == -5, (n, st)  # SEKV_ERR_UNSUPPORTED
