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
