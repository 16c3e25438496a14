"""Reader and writer of the C-ABI byte layouts, written for the oracle alone.

TEST INFRASTRUCTURE ONLY.  This module restates, in numpy, the layouts that
``include/sekv.h`` specifies (one layer of the span cache and the packed
basis-record store) so that the oracle can read what the generator or the GPU
wrote and can hand its own results to the GPU stages.  It shares no code with
the product or with the generator.

bfloat16 arrays travel as uint16 bit patterns.
"""

from __future__ import annotations

from typing import Dict, List, Optional

import numpy as np

from .sekv_oracle import HEAD_DIM, ROUTE_DIM, LayerCache, SpanFactors, bf16_round


def _r4(r: int) -> int:
    return (r + 3) // 4 * 4


def _r8(r: int) -> int:
    return (r + 7) // 8 * 8


def record_size(b: int, rK: int, rV: int) -> int:
    """Bytes of one basis record (header, key part, U blocks, value part)."""
    if b <= 0:
        return 0
    return (16 + 8 * _r4(rK) + 256 * rK + 2 * b * _r8(rK) + 2 * b * _r8(rV)
            + 8 * _r4(rV) + 256 * rV)


def swizzle_vt(vt: np.ndarray) -> np.ndarray:
    """Chunk permutation of Vt rows (its own inverse): for row j, the 16-byte
    chunk c (columns 8c..8c+7) goes to chunk position c ^ (j & 7)."""
    r = vt.shape[0]
    out = np.empty_like(vt)
    for j in range(r):
        for c in range(16):
            p = c ^ (j & 7)
            out[j, 8 * p:8 * p + 8] = vt[j, 8 * c:8 * c + 8]
    return out


def u_swz(t: int, W: int) -> int:
    """Chunk permutation key of U row t (W sixteen-byte chunks per row): with g
    the largest power of two dividing W, bits of t above log2(8/g), below g."""
    g = W & -W
    s = 3 - ((g > 1) + (g > 2) + (g > 4))
    return (t >> s) & (g - 1)


def swizzle_u(u: np.ndarray) -> np.ndarray:
    """Chunk permutation of U rows (its own inverse): for token row t of a U
    block with W = u.shape[1] / 8 chunks per row, chunk c goes to chunk
    position c ^ u_swz(t, W)."""
    b, w8 = u.shape
    W = w8 // 8
    out = np.empty_like(u)
    for t in range(b):
        m = u_swz(t, W)
        for c in range(W):
            p = c ^ m
            out[t, 8 * p:8 * p + 8] = u[t, 8 * c:8 * c + 8]
    return out


def bf16_bits(x) -> np.ndarray:
    """uint16 patterns of values that are already bfloat16-representable."""
    x = np.asarray(x, np.float64)
    r = bf16_round(x)
    if not np.array_equal(r, x):
        raise ValueError("value is not a bfloat16 value")
    return (r.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def bits_bf16(u) -> np.ndarray:
    u = np.asarray(u, np.uint16)
    return (u.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


# ----------------------------------------------------------------------------
# one record
# ----------------------------------------------------------------------------

def pack_record(F: SpanFactors) -> bytes:
    b = F.UK.shape[0]
    rK, rV = F.sK.shape[0], F.sV.shape[0]
    out = bytearray(record_size(b, rK, rV))
    pos = 0

    def put(arr: np.ndarray, nbytes_padded: int):
        nonlocal pos
        raw = arr.tobytes()
        out[pos:pos + len(raw)] = raw
        pos += nbytes_padded

    put(np.array([b, rK, rV, 0], np.int32), 16)
    sk = np.zeros(_r4(rK), np.float32); sk[:rK] = F.sK
    gk = np.zeros(_r4(rK), np.float32); gk[:rK] = F.gK
    put(sk, 4 * _r4(rK)); put(gk, 4 * _r4(rK))
    put(swizzle_vt(bf16_bits(F.VtK).reshape(rK, HEAD_DIM)).reshape(-1), 256 * rK)
    uk = np.zeros((b, _r8(rK)), np.uint16); uk[:, :rK] = bf16_bits(F.UK)
    uv = np.zeros((b, _r8(rV)), np.uint16); uv[:, :rV] = bf16_bits(F.UV)
    put(swizzle_u(uk).reshape(-1), 2 * b * _r8(rK))
    put(swizzle_u(uv).reshape(-1), 2 * b * _r8(rV))
    sv = np.zeros(_r4(rV), np.float32); sv[:rV] = F.sV
    gv = np.zeros(_r4(rV), np.float32); gv[:rV] = F.gV
    put(sv, 4 * _r4(rV)); put(gv, 4 * _r4(rV))
    put(swizzle_vt(bf16_bits(F.VtV).reshape(rV, HEAD_DIM)).reshape(-1), 256 * rV)
    assert pos == len(out)
    return bytes(out)


def unpack_record(buf: np.ndarray, off: int, b_expected: Optional[int] = None) -> SpanFactors:
    """Parse one record starting at byte ``off`` of the uint8 array ``buf``."""
    hdr = buf[off:off + 16].view(np.int32)
    b, rK, rV = int(hdr[0]), int(hdr[1]), int(hdr[2])
    if b_expected is not None and b != b_expected:
        raise ValueError(f"record body {b} != span body {b_expected}")
    pos = off + 16

    def take(nbytes: int, nbytes_padded: int, dtype) -> np.ndarray:
        nonlocal pos
        a = buf[pos:pos + nbytes].view(dtype)
        pos += nbytes_padded
        return a

    sK = take(4 * rK, 4 * _r4(rK), np.float32).astype(np.float64)
    gK = take(4 * rK, 4 * _r4(rK), np.float32).astype(np.float64)
    VtK = swizzle_vt(bits_bf16(take(256 * rK, 256 * rK, np.uint16)).reshape(rK, HEAD_DIM))
    UK = bits_bf16(swizzle_u(take(2 * b * _r8(rK), 2 * b * _r8(rK), np.uint16)
                             .reshape(b, _r8(rK))))[:, :rK]
    UV = bits_bf16(swizzle_u(take(2 * b * _r8(rV), 2 * b * _r8(rV), np.uint16)
                             .reshape(b, _r8(rV))))[:, :rV]
    sV = take(4 * rV, 4 * _r4(rV), np.float32).astype(np.float64)
    gV = take(4 * rV, 4 * _r4(rV), np.float32).astype(np.float64)
    VtV = swizzle_vt(bits_bf16(take(256 * rV, 256 * rV, np.uint16)).reshape(rV, HEAD_DIM))
    return SpanFactors(UK=UK, sK=sK, gK=gK, VtK=VtK, UV=UV, sV=sV, gV=gV, VtV=VtV)


# ----------------------------------------------------------------------------
# one layer
# ----------------------------------------------------------------------------

def pack_layer(cache: LayerCache, max_spans: int) -> Dict[str, np.ndarray]:
    """ABI arrays of one layer from a logical cache (records packed densely,
    group by group, in span order)."""
    B, Hkv = cache.batch, cache.n_kv_heads
    cap = cache.n_sink + max_spans + cache.n_recent
    n_spans = np.array([cache.n_spans(b) for b in range(B)], np.int32)
    if n_spans.max(initial=0) > max_spans:
        raise ValueError("max_spans too small")
    body_len = np.zeros((B, max_spans), np.int32)
    k_full = np.zeros((B, Hkv, cap, HEAD_DIM), np.uint16)
    v_full = np.zeros_like(k_full)
    s_route = np.zeros((B, Hkv, max_spans, ROUTE_DIM), np.float32)
    k_sum = np.zeros((B, Hkv, max_spans, HEAD_DIM), np.uint16)
    v_sum = np.zeros_like(k_sum)
    rec_off = np.zeros((B, Hkv, max_spans), np.int64)
    rec_rank = np.zeros((B, Hkv, max_spans), np.int32)
    chunks: List[bytes] = []
    pos = 0
    for b in range(B):
        ns = n_spans[b]
        body_len[b, :ns] = cache.body_len[b]
        for c in range(Hkv):
            nf = cache.k_full[b][c].shape[0]
            k_full[b, c, :nf] = bf16_bits(cache.k_full[b][c])
            v_full[b, c, :nf] = bf16_bits(cache.v_full[b][c])
            s_route[b, c, :ns] = cache.s_route[b][c]
            k_sum[b, c, :ns] = bf16_bits(cache.k_sum[b][c])
            v_sum[b, c, :ns] = bf16_bits(cache.v_sum[b][c])
            for k in range(ns):
                F = cache.factors[b][c][k]
                rec_off[b, c, k] = pos
                if F is None:
                    continue
                raw = pack_record(F)
                rec_rank[b, c, k] = F.sK.shape[0] | (F.sV.shape[0] << 16)
                chunks.append(raw)
                pos += len(raw)
    store = np.frombuffer(b"".join(chunks) + b"\0" * 16, np.uint8).copy()
    return dict(n_spans=n_spans, body_len=body_len, k_full=k_full, v_full=v_full,
                s_route=s_route, k_sum=k_sum, v_sum=v_sum, rec_off=rec_off,
                rec_rank=rec_rank, store=store)


def unpack_layer(arrs: Dict[str, np.ndarray], n_sink: int, n_recent: int,
                 groups=None, records: bool = True) -> LayerCache:
    """Logical cache from ABI arrays.  ``groups``: optional set of (b, c) to
    decode fully; the others get empty per-head lists (for sampled checks).
    ``records=False`` leaves every span's factors as None (routing needs no
    basis records; it saves unpacking them).  An ``n_tail`` array in
    ``arrs`` gives each sequence's rows after the anchors (else n_recent)."""
    n_spans = np.asarray(arrs["n_spans"])
    n_tail = arrs.get("n_tail")
    B = n_spans.shape[0]
    Hkv = arrs["k_full"].shape[1]
    store = np.asarray(arrs["store"], np.uint8)
    out = LayerCache(n_sink=n_sink, n_recent=n_recent, body_len=[], k_full=[],
                     v_full=[], s_route=[], k_sum=[], v_sum=[], factors=[])
    for b in range(B):
        ns = int(n_spans[b])
        body = np.asarray(arrs["body_len"][b, :ns], np.int64)
        out.body_len.append(body)
        nf = n_sink + ns + (n_recent if n_tail is None else int(n_tail[b]))
        kf, vf, sr, ks, vs, fac = [], [], [], [], [], []
        for c in range(Hkv):
            if groups is not None and (b, c) not in groups:
                for lst in (kf, vf, sr, ks, vs, fac):
                    lst.append(None)
                continue
            kf.append(bits_bf16(arrs["k_full"][b, c, :nf]))
            vf.append(bits_bf16(arrs["v_full"][b, c, :nf]))
            sr.append(np.asarray(arrs["s_route"][b, c, :ns], np.float64))
            ks.append(bits_bf16(arrs["k_sum"][b, c, :ns]))
            vs.append(bits_bf16(arrs["v_sum"][b, c, :ns]))
            row: List[Optional[SpanFactors]] = []
            for k in range(ns):
                if body[k] <= 0 or not records:
                    row.append(None)
                    continue
                F = unpack_record(store, int(arrs["rec_off"][b, c, k]), int(body[k]))
                rr = int(arrs["rec_rank"][b, c, k])
                if (rr & 0xFFFF) != F.sK.shape[0] or (rr >> 16) != F.sV.shape[0]:
                    raise ValueError("rec_rank disagrees with the record header")
                row.append(F)
            fac.append(row)
        out.k_full.append(kf)
        out.v_full.append(vf)
        out.s_route.append(sr)
        out.k_sum.append(ks)
        out.v_sum.append(vs)
        out.factors.append(fac)
    return out
