"""fp64 reference arithmetic for SeKV's span cache (test infrastructure only).

Every function restates one step that the SeKV pages describe, in plain numpy
float64, with no blocking, fusion or reordering beyond the definition.  Where
the pages leave a step open the reading taken is stated in the docstring
("Reading: ...").  Page citations use the short names defined in
``oracle/__init__.py`` ([DE], [ZH], [EN]).

Stored precisions (the pages fix none; the C-ABI does): keys, values, summary
keys/values and SVD factors are bfloat16; surprisal, routing summaries,
singular values, gates, routing weights and thresholds are float32.  The
oracle reads stored values exactly (widened to float64) and rounds only where
it produces a stored value.
"""

from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence, Tuple

import numpy as np

HEAD_DIM = 128
ROUTE_DIM = 64


# ----------------------------------------------------------------------------
# Rounding helpers (storage formats, not part of the method)
# ----------------------------------------------------------------------------

def bf16_round(x) -> np.ndarray:
    """Round to the nearest bfloat16 value (ties to even), returned as float64.

    The value is first rounded to float32 (ties to even, numpy's cast), then
    the low 16 bits of the float32 pattern are rounded away with ties to even.
    Inputs must be finite.
    """
    x32 = np.ascontiguousarray(np.asarray(x, dtype=np.float64).astype(np.float32))
    bits = x32.view(np.uint32).astype(np.uint64)
    lsb = (bits >> np.uint64(16)) & np.uint64(1)
    bits = (bits + np.uint64(0x7FFF) + lsb) & np.uint64(0xFFFF0000)
    return bits.astype(np.uint32).view(np.float32).astype(np.float64)


def f32_round(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


# ----------------------------------------------------------------------------
# Step 1: regions and entropy-guided segmentation
# ----------------------------------------------------------------------------

def regions(T: int, n_sink: int, n_recent: int) -> Tuple[int, int]:
    """Return the middle region [m0, m1) in which spans live.

    [DE] lay explainer part 2 / [ZH] 两层记忆: the GPU keeps the very first and
    the very last part of the context at full resolution.  Reading: these are
    ``n_sink`` sink tokens [0, n_sink) and ``n_recent`` recent tokens
    [T - n_recent, T); spans only cover the tokens in between.
    """
    if T < n_sink + n_recent:
        raise ValueError("context shorter than sinks + recent window")
    return n_sink, T - n_recent


def segment(H, n_sink: int, n_recent: int, tau: float,
            len_min: int, len_max: int) -> Tuple[np.ndarray, np.ndarray]:
    """Entropy-guided span segmentation; returns (anchor positions, lengths).

    [DE] Methodik 1 / [ZH] 方法论 1: tokens whose surprisal is high are span
    boundaries; each boundary token is an anchor kept at full resolution; a
    span is the run of tokens between two neighbouring anchors.

    Readings (the pages give no clamps): the first middle token opens span 0;
    walking t = s+1 ... m1-1 with ``s`` the current span's anchor and
    ``n = t - s`` its length so far, token t opens a new span iff
    (H_t > tau and n >= len_min) or n == len_max.  The comparison is a strict
    float32 ``>``.  The last span ends at m1 and may be shorter than len_min.
    A span's length counts its anchor; its body is the len-1 tokens after it.
    """
    H = np.asarray(H, dtype=np.float32)
    tau32 = np.float32(tau)
    m0, m1 = regions(H.shape[0], n_sink, n_recent)
    if m1 <= m0:
        return np.zeros(0, np.int64), np.zeros(0, np.int64)
    starts = [m0]
    s = m0
    for t in range(m0 + 1, m1):
        n = t - s
        if (H[t] > tau32 and n >= len_min) or n == len_max:
            starts.append(t)
            s = t
    starts_a = np.asarray(starts, dtype=np.int64)
    ends = np.append(starts_a[1:], m1)
    return starts_a, ends - starts_a


# ----------------------------------------------------------------------------
# Step 2: the two per-span representations
# ----------------------------------------------------------------------------

def routing_summary(K_body, H_body, W_r) -> Optional[np.ndarray]:
    """Routing summary s_S of one span (float64, unit L2 norm).

    [DE] Methodik 2 / [ZH] 方法论 2: the GPU copy of a span is a normalised,
    surprisal-weighted average of projected key vectors.
    Reading: u = sum_i H_i * (W_r k_i) over the body tokens, s = u / ||u||.
    Dividing by sum H first would change nothing after the normalisation.
    An empty body has no summary (returns None); u == 0 gives the zero vector.
    """
    K_body = np.asarray(K_body, dtype=np.float64)
    if K_body.shape[0] == 0:
        return None
    W = np.asarray(W_r, dtype=np.float64)
    Hb = np.asarray(H_body, dtype=np.float64)
    u = np.zeros(W.shape[0])
    for i in range(K_body.shape[0]):
        u += Hb[i] * (W @ K_body[i])
    nrm = np.sqrt(np.sum(u * u))
    return u / nrm if nrm > 0 else u


def attention_summary(K_body, V_body) -> Tuple[np.ndarray, np.ndarray]:
    """Summary key and value that an unexpanded span contributes to attention.

    [DE] Methodik 3 / [ZH] 方法论 3: unexpanded spans enter the mixed-resolution
    attention as coarse summaries with a size correction.  Reading: the
    summary key/value are the uniform means of the body's keys/values in head
    space (the 64-d routing summary cannot serve as a 128-d key); the size
    correction (``decode_attention``) adds ln|S| to its logit.  Returned
    unrounded (float64); storage rounds them to bfloat16.
    """
    K_body = np.asarray(K_body, dtype=np.float64)
    V_body = np.asarray(V_body, dtype=np.float64)
    return K_body.mean(axis=0), V_body.mean(axis=0)


@dataclasses.dataclass
class SVDResult:
    U: np.ndarray       # b x r
    sigma: np.ndarray   # r
    gate: np.ndarray    # r
    Vt: np.ndarray      # r x 128
    rank: int
    sigma_all: np.ndarray  # every singular value of M (for checks)


def span_svd(M, gates, rank_cap: int) -> SVDResult:
    """Truncated, gated SVD basis of one span body M (b x 128), unrounded.

    [DE] Methodik 2 / [ZH] 方法论 2: the CPU copy of a span is a low-rank SVD
    basis; a predictor gives every singular component a soft gate, which sets
    the span's rank budget r_S.  The predictor is trained and out of scope:
    the gates arrive as an input.

    Readings: R = min(rank_cap, b) components are candidates; r_S is the
    length of the longest prefix (components in descending sigma) whose gates
    exceed 0.5; reconstruction uses sigma_j * g_j.  Signs: each kept pair
    (u_j, v_j) is flipped so that the largest-magnitude entry of v_j is
    positive (lowest index on ties).
    """
    M = np.asarray(M, dtype=np.float64)
    b = M.shape[0]
    U, s, Vt = np.linalg.svd(M, full_matrices=False)
    R = min(rank_cap, b)
    g = np.asarray(gates, dtype=np.float64)[:R]
    r = 0
    while r < R and g[r] > 0.5:
        r += 1
    U = U[:, :r].copy()
    Vt = Vt[:r].copy()
    for j in range(r):
        idx = int(np.argmax(np.abs(Vt[j])))
        if Vt[j, idx] < 0:
            Vt[j] = -Vt[j]
            U[:, j] = -U[:, j]
    return SVDResult(U=U, sigma=s[:r].copy(), gate=g[:r].copy(), Vt=Vt,
                     rank=r, sigma_all=s)


@dataclasses.dataclass
class SpanFactors:
    """Stored factors of one span (values exactly as stored, in float64)."""
    UK: np.ndarray
    sK: np.ndarray
    gK: np.ndarray
    VtK: np.ndarray
    UV: np.ndarray
    sV: np.ndarray
    gV: np.ndarray
    VtV: np.ndarray

    @property
    def body(self) -> int:
        return self.UK.shape[0]


def reconstruct(U, sigma, gate, Vt) -> np.ndarray:
    """Token-level reconstruction U diag(sigma * g) V^T of one span.

    [DE] Methodik 3 / [ZH] 方法论 3: an expanded span's basis is loaded and its
    token-level K/V are rebuilt before they join attention.
    """
    U = np.asarray(U, np.float64)
    w = np.asarray(sigma, np.float64) * np.asarray(gate, np.float64)
    return U @ np.diag(w) @ np.asarray(Vt, np.float64)


# ----------------------------------------------------------------------------
# The cache of one layer, in logical form
# ----------------------------------------------------------------------------

@dataclasses.dataclass
class LayerCache:
    """Logical contents of one layer's span cache (all values as stored).

    Per sequence b: ``body_len[b]`` (n_spans[b] ints).  Per (b, kv head c):
    ``k_full[b][c]``/``v_full[b][c]`` rows = sinks, then one anchor per span
    in span order, then the recent window; ``s_route[b][c]`` (n_spans x 64,
    zero rows for empty bodies); ``k_sum``/``v_sum`` (n_spans x 128);
    ``factors[b][c][k]`` (SpanFactors, or None for an empty body).
    """
    n_sink: int
    n_recent: int
    body_len: List[np.ndarray]
    k_full: List[List[np.ndarray]]
    v_full: List[List[np.ndarray]]
    s_route: List[List[np.ndarray]]
    k_sum: List[List[np.ndarray]]
    v_sum: List[List[np.ndarray]]
    factors: List[List[List[Optional[SpanFactors]]]]
    anchors: Optional[List[np.ndarray]] = None

    @property
    def batch(self) -> int:
        return len(self.body_len)

    @property
    def n_kv_heads(self) -> int:
        return len(self.k_full[0])

    def n_spans(self, b: int) -> int:
        return int(len(self.body_len[b]))


def build_span(Kb, Vb, Hb, W_r_c, gates_k, gates_v, rank_cap: int):
    """Stored representations of one span with a non-empty body: (routing
    summary, summary key, summary value, SpanFactors), each rounded to its
    storage format.

    [DE] Methodik 2 / [ZH] 方法论 2: the GPU copy (routing summary) and the CPU
    copy (gated SVD basis) of the span, plus the summary key/value that an
    unexpanded span contributes to attention ([DE] Methodik 3).
    """
    s_row = f32_round(routing_summary(Kb, Hb, W_r_c))
    km, vm = attention_summary(Kb, Vb)
    fk = span_svd(Kb, gates_k, rank_cap)
    fv = span_svd(Vb, gates_v, rank_cap)
    F = SpanFactors(UK=bf16_round(fk.U), sK=f32_round(fk.sigma), gK=f32_round(fk.gate),
                    VtK=bf16_round(fk.Vt), UV=bf16_round(fv.U), sV=f32_round(fv.sigma),
                    gV=f32_round(fv.gate), VtV=bf16_round(fv.Vt))
    return s_row, bf16_round(km), bf16_round(vm), F


def build_layer(K, V, H, W_r, gates, *, n_sink: int, n_recent: int, tau: float,
                len_min: int, len_max: int, rank_cap: int) -> LayerCache:
    """Prefill cache build of one layer: segmentation, summaries, SVD bases.

    K, V: [B][Hkv][T][128] (bfloat16 values); H: [B][T] float32 surprisal
    ([DE]/[ZH] Methodik 1: H_t = -log p(x_t | x_<t) from the prefill pass; an
    input here); W_r: [Hkv][64][128] float32; gates: [B][Hkv][2][n][rank_cap]
    float32 indexed by span ordinal (index 0 = keys, 1 = values).
    """
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    B, Hkv, T, _ = K.shape
    out = LayerCache(n_sink=n_sink, n_recent=n_recent, body_len=[], k_full=[],
                     v_full=[], s_route=[], k_sum=[], v_sum=[], factors=[],
                     anchors=[])
    for b in range(B):
        starts, lens = segment(H[b], n_sink, n_recent, tau, len_min, len_max)
        body = lens - 1
        out.body_len.append(body.astype(np.int64))
        out.anchors.append(starts)
        m0, m1 = regions(T, n_sink, n_recent)
        full_idx = np.concatenate([np.arange(0, n_sink), starts,
                                   np.arange(m1, T)]).astype(np.int64)
        kf, vf, sr, ks, vs, fac = [], [], [], [], [], []
        for c in range(Hkv):
            kf.append(K[b, c, full_idx])
            vf.append(V[b, c, full_idx])
            s_rows = np.zeros((len(starts), ROUTE_DIM))
            k_rows = np.zeros((len(starts), HEAD_DIM))
            v_rows = np.zeros((len(starts), HEAD_DIM))
            f_row: List[Optional[SpanFactors]] = []
            for k, (a, n) in enumerate(zip(starts, lens)):
                lo, hi = int(a) + 1, int(a) + int(n)
                if hi <= lo:
                    f_row.append(None)
                    continue
                s_rows[k], k_rows[k], v_rows[k], F = build_span(
                    K[b, c, lo:hi], V[b, c, lo:hi], H[b][lo:hi], W_r[c],
                    gates[b][c][0][k], gates[b][c][1][k], rank_cap)
                f_row.append(F)
            sr.append(s_rows)
            ks.append(k_rows)
            vs.append(v_rows)
            fac.append(f_row)
        out.k_full.append(kf)
        out.v_full.append(vf)
        out.s_route.append(sr)
        out.k_sum.append(ks)
        out.v_sum.append(vs)
        out.factors.append(fac)
    return out


# ----------------------------------------------------------------------------
# Step 3: zoom-in routing
# ----------------------------------------------------------------------------

def route_logits(q, W_r, cache: LayerCache) -> List[np.ndarray]:
    """Gate logits z[b][h] (n_spans values) of every query head.

    [DE] Methodik 3 / [ZH] 方法论 3: the query is projected into the routing
    space of the summaries and a sigmoid gate gives each span's relevance.
    Readings: the same W_r (64 x 128, one per KV head) projects queries and
    keys; query head h uses the W_r of its KV head c = h // (Hq / Hkv); the
    gate is sigmoid(y . s_S) with no temperature or bias, so comparing the
    probability with sigmoid(theta) is comparing the logit z = y . s_S with a
    threshold theta kept in logit space.
    """
    q = np.asarray(q, np.float64)
    B, Hq, _ = q.shape
    Hkv = cache.n_kv_heads
    G = Hq // Hkv
    z = []
    for b in range(B):
        zb = []
        for h in range(Hq):
            c = h // G
            y = np.asarray(W_r[c], np.float64) @ q[b, h]
            zb.append(np.asarray(cache.s_route[b][c], np.float64) @ y)
        z.append(zb)
    return z


def route(q, W_r, cache: LayerCache, theta) -> Tuple[List[List[np.ndarray]], list]:
    """Expansion sets E[b][c] (ascending span indices) and the logits.

    [DE] Methodik 3 / [ZH] 方法论 3: a learned per-head, per-layer threshold
    decides whether a span is expanded.  Readings: head h expands S iff
    z_{h,S} > theta_h (strict); a span's basis is per KV head, so KV head c
    expands the union over its query heads; spans with an empty body are
    never expanded.
    """
    z = route_logits(q, W_r, cache)
    B = len(z)
    Hq = len(z[0])
    Hkv = cache.n_kv_heads
    G = Hq // Hkv
    theta = np.asarray(theta, np.float64)
    E = []
    for b in range(B):
        Eb = []
        nonempty = cache.body_len[b] > 0
        for c in range(Hkv):
            hit = np.zeros(cache.n_spans(b), dtype=bool)
            for h in range(c * G, (c + 1) * G):
                hit |= z[b][h] > theta[h]
            Eb.append(np.flatnonzero(hit & nonempty).astype(np.int64))
        E.append(Eb)
    return E, z


# ----------------------------------------------------------------------------
# Step 4: mixed-resolution attention
# ----------------------------------------------------------------------------

def _softmax_out(logits: np.ndarray, values: np.ndarray) -> Tuple[np.ndarray, float]:
    m = np.max(logits)
    e = np.exp(logits - m)
    ssum = np.sum(e)
    return (e @ values) / ssum, float(m + np.log(ssum))


def decode_attention(q, cache: LayerCache, expanded, scale: float):
    """Mixed-resolution decode attention of one layer; returns (o, lse).

    [DE] Methodik 3 / [ZH] 方法论 3: anchors (and, per the lay explainers,
    sinks and recent tokens) contribute their full K/V; an unexpanded span
    contributes its summary with a size correction; an expanded span
    contributes its reconstructed token-level K/V pairs.

    Written out explicitly: for query head h of KV head c the entries are
      full-res rows i:          logit  q.k_i * scale,           value v_i
      unexpanded span, |S|>=1:  logit  q.kbar_S * scale + ln|S|, value vbar_S
      expanded span, body i:    logit  q.khat_i * scale,        value vhat_i
    with khat = U_K diag(sigma_K g_K) Vt_K (likewise vhat), followed by an
    explicit max-subtracted softmax.  lse = max + ln(sum exp(l - max)).
    o: [B][Hq][128] float64, lse: [B][Hq] float64.
    """
    q = np.asarray(q, np.float64)
    B, Hq, _ = q.shape
    Hkv = cache.n_kv_heads
    G = Hq // Hkv
    o = np.zeros((B, Hq, HEAD_DIM))
    lse = np.zeros((B, Hq))
    for b in range(B):
        for c in range(Hkv):
            keys = [np.asarray(cache.k_full[b][c], np.float64)]
            vals = [np.asarray(cache.v_full[b][c], np.float64)]
            bias = [np.zeros(keys[0].shape[0])]
            exp_set = set(int(k) for k in expanded[b][c])
            body = cache.body_len[b]
            unexp = [k for k in range(len(body)) if body[k] > 0 and k not in exp_set]
            if unexp:
                idx = np.asarray(unexp)
                keys.append(np.asarray(cache.k_sum[b][c], np.float64)[idx])
                vals.append(np.asarray(cache.v_sum[b][c], np.float64)[idx])
                bias.append(np.log(body[idx].astype(np.float64)))
            for k in sorted(exp_set):
                F = cache.factors[b][c][k]
                keys.append(reconstruct(F.UK, F.sK, F.gK, F.VtK))
                vals.append(reconstruct(F.UV, F.sV, F.gV, F.VtV))
                bias.append(np.zeros(F.UK.shape[0]))
            Kall = np.concatenate(keys, axis=0)
            Vall = np.concatenate(vals, axis=0)
            Ball = np.concatenate(bias)
            for h in range(c * G, (c + 1) * G):
                logits = (Kall @ q[b, h]) * scale + Ball
                o[b, h], lse[b, h] = _softmax_out(logits, Vall)
    return o, lse


def full_attention(q, K, V, scale: float):
    """Textbook softmax attention of each query head over all T tokens.

    The full-KV attention that SeKV approximates (the teacher the pages train
    against).  q: [B][Hq][128]; K, V: [B][Hkv][T][128].
    """
    q = np.asarray(q, np.float64)
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    B, Hq, _ = q.shape
    Hkv = K.shape[1]
    G = Hq // Hkv
    o = np.zeros((B, Hq, HEAD_DIM))
    lse = np.zeros((B, Hq))
    for b in range(B):
        for h in range(Hq):
            c = h // G
            o[b, h], lse[b, h] = _softmax_out((K[b, c] @ q[b, h]) * scale, V[b, c])
    return o, lse
