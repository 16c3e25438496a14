"""Incremental maintenance of one layer's span cache during decode (test
infrastructure only, like the rest of ``oracle``).

The pages describe the cache built at prefill and the zoom-in during decode;
they do not say how the cache follows the tokens that decoding appends.
Reading taken here (from the pages' own definitions):

* [DE] lay explainer part 2 / [ZH] 两层记忆: the GPU keeps the very last part
  of the text at full resolution.  The newest token joins that recent window,
  and the oldest token of the window leaves it.
* [DE] Methodik 1 / [ZH] 方法论 1: a span is the run of tokens *between* two
  neighbouring anchors, and high-surprisal tokens are the boundaries.  The
  token leaving the window continues the segmentation walk with the rule of
  ``segment``: it opens a new span iff (H_t > tau and the open span's length
  >= len_min) or that length == len_max.
* A span can be built (routing summary, summary key/value, gated SVD basis:
  [DE] Methodik 2 / [ZH] 方法论 2) once the next anchor closes it.  Until it
  is built it stays at full resolution -- anchor and body -- with the open
  span and the recent window: the *tail* of the full-resolution rows.  Closed
  spans wait in the tail until a flush builds them (all at once), so the
  caller chooses how often the builds run; flushing after every append builds
  each span as soon as it closes.

Invariant (what the tests pin): after every append or flush, the maintained
cache of a prefix of length T equals ``build_layer`` of that prefix with the
recent window taken to start at the anchor of the first span not yet built
(``closed_build``): the batch walk over [n_sink, that anchor) makes exactly
the built spans, because the walk is online (no look-ahead) and the anchor
was itself a boundary.
"""

from __future__ import annotations

import dataclasses
from typing import List, Optional

import numpy as np

from .sekv_oracle import LayerCache, build_layer, build_span, segment


@dataclasses.dataclass
class MaintState:
    """One layer's maintained cache for a batch of sequences.

    ``caches[b]`` is a batch-1 ``LayerCache`` of the closed spans: its
    ``k_full``/``v_full`` rows are the sinks, the closed spans' anchors, then
    the tail (open span's anchor and body, then the recent window).
    ``s_open[b]`` is the open span's anchor position (None while the middle
    region is empty); ``pending[b]`` the lengths (anchor + body) of the closed
    spans not yet built, in order, at the head of the tail; ``tail_H[b]`` the
    surprisal of the tail's tokens; ``T[b]`` the sequence length.
    """
    T: List[int]
    caches: List[LayerCache]
    s_open: List[Optional[int]]
    pending: List[List[int]]
    tail_H: List[np.ndarray]
    n_sink: int
    n_recent: int
    tau: float
    len_min: int
    len_max: int
    rank_cap: int

    def n_tail(self, b: int) -> int:
        return self.caches[b].k_full[0][0].shape[0] - self.caches[b].n_sink - \
            self.caches[b].n_spans(0)


def open_anchor(H, n_sink: int, n_recent: int, tau: float, len_min: int, len_max: int):
    """Anchor position of the open (last) span of a prefix, or None when its
    middle region is empty."""
    starts, _ = segment(H, n_sink, n_recent, tau, len_min, len_max)
    return int(starts[-1]) if len(starts) else None


def closed_build(K, V, H, W_r, gates, *, n_sink: int, n_recent: int, tau: float,
                 len_min: int, len_max: int, rank_cap: int,
                 n_built=None) -> List[LayerCache]:
    """The reference form of a maintained cache: per sequence b, the batch
    build of the prefix whose recent window starts at the anchor of span
    n_built[b] (default: the open span, i.e. every closed span built), so
    that spans 0 .. n_built[b]-1 are built and everything from that anchor on
    is at full resolution.  K, V: [B][Hkv][T][128]; H: [B][T]; gates as
    ``build_layer``."""
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    B, _, T, _ = K.shape
    out = []
    for b in range(B):
        starts, _ = segment(H[b], n_sink, n_recent, tau, len_min, len_max)
        k = len(starts) - 1 if n_built is None else n_built[b]
        s = int(starts[k]) if 0 <= k < len(starts) else None
        nr = n_recent if s is None else T - s
        out.append(build_layer(K[b:b + 1], V[b:b + 1], np.asarray(H)[b:b + 1], W_r,
                               np.asarray(gates)[b:b + 1], n_sink=n_sink, n_recent=nr, tau=tau,
                               len_min=len_min, len_max=len_max, rank_cap=rank_cap))
    return out


def init_state(K, V, H, W_r, gates, *, n_sink: int, n_recent: int, tau: float,
               len_min: int, len_max: int, rank_cap: int) -> MaintState:
    """The state after the prefill of a prefix (T >= n_sink + n_recent): its
    closed build, by definition."""
    K = np.asarray(K, np.float64)
    H = np.asarray(H, np.float32)
    B, _, T, _ = K.shape
    if T < n_sink + n_recent:
        raise ValueError("prefix shorter than sinks + recent window")
    caches = closed_build(K, V, H, W_r, gates, n_sink=n_sink, n_recent=n_recent, tau=tau,
                          len_min=len_min, len_max=len_max, rank_cap=rank_cap)
    s_open, tail_H = [], []
    for b in range(B):
        s = open_anchor(H[b], n_sink, n_recent, tau, len_min, len_max)
        s_open.append(s)
        tail_H.append(H[b, (T - n_recent if s is None else s):].astype(np.float32))
    return MaintState(T=[T] * B, caches=caches, s_open=s_open, pending=[[] for _ in range(B)],
                      tail_H=tail_H, n_sink=n_sink,
                      n_recent=n_recent, tau=tau, len_min=len_min, len_max=len_max,
                      rank_cap=rank_cap)


def append_token(st: MaintState, k_new, v_new, h_new, W_r=None, gates=None,
                 build: bool = True) -> MaintState:
    """One decode step's maintenance: every sequence b appends its new token
    (k_new, v_new [B][Hkv][128], surprisal h_new [B]) to the tail; the token
    leaving its recent window continues the segmentation walk, and a span
    that this closes joins the pending spans.  With ``build`` the pending
    spans are built at once (``flush``, which then needs W_r and gates).
    Updates ``st`` in place and returns it."""
    k_new = np.asarray(k_new, np.float64)
    v_new = np.asarray(v_new, np.float64)
    tau32 = np.float32(st.tau)
    for b, cache in enumerate(st.caches):
        Hkv = len(cache.k_full[0])
        for c in range(Hkv):
            cache.k_full[0][c] = np.vstack([cache.k_full[0][c], k_new[b, c][None]])
            cache.v_full[0][c] = np.vstack([cache.v_full[0][c], v_new[b, c][None]])
        st.tail_H[b] = np.append(st.tail_H[b], np.float32(h_new[b]))
        t = st.T[b] - st.n_recent  # the token leaving the recent window
        st.T[b] += 1
        if t < st.n_sink:
            continue
        s = st.s_open[b]
        if s is None:
            st.s_open[b] = t  # the first middle token opens span 0
            continue
        n = t - s
        i_t = sum(st.pending[b]) + n  # token t's place in the tail
        if (st.tail_H[b][i_t] > tau32 and n >= st.len_min) or n == st.len_max:
            st.pending[b].append(n)  # the open span [s, t) is closed
            st.s_open[b] = t
    if build:
        flush(st, W_r, gates)
    return st


def flush(st: MaintState, W_r, gates) -> MaintState:
    """Builds every pending span, in order, from its rows in the tail
    (``build_span``, the prefill's per-span step, with the gates of its span
    ordinal); each keeps its anchor row, as anchor k, and its body rows leave
    full resolution.  Updates ``st`` in place and returns it."""
    for b, cache in enumerate(st.caches):
        Hkv = len(cache.k_full[0])
        for n in st.pending[b]:
            k = cache.n_spans(0)
            row0 = cache.n_sink + k  # the span's anchor row: it stays, as anchor k
            s = int(cache.anchors[0][-1]) + int(cache.body_len[0][-1]) + 1 if k else None
            cache.body_len[0] = np.append(cache.body_len[0], n - 1)
            cache.anchors[0] = np.append(cache.anchors[0], st.n_sink if s is None else s)
            for c in range(Hkv):
                Kt, Vt = cache.k_full[0][c], cache.v_full[0][c]
                s_row = np.zeros(64)
                k_row = np.zeros(Kt.shape[1])
                v_row = np.zeros(Vt.shape[1])
                F = None
                if n > 1:
                    s_row, k_row, v_row, F = build_span(
                        Kt[row0 + 1:row0 + n], Vt[row0 + 1:row0 + n], st.tail_H[b][1:n], W_r[c],
                        gates[b][c][0][k], gates[b][c][1][k], st.rank_cap)
                cache.s_route[0][c] = np.vstack([cache.s_route[0][c].reshape(-1, 64), s_row[None]])
                cache.k_sum[0][c] = np.vstack([cache.k_sum[0][c].reshape(-1, Kt.shape[1]),
                                               k_row[None]])
                cache.v_sum[0][c] = np.vstack([cache.v_sum[0][c].reshape(-1, Vt.shape[1]),
                                               v_row[None]])
                cache.factors[0][c].append(F)
                # the body rows leave full resolution; the anchor row stays
                cache.k_full[0][c] = np.vstack([Kt[:row0 + 1], Kt[row0 + n:]])
                cache.v_full[0][c] = np.vstack([Vt[:row0 + 1], Vt[row0 + n:]])
            st.tail_H[b] = st.tail_H[b][n:]
        st.pending[b] = []
    return st
