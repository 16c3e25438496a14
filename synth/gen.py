"""Seeded generators (torch RNG on the requested device; CPU for small cases).

Recipes (stated once here; the design doc repeats them):

* Surprisal H_t ~ Gamma(2, 1), drawn as the sum of two unit exponentials.
* Span lengths: surprisal-threshold spans over i.i.d. surprisal have length
  min(len_min + G, len_max) with G geometric (failures before the first
  success) of success probability p = P(H > tau) = (1 + tau) exp(-tau); the
  last span is cut at the end of the middle region.  ``planted_surprisal``
  draws H *given* such lengths: tokens that must not open a span are drawn
  from Gamma(2,1) conditioned on H <= tau, tokens that must open one from the
  law conditioned on H > tau, all others unconditioned.  This is the same
  joint law as i.i.d. Gamma(2,1) surprisal, and it tells the generator where
  the spans are so that key/value blocks can follow them.
* Every H is kept at least ``margin`` (1e-3) from tau, in float32.
* Keys/values per block (a span including its anchor, the sink block, the
  recent block): A (n x rho) ~ N(0,1), B (rho x 128) ~ N(0, 1/rho), plus
  N(0, 0.05) noise (0.05 is the variance), rounded to bfloat16.
* Queries ~ N(0, 1) rounded to bfloat16; routing weights ~ N(0, 1/128) fp32.
* Soft rank gates for a span of rank budget rho: g_j = sigmoid(2 (rho - j - 0.5)).
"""

from __future__ import annotations

import math
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np
import torch

from .configs import WorkloadConfig

HEAD_DIM = 128
ROUTE_DIM = 64


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _uniform(gen: torch.Generator, n: int, device="cpu") -> torch.Tensor:
    u = torch.rand(n, generator=gen, device=device, dtype=torch.float64)
    return u.clamp_(1e-300, 1.0)


# ----------------------------------------------------------------------------
# surprisal and span lengths
# ----------------------------------------------------------------------------

def gamma2_survival(x: np.ndarray) -> np.ndarray:
    return (1.0 + x) * np.exp(-x)


def _gamma2_inverse(target_survival: np.ndarray) -> np.ndarray:
    """x with (1+x) e^{-x} = target (vectorised bisection in float64)."""
    lo = np.zeros_like(target_survival)
    hi = np.full_like(target_survival, 80.0)
    for _ in range(80):
        mid = 0.5 * (lo + hi)
        above = gamma2_survival(mid) > target_survival
        lo = np.where(above, mid, lo)
        hi = np.where(above, hi, mid)
    return 0.5 * (lo + hi)


def span_lengths(gen: torch.Generator, n_tokens: int, tau: float, len_min: int,
                 len_max: int) -> np.ndarray:
    """Lengths (anchor included) of consecutive spans covering n_tokens."""
    if n_tokens <= 0:
        return np.zeros(0, np.int64)
    p = float(gamma2_survival(np.float64(tau)))
    est = int(n_tokens / (len_min + (1 - p) / p)) + 64
    out: List[np.ndarray] = []
    total = 0
    while total < n_tokens:
        u = _uniform(gen, est).numpy()
        G = np.floor(np.log(u) / math.log1p(-p)).astype(np.int64)
        L = np.minimum(len_min + G, len_max)
        out.append(L)
        total += int(L.sum())
    L = np.concatenate(out)
    cs = np.cumsum(L)
    k = int(np.searchsorted(cs, n_tokens))  # first span reaching the end
    L = L[:k + 1].copy()
    L[k] -= int(cs[k] - n_tokens)
    assert L.sum() == n_tokens and L.min() >= 1
    return L


def planted_surprisal(gen: torch.Generator, T: int, n_sink: int, n_recent: int,
                      lens: np.ndarray, tau: float, len_min: int, len_max: int,
                      margin: float = 1e-3) -> np.ndarray:
    """float32 surprisal [T] whose threshold segmentation gives ``lens``."""
    m0, m1 = n_sink, T - n_recent
    assert int(np.sum(lens)) == m1 - m0
    H = (-torch.log(_uniform(gen, T)) - torch.log(_uniform(gen, T))).numpy()
    starts = m0 + np.concatenate([[0], np.cumsum(lens)[:-1]]).astype(np.int64)
    span_of = np.repeat(np.arange(len(lens)), lens)
    offset = np.arange(m0, m1) - starts[span_of]
    pos = np.arange(m0, m1)
    # must not open a span: offset >= len_min (inside a span, past the minimum)
    le_mask = offset >= len_min
    # must open a span: anchors of spans 1.., unless the previous one hit len_max
    ge_pos = starts[1:][lens[:-1] < len_max]
    S_tau = float(gamma2_survival(np.float64(tau)))
    n_le = int(le_mask.sum())
    if n_le:
        u = _uniform(gen, n_le).numpy()
        # survival in (S_tau, 1]  <=>  H in [0, tau)
        H[pos[le_mask]] = _gamma2_inverse(S_tau + u * (1.0 - S_tau))
    if len(ge_pos):
        u = _uniform(gen, len(ge_pos)).numpy()
        H[ge_pos] = _gamma2_inverse(u * S_tau)
    H32 = H.astype(np.float32)
    t32 = np.float32(tau)
    lo, hi = np.float32(tau - margin), np.float32(tau + margin)
    while lo > t32 - np.float32(margin):
        lo = np.nextafter(lo, np.float32(-np.inf))
    while hi < t32 + np.float32(margin):
        hi = np.nextafter(hi, np.float32(np.inf))
    near = np.abs(H32.astype(np.float64) - float(t32)) < margin
    H32[near & (H32 > t32)] = hi
    H32[near & (H32 <= t32)] = lo
    return H32


# ----------------------------------------------------------------------------
# keys / values / queries / weights / gates
# ----------------------------------------------------------------------------

def lowrank_tokens(gen: torch.Generator, block_lens: np.ndarray, block_rank: np.ndarray,
                   noise_var: float, device="cpu", chunk: int = 8192) -> torch.Tensor:
    """[sum(block_lens), 128] bfloat16 rows, low rank + noise per block."""
    nb = len(block_lens)
    rmax = int(block_rank.max())
    T = int(np.sum(block_lens))
    Bm = torch.randn(nb, rmax, HEAD_DIM, generator=gen, device=device)
    rk = torch.as_tensor(block_rank, device=device, dtype=torch.float32)
    col = torch.arange(rmax, device=device)
    colmask = (col[None, :] < rk[:, None]).float()               # nb x rmax
    Bm = Bm * (colmask / rk.sqrt()[:, None])[:, :, None]
    A = torch.randn(T, rmax, generator=gen, device=device)
    noise = torch.randn(T, HEAD_DIM, generator=gen, device=device) * math.sqrt(noise_var)
    blk = torch.as_tensor(np.repeat(np.arange(nb), block_lens), device=device)
    out = torch.empty(T, HEAD_DIM, device=device, dtype=torch.bfloat16)
    for s in range(0, T, chunk):
        e = min(T, s + chunk)
        Bt = Bm[blk[s:e]]                                       # n x rmax x 128
        rows = torch.bmm(A[s:e, None, :], Bt)[:, 0, :] + noise[s:e]
        out[s:e] = rows.to(torch.bfloat16)
    return out


def rank_budget_gates(rho: np.ndarray, n_comp: int) -> np.ndarray:
    """g_j = sigmoid(2 (rho - j - 0.5)), j < n_comp, for each budget rho."""
    j = np.arange(n_comp)[None, :]
    x = 2.0 * (np.asarray(rho, np.float64)[:, None] - j - 0.5)
    return (1.0 / (1.0 + np.exp(-x))).astype(np.float32)


def query(gen: torch.Generator, batch: int, n_q_heads: int, device="cpu") -> torch.Tensor:
    return torch.randn(batch, n_q_heads, HEAD_DIM, generator=gen,
                       device=device).to(torch.bfloat16)


def routing_weights(gen: torch.Generator, n_kv_heads: int, device="cpu") -> torch.Tensor:
    return torch.randn(n_kv_heads, ROUTE_DIM, HEAD_DIM, generator=gen,
                       device=device) / math.sqrt(HEAD_DIM)


# ----------------------------------------------------------------------------
# thresholds
# ----------------------------------------------------------------------------

def per_head_fraction(union_frac: float, group: int) -> float:
    """Per-head expansion rate whose union over ``group`` independent heads
    has rate ``union_frac``."""
    return 1.0 - (1.0 - union_frac) ** (1.0 / group)


def pick_threshold(z: np.ndarray, frac: float, margin: float = 1e-3) -> np.float32:
    """float32 threshold with about ``frac`` of ``z`` above it and every value
    at least ``margin`` away from it."""
    zs = np.sort(np.asarray(z, np.float64))
    n = len(zs)
    if n == 0:
        return np.float32(0.0)
    target = int(round((1.0 - frac) * n))

    def ok(theta32) -> bool:
        return bool(np.all(np.abs(zs - float(theta32)) >= margin))

    for d in range(0, n + 1):
        for i in (target - d, target + d):
            if i < 0 or i > n:
                continue
            if i == 0:
                th = np.float32(zs[0] - 4 * margin)
            elif i == n:
                th = np.float32(zs[-1] + 4 * margin)
            else:
                if zs[i] - zs[i - 1] <= 2 * margin + 1e-6:
                    continue
                th = np.float32(0.5 * (zs[i] + zs[i - 1]))
            if ok(th):
                return th
    raise RuntimeError("no threshold with the requested margin")


# ----------------------------------------------------------------------------
# prefill-build inputs (tokens, surprisal, gates) of one layer
# ----------------------------------------------------------------------------

def _round_up(x: int, m: int) -> int:
    return (x + m - 1) // m * m


def sequence_spans(cfg: WorkloadConfig, b: int) -> np.ndarray:
    """Planted span lengths of sequence b (shared by every layer and head)."""
    gen = _gen(cfg.seed * 1000003 + 17 * b + 1)
    return span_lengths(gen, cfg.ctx - cfg.n_sink - cfg.n_recent, cfg.tau,
                        cfg.len_min, cfg.len_max)


def max_spans_for(cfg: WorkloadConfig) -> int:
    n = max(len(sequence_spans(cfg, b)) for b in range(cfg.batch))
    return _round_up(max(n, 1), 64)


def build_inputs(cfg: WorkloadConfig, layer: int, device="cpu",
                 max_spans: Optional[int] = None) -> Dict[str, object]:
    """K, V [B][Hkv][T][128] bf16, H [B][T] f32, W_r, gates, q of one layer.

    gates: [B][Hkv][2][max_spans][rank_cap] float32 (index 0 keys, 1 values),
    indexed by span ordinal; ``lens`` are the planted span lengths.
    """
    B, Hkv, T = cfg.batch, cfg.n_kv_heads, cfg.ctx
    lens = [sequence_spans(cfg, b) for b in range(B)]
    if max_spans is None:
        max_spans = _round_up(max(max(len(l) for l in lens), 1), 64)
    H = np.zeros((B, T), np.float32)
    for b in range(B):
        H[b] = planted_surprisal(_gen(cfg.seed * 7919 + b + 3), T, cfg.n_sink,
                                 cfg.n_recent, lens[b], cfg.tau, cfg.len_min,
                                 cfg.len_max)
    gen = _gen(cfg.seed * 104729 + layer * 31 + 5, device)
    K = torch.empty(B, Hkv, T, HEAD_DIM, dtype=torch.bfloat16, device=device)
    V = torch.empty_like(K)
    rgen = _gen(cfg.seed * 65537 + layer * 13 + 7)
    for b in range(B):
        blocks = np.concatenate([[cfg.n_sink], lens[b], [cfg.n_recent]]).astype(np.int64)
        keep = blocks > 0
        blocks = blocks[keep]
        for c in range(Hkv):
            for X in (K, V):
                if cfg.true_rank:
                    rk = np.full(len(blocks), cfg.true_rank, np.int64)
                else:
                    rk = torch.randint(cfg.rank_lo, cfg.rank_cap + 1, (len(blocks),),
                                       generator=rgen).numpy()
                X[b, c] = lowrank_tokens(gen, blocks, rk, 0.05, device)
    gates = np.zeros((B, Hkv, 2, max_spans, cfg.rank_cap), np.float32)
    if cfg.unit_gates:
        gates[:] = 1.0
    else:
        for b in range(B):
            n = len(lens[b])
            rho = torch.randint(cfg.rank_lo, cfg.rank_cap + 1, (Hkv * 2 * n,),
                                generator=rgen).numpy()
            gates[b, :, :, :n] = rank_budget_gates(rho, cfg.rank_cap).reshape(
                Hkv, 2, n, cfg.rank_cap)
    qgen = _gen(cfg.seed * 999331 + layer * 7 + 11, device)
    return dict(K=K, V=V, H=H, W_r=routing_weights(qgen, Hkv, device),
                q=query(qgen, B, cfg.n_q_heads, device), gates=gates, lens=lens,
                max_spans=max_spans)


# ----------------------------------------------------------------------------
# synthetic decode caches, packed straight into the C-ABI layout
# ----------------------------------------------------------------------------

def record_size(b, rK, rV):
    """Basis record bytes (C-ABI layout); works on ints and integer arrays."""
    def r4(r):
        return (r + 3) // 4 * 4

    def r8(r):
        return (r + 7) // 8 * 8
    size = (16 + 8 * r4(rK) + 256 * rK + 2 * b * r8(rK) + 2 * b * r8(rV)
            + 8 * r4(rV) + 256 * rV)
    if isinstance(b, (int, np.integer)):
        return int(size) if b > 0 else 0
    return size * (b > 0)


def decode_cache(cfg: WorkloadConfig, layer: int, device="cpu",
                 max_spans: Optional[int] = None) -> Dict[str, torch.Tensor]:
    """One layer's span cache in the C-ABI layout, drawn directly.

    Span lengths are the planted lengths (the same for every layer and head).
    Full-resolution rows ~ N(0,1); summary key/value of a span with body b ~
    N(0, 1/b) (the spread of a mean of b unit-variance rows); routing
    summaries are uniform random unit vectors.  Basis records hold N(0,1)
    matrices U, Vt and singular values scaled so that reconstructed rows have
    unit variance, with gated rank r = min(rho, b), rho ~ U{rank_lo..rank_cap}
    drawn separately for keys and values; the matrices are not orthonormal
    (the decode step never relies on orthonormality).
    """
    B, Hkv = cfg.batch, cfg.n_kv_heads
    lens = [sequence_spans(cfg, b) for b in range(B)]
    if max_spans is None:
        max_spans = _round_up(max(max(len(l) for l in lens), 1), 64)
    cap = cfg.n_sink + max_spans + cfg.n_recent
    gen = _gen(cfg.seed * 15485863 + layer * 101 + 13, device)
    n_spans = torch.tensor([len(l) for l in lens], dtype=torch.int32)
    body = torch.zeros(B, max_spans, dtype=torch.int64)
    for b in range(B):
        body[b, :len(lens[b])] = torch.as_tensor(lens[b] - 1)
    k_full = torch.zeros(B, Hkv, cap, HEAD_DIM, dtype=torch.bfloat16, device=device)
    v_full = torch.zeros_like(k_full)
    for b in range(B):
        nf = cfg.n_sink + len(lens[b]) + cfg.n_recent
        k_full[b, :, :nf] = torch.randn(Hkv, nf, HEAD_DIM, generator=gen, device=device).to(torch.bfloat16)
        v_full[b, :, :nf] = torch.randn(Hkv, nf, HEAD_DIM, generator=gen, device=device).to(torch.bfloat16)
    bodyd = body.to(device)
    valid = (bodyd > 0)[:, None, :, None]                       # B,1,S,1
    inv = torch.where(bodyd > 0, 1.0 / bodyd.clamp(min=1).double().sqrt(),
                      torch.zeros((), dtype=torch.float64, device=device)).float()
    k_sum = (torch.randn(B, Hkv, max_spans, HEAD_DIM, generator=gen, device=device)
             * inv[:, None, :, None]).to(torch.bfloat16)
    v_sum = (torch.randn(B, Hkv, max_spans, HEAD_DIM, generator=gen, device=device)
             * inv[:, None, :, None]).to(torch.bfloat16)
    s = torch.randn(B, Hkv, max_spans, ROUTE_DIM, generator=gen, device=device)
    s = s / s.norm(dim=-1, keepdim=True)
    s_route = torch.where(valid, s, torch.zeros((), device=device)).float().contiguous()

    # ranks: rho ~ U{rank_lo..rank_cap}, r = min(rho, body)
    rho = torch.randint(cfg.rank_lo, cfg.rank_cap + 1, (B, Hkv, max_spans, 2),
                        generator=gen, device=device)
    bb = bodyd[:, None, :].expand(B, Hkv, max_spans)
    rK = torch.minimum(rho[..., 0], bb) * (bb > 0)
    rV = torch.minimum(rho[..., 1], bb) * (bb > 0)
    sizes = record_size(bb, rK, rV)
    flat = sizes.reshape(-1)
    off = torch.cumsum(flat, 0) - flat
    total = int(flat.sum().item()) + 16
    store = torch.empty(total, dtype=torch.uint8, device=device)
    store.view(torch.bfloat16).normal_(generator=gen)
    f32 = store.view(torch.float32)
    i32 = store.view(torch.int32)
    rec = torch.nonzero(flat > 0).squeeze(1)
    o = off[rec]
    b_r, rK_r, rV_r = bb.reshape(-1)[rec], rK.reshape(-1)[rec], rV.reshape(-1)[rec]
    rhoK, rhoV = rho[..., 0].reshape(-1)[rec], rho[..., 1].reshape(-1)[rec]
    hw = o // 4
    i32[hw] = b_r.int()
    i32[hw + 1] = rK_r.int()
    i32[hw + 2] = rV_r.int()
    i32[hw + 3] = 0

    def r4(r):
        return (r + 3) // 4 * 4

    def r8(r):
        return (r + 7) // 8 * 8

    def put_sigma_gate(base_bytes, r, rho_, scale_row):
        # sigma_j = c * exp(-j / (2 r)), g_j = sigmoid(2 (rho - j - 0.5)); zero pad to r4
        n4 = r4(r)
        idx_rec = torch.repeat_interleave(torch.arange(len(r), device=device), n4)
        start = torch.cumsum(n4, 0) - n4
        j = torch.arange(int(n4.sum().item()), device=device) - start[idx_rec]
        rr = r[idx_rec].double()
        live = j < r[idx_rec]
        sig = torch.exp(-j.double() / (2 * rr.clamp(min=1))) * scale_row[idx_rec]
        gate = torch.sigmoid(2.0 * (rho_[idx_rec].double() - j.double() - 0.5))
        w = base_bytes[idx_rec] // 4 + j
        f32[w] = torch.where(live, sig, torch.zeros_like(sig)).float()
        f32[w + n4[idx_rec]] = torch.where(live, gate, torch.zeros_like(gate)).float()

    def scale_for(r, b_):
        # U, Vt entries ~ N(0,1): an element of row i of U diag(sigma g) Vt has
        # variance sum_j sigma_j^2 g_j^2; aim for about one.
        jj = torch.arange(cfg.rank_cap, device=device, dtype=torch.float64)
        prof = torch.exp(-jj[None, :] / (r.double().clamp(min=1)[:, None]))
        prof = (prof * (jj[None, :] < r[:, None])).sum(1)
        return 1.0 / torch.sqrt(prof.clamp(min=1e-30))

    put_sigma_gate(o + 16, rK_r, rhoK, scale_for(rK_r, b_r))
    uk_off = o + 16 + 8 * r4(rK_r) + 256 * rK_r
    uv_off = uk_off + 2 * b_r * r8(rK_r)
    vpart = uv_off + 2 * b_r * r8(rV_r)
    put_sigma_gate(vpart, rV_r, rhoV, scale_for(rV_r, b_r))
    bf = store.view(torch.bfloat16)

    def zero_u_padding(base_bytes, b_, r_):
        # U rows hold r8(r) columns; columns r.. must be zero
        pad = r8(r_) - r_
        sel = (pad > 0) & (b_ > 0)
        base_bytes, b_, r_, pad = base_bytes[sel], b_[sel], r_[sel], pad[sel]
        n_el = b_ * pad
        if n_el.numel() == 0 or int(n_el.sum().item()) == 0:
            return
        rec_i = torch.repeat_interleave(torch.arange(len(n_el), device=device), n_el)
        start = torch.cumsum(n_el, 0) - n_el
        e = torch.arange(int(n_el.sum().item()), device=device) - start[rec_i]
        row, colp = e // pad[rec_i], e % pad[rec_i]
        # the padding columns are in the row's last 16-byte chunk, which the
        # record layout stores at chunk position (W - 1) ^ u_swz(row, W)
        W = r8(r_)[rec_i] // 8
        g = W & -W
        sh = 3 - ((g > 1).long() + (g > 2).long() + (g > 4).long())
        key = (row >> sh) & (g - 1)
        col = r_[rec_i] + colp
        phys = (((col >> 3) ^ key) << 3) | (col & 7)
        idx = base_bytes[rec_i] // 2 + row * r8(r_)[rec_i] + phys
        bf[idx] = 0

    zero_u_padding(uk_off, b_r, rK_r)
    zero_u_padding(uv_off, b_r, rV_r)
    rec_off = off.reshape(B, Hkv, max_spans).contiguous()
    rec_rank = (rK | (rV << 16)).int().contiguous()
    return dict(n_spans=n_spans.to(device), body_len=body.int().to(device).contiguous(),
                k_full=k_full, v_full=v_full, s_route=s_route, k_sum=k_sum.contiguous(),
                v_sum=v_sum.contiguous(), rec_off=rec_off, rec_rank=rec_rank, store=store,
                max_spans=max_spans, lens=lens)


def full_kv_cache(cfg: WorkloadConfig, layer: int, T: int, device="cpu",
                  max_spans: int = 64) -> Dict[str, torch.Tensor]:
    """One layer of a full-KV cache in the C-ABI layout: no spans, every one of
    the T context tokens a full-resolution row.

    The decode step over such a cache (configured with n_sink = 0 and
    n_recent = T) is plain softmax attention over all T tokens, the full-KV
    decode that SeKV is compared with.  Rows ~ N(0,1) in bf16, like the
    full-resolution rows of ``decode_cache``; the span arrays are zero and the
    basis store is a zero stub.
    """
    B, Hkv = cfg.batch, cfg.n_kv_heads
    cap = max_spans + T
    gen = _gen(cfg.seed * 15485863 + layer * 101 + 17, device)
    k_full = torch.zeros(B, Hkv, cap, HEAD_DIM, dtype=torch.bfloat16, device=device)
    v_full = torch.zeros_like(k_full)
    for b in range(B):
        k_full[b, :, :T] = torch.randn(Hkv, T, HEAD_DIM, generator=gen, device=device).to(torch.bfloat16)
        v_full[b, :, :T] = torch.randn(Hkv, T, HEAD_DIM, generator=gen, device=device).to(torch.bfloat16)
    z = dict(device=device)
    return dict(n_spans=torch.zeros(B, dtype=torch.int32, **z),
                body_len=torch.zeros(B, max_spans, dtype=torch.int32, **z),
                k_full=k_full, v_full=v_full,
                s_route=torch.zeros(B, Hkv, max_spans, ROUTE_DIM, dtype=torch.float32, **z),
                k_sum=torch.zeros(B, Hkv, max_spans, HEAD_DIM, dtype=torch.bfloat16, **z),
                v_sum=torch.zeros(B, Hkv, max_spans, HEAD_DIM, dtype=torch.bfloat16, **z),
                rec_off=torch.zeros(B, Hkv, max_spans, dtype=torch.int64, **z),
                rec_rank=torch.zeros(B, Hkv, max_spans, dtype=torch.int32, **z),
                store=torch.zeros(256, dtype=torch.uint8, **z), max_spans=max_spans)


def abi_to_numpy(d: Dict[str, object]) -> Dict[str, np.ndarray]:
    """numpy copies of ABI tensors (bfloat16 as uint16 bit patterns)."""
    out = {}
    for k, v in d.items():
        if isinstance(v, torch.Tensor):
            t = v.detach().cpu()
            if t.dtype == torch.bfloat16:
                out[k] = t.view(torch.int16).numpy().view(np.uint16)
            else:
                out[k] = t.numpy()
        else:
            out[k] = v
    return out
