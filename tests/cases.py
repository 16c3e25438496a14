"""Shared construction of parity cases: synthetic inputs -> oracle results.

Everything here runs on the CPU; expected values come from ``oracle`` only.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

import oracle
import synth
from oracle import layout
from synth import gen

TOL_ABS = 1e-2      # max abs error of attention outputs (bf16 inputs, fp32 accumulation)
TOL_REL = 5e-3      # relative L2 error of attention outputs
SCALE = 1.0 / math.sqrt(128.0)


@dataclasses.dataclass
class DecodeCase:
    wcfg: object
    tensors: dict          # ABI tensors (CPU)
    arrays: dict           # numpy copies for the oracle
    cache: object          # oracle LayerCache
    q: torch.Tensor        # bf16 [B][Hq][128]
    W: torch.Tensor        # f32 [Hkv][64][128]
    theta: np.ndarray      # f32 [Hq]
    E: list                # oracle expansion sets
    z: list                # oracle logits
    o: Optional[np.ndarray] = None
    lse: Optional[np.ndarray] = None


def thresholds(z, n_q_heads: int, frac: float, group: int, mode: str = "frac") -> np.ndarray:
    if mode == "none":
        return np.full(n_q_heads, np.inf, np.float32)
    if mode == "all":
        return np.full(n_q_heads, -np.inf, np.float32)
    p = gen.per_head_fraction(frac, group)
    th = []
    for h in range(n_q_heads):
        zz = np.concatenate([z[b][h] for b in range(len(z))])
        th.append(gen.pick_threshold(zz, p))
    return np.asarray(th, np.float32)


def decode_case(name: str, layer: int = 0, mode: str = "frac", seed: int = 7, run_oracle=True,
                **overrides) -> DecodeCase:
    w = synth.get_config(name, **overrides)
    d = gen.decode_cache(w, layer, device="cpu")
    a = gen.abi_to_numpy(d)
    cache = layout.unpack_layer(a, w.n_sink, w.n_recent)
    g = gen._gen(seed * 31 + layer)
    q = gen.query(g, w.batch, w.n_q_heads)
    W = gen.routing_weights(g, w.n_kv_heads)
    z = oracle.route_logits(q.float().numpy(), W.numpy(), cache)
    theta = thresholds(z, w.n_q_heads, w.expand_frac, w.group, mode)
    E, _ = oracle.route(q.float().numpy(), W.numpy(), cache, theta)
    case = DecodeCase(w, d, a, cache, q, W, theta, E, z)
    if run_oracle:
        case.o, case.lse = oracle.decode_attention(q.float().numpy(), cache, E, SCALE)
    return case


def compare_out(o_gpu: np.ndarray, o_ref: np.ndarray, what: str = ""):
    o_gpu = np.asarray(o_gpu, np.float64)
    err = float(np.abs(o_gpu - o_ref).max())
    rel = float(np.linalg.norm(o_gpu - o_ref) / max(np.linalg.norm(o_ref), 1e-30))
    assert np.all(np.isfinite(o_gpu)), f"{what}: non-finite output"
    assert err <= TOL_ABS and rel <= TOL_REL, f"{what}: max abs {err:.3e}, rel L2 {rel:.3e}"
    return err, rel


# ----------------------------------------------------------------------------
# full-size cases: every group routed, a stated sample of groups attended
# ----------------------------------------------------------------------------

def group_arrays(a: dict, b: int, c: int) -> dict:
    """ABI arrays of one (sequence, KV head) as a batch-1, one-KV-head layer
    (the record store is shared: record offsets stay valid)."""
    out = dict(a)
    out["n_spans"] = a["n_spans"][b:b + 1]
    out["body_len"] = a["body_len"][b:b + 1]
    for k in ("k_full", "v_full", "s_route", "k_sum", "v_sum", "rec_off", "rec_rank"):
        out[k] = a[k][b:b + 1, c:c + 1]
    return out


@dataclasses.dataclass
class SampledCase:
    wcfg: object
    tensors: dict          # ABI tensors (on `device`)
    q: torch.Tensor        # bf16 [B][Hq][128] (CPU)
    W: torch.Tensor        # f32 [Hkv][64][128] (CPU)
    theta: np.ndarray      # f32 [Hq]
    E: dict                # (b, c) -> oracle expansion set, every group
    o: dict                # (b, c) -> oracle output [G][128], sampled groups
    lse: dict              # (b, c) -> oracle lse [G], sampled groups


def sampled_case(name: str, layer: int = 0, sample=None, device="cpu", mode: str = "frac",
                 seed: int = 7, scale: float = SCALE, **overrides) -> SampledCase:
    """One layer of a workload at its stated shape.  The oracle routes every
    (sequence, KV head) group and attends the groups in ``sample`` (None: all
    of them), each as a one-group layer of its own."""
    w = synth.get_config(name, **overrides)
    d = gen.decode_cache(w, layer, device=device)
    a = gen.abi_to_numpy(d)
    g = gen._gen(seed * 31 + layer)
    q = gen.query(g, w.batch, w.n_q_heads)
    W = gen.routing_weights(g, w.n_kv_heads)
    G = w.group
    qn, Wn = q.float().numpy(), W.numpy()
    groups = [(b, c) for b in range(w.batch) for c in range(w.n_kv_heads)]
    sample = set(groups if sample is None else sample)
    sub, z = {}, {}
    for (b, c) in groups:
        sub[(b, c)] = layout.unpack_layer(group_arrays(a, b, c), w.n_sink, w.n_recent,
                                          records=(b, c) in sample)
        z[(b, c)] = oracle.route_logits(qn[b:b + 1, c * G:(c + 1) * G], Wn[c:c + 1],
                                        sub[(b, c)])[0]
    zz = [[z[(b, h // G)][h % G] for h in range(w.n_q_heads)] for b in range(w.batch)]
    theta = thresholds(zz, w.n_q_heads, w.expand_frac, G, mode)
    E, o, lse = {}, {}, {}
    for (b, c) in groups:
        th = theta[c * G:(c + 1) * G]
        Eg, _ = oracle.route(qn[b:b + 1, c * G:(c + 1) * G], Wn[c:c + 1], sub[(b, c)], th)
        E[(b, c)] = Eg[0][0]
        if (b, c) in sample:
            og, lg = oracle.decode_attention(qn[b:b + 1, c * G:(c + 1) * G], sub[(b, c)], Eg,
                                             scale)
            o[(b, c)], lse[(b, c)] = og[0], lg[0]
    return SampledCase(w, d, q, W, theta, E, o, lse)
