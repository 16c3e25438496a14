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
