"""Thin ctypes binding of libsekv (argument marshalling only).

Every computation runs in the CUDA kernels behind the C ABI in
``include/sekv.h``; this module checks tensor placement and dtypes, passes raw
pointers and the current CUDA stream, and raises on a non-OK status.  There is
no CPU fallback: if the library is missing, every call raises.
"""

from __future__ import annotations

import ctypes
import dataclasses
import math
import os
from typing import Dict, Optional, Tuple

import torch

from . import build as _build

_c_i32, _c_f32, _c_vp, _c_sz, _c_i64 = (ctypes.c_int32, ctypes.c_float, ctypes.c_void_p,
                                        ctypes.c_size_t, ctypes.c_int64)

SEKV_CALL_ROUTE, SEKV_CALL_FETCH, SEKV_CALL_DECODE, SEKV_CALL_BUILD = 0, 1, 2, 3
FLAG_OVERLAP_PREVIOUS = 1
FLAG_SHORT_WAITS = 2
STATUS = {0: "SEKV_OK", -1: "SEKV_ERR_INVALID", -2: "SEKV_ERR_CAPACITY", -3: "SEKV_ERR_CUDA",
          -4: "SEKV_ERR_TIMEOUT", -5: "SEKV_ERR_UNSUPPORTED", -6: "SEKV_ERR_DEVICE"}

# every symbol include/sekv.h declares
EXPORTS = ("sekv_record_size", "sekv_workspace_size", "sekv_workspace_init",
           "sekv_workspace_status", "sekv_route", "sekv_fetch_bases", "sekv_decode_attention",
           "sekv_decode_step", "sekv_decode_step_multi", "sekv_query_blocks",
           "sekv_decode_step_noalloc",
           "sekv_noalloc_status",
           "sekv_build_spans",
           "sekv_fetch_bases_copy", "sekv_basis_cache_bytes", "sekv_basis_cache_init",
           "sekv_fetch_bases_cached", "sekv_build_flops", "sekv_maint_state_size",
           "sekv_maint_init", "sekv_append_token", "sekv_maint_flush",
           "sekv_status_string", "sekv_last_launch_count")


class SekvError(RuntimeError):
    def __init__(self, call: str, status: int):
        super().__init__(f"{call} returned {STATUS.get(status, status)}")
        self.status = status


class SekvConfig(ctypes.Structure):
    _fields_ = [("batch", _c_i32), ("n_q_heads", _c_i32), ("n_kv_heads", _c_i32),
                ("head_dim", _c_i32), ("route_dim", _c_i32), ("n_sink", _c_i32),
                ("n_recent", _c_i32), ("max_spans", _c_i32), ("rank_cap", _c_i32),
                ("len_min", _c_i32), ("len_max", _c_i32), ("tau", _c_f32), ("flags", _c_i32)]


class SekvCacheOut(ctypes.Structure):
    _fields_ = [("n_spans", _c_vp), ("body_len", _c_vp), ("k_full", _c_vp), ("v_full", _c_vp),
                ("s_route", _c_vp), ("k_sum", _c_vp), ("v_sum", _c_vp), ("rec_off", _c_vp),
                ("rec_rank", _c_vp), ("store", _c_vp), ("store_capacity", _c_i64)]


class SekvLayerCache(ctypes.Structure):
    _fields_ = [("n_spans", _c_vp), ("body_len", _c_vp), ("k_full", _c_vp), ("v_full", _c_vp),
                ("s_route", _c_vp), ("k_sum", _c_vp), ("v_sum", _c_vp), ("rec_off", _c_vp),
                ("rec_rank", _c_vp), ("store", _c_vp), ("store_on_host", _c_i32),
                ("n_tail", _c_vp)]


_LIB = None


def library_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """The loaded libsekv; raises if it has not been built."""
    global _LIB
    if _LIB is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"libsekv is not built ({path} missing); run "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(path)
        L.sekv_record_size.restype = _c_i64
        L.sekv_record_size.argtypes = [_c_i32, _c_i32, _c_i32]
        L.sekv_workspace_size.restype = _c_sz
        L.sekv_workspace_size.argtypes = [ctypes.POINTER(SekvConfig), _c_i32, _c_i64]
        L.sekv_workspace_init.restype = _c_i32
        L.sekv_workspace_init.argtypes = [_c_vp, _c_sz, _c_vp]
        L.sekv_workspace_status.restype = _c_i32
        L.sekv_workspace_status.argtypes = [_c_vp, _c_vp, ctypes.POINTER(_c_i32),
                                            ctypes.POINTER(_c_i32)]
        L.sekv_route.restype = _c_i32
        L.sekv_route.argtypes = [ctypes.POINTER(SekvConfig), ctypes.POINTER(SekvLayerCache),
                                 _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_sz, _c_vp]
        L.sekv_fetch_bases.restype = _c_i32
        L.sekv_fetch_bases.argtypes = [ctypes.POINTER(SekvConfig), ctypes.POINTER(SekvLayerCache),
                                       _c_vp, _c_vp, _c_vp, _c_i64, _c_vp, _c_vp, _c_sz, _c_vp]
        L.sekv_query_blocks.restype = _c_i32
        L.sekv_query_blocks.argtypes = [ctypes.POINTER(SekvConfig), _c_i32]
        L.sekv_build_flops.restype = _c_i32
        L.sekv_build_flops.argtypes = [_c_vp, _c_vp, ctypes.POINTER(_c_i64)]
        L.sekv_maint_state_size.restype = _c_sz
        L.sekv_maint_state_size.argtypes = [ctypes.POINTER(SekvConfig)]
        L.sekv_maint_init.restype = _c_i32
        L.sekv_maint_init.argtypes = [ctypes.POINTER(SekvConfig), _c_i64, _c_vp, _c_vp, _c_vp,
                                      ctypes.POINTER(SekvCacheOut), _c_vp, _c_vp, _c_sz, _c_vp,
                                      _c_sz, _c_vp]
        L.sekv_append_token.restype = _c_i32
        L.sekv_append_token.argtypes = [ctypes.POINTER(SekvConfig), _c_vp, _c_vp, _c_vp,
                                        ctypes.POINTER(SekvCacheOut), _c_vp, _c_vp, _c_sz, _c_vp,
                                        _c_sz, _c_vp]
        L.sekv_maint_flush.restype = _c_i32
        L.sekv_maint_flush.argtypes = [ctypes.POINTER(SekvConfig), _c_vp, _c_vp,
                                       ctypes.POINTER(SekvCacheOut), _c_vp, _c_vp, _c_sz, _c_vp,
                                       _c_sz, _c_vp]
        L.sekv_basis_cache_bytes.restype = _c_sz
        L.sekv_basis_cache_bytes.argtypes = [ctypes.POINTER(SekvConfig), _c_i32]
        L.sekv_basis_cache_init.restype = _c_i32
        L.sekv_basis_cache_init.argtypes = [ctypes.POINTER(SekvConfig), _c_vp, _c_i32, _c_vp]
        L.sekv_fetch_bases_cached.restype = _c_i32
        L.sekv_fetch_bases_cached.argtypes = [ctypes.POINTER(SekvConfig),
                                              ctypes.POINTER(SekvLayerCache), _c_vp, _c_vp, _c_vp,
                                              _c_i64, _c_vp, _c_i32, _c_i32, _c_vp, _c_vp, _c_vp,
                                              _c_vp, _c_sz, _c_vp]
        L.sekv_fetch_bases_copy.restype = _c_i32
        L.sekv_fetch_bases_copy.argtypes = [ctypes.POINTER(SekvConfig),
                                            ctypes.POINTER(SekvLayerCache), _c_vp, _c_vp, _c_vp,
                                            _c_vp, _c_i64, _c_vp, _c_vp, ctypes.POINTER(_c_i32),
                                            _c_vp, _c_vp]
        L.sekv_decode_attention.restype = _c_i32
        L.sekv_decode_attention.argtypes = [ctypes.POINTER(SekvConfig),
                                            ctypes.POINTER(SekvLayerCache), _c_vp, _c_vp, _c_vp,
                                            _c_vp, _c_vp, _c_f32, _c_vp, _c_vp, _c_vp, _c_sz,
                                            _c_vp]
        L.sekv_decode_step.restype = _c_i32
        L.sekv_decode_step.argtypes = [ctypes.POINTER(SekvConfig), ctypes.POINTER(SekvLayerCache),
                                       _c_vp, _c_vp, _c_vp, _c_f32, _c_vp, _c_vp, _c_vp, _c_vp,
                                       _c_vp, _c_sz, _c_vp]
        L.sekv_decode_step_multi.restype = _c_i32
        L.sekv_decode_step_multi.argtypes = [ctypes.POINTER(SekvConfig),
                                             ctypes.POINTER(SekvLayerCache), _c_vp, _c_i32,
                                             _c_vp, _c_vp, _c_f32, _c_vp, _c_vp, _c_vp, _c_vp,
                                             _c_vp, _c_sz, _c_vp]
        L.sekv_decode_step_noalloc.restype = _c_i32
        L.sekv_decode_step_noalloc.argtypes = [ctypes.POINTER(SekvConfig),
                                               ctypes.POINTER(SekvLayerCache), _c_vp, _c_vp,
                                               _c_vp, _c_f32, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp]
        L.sekv_noalloc_status.restype = _c_i32
        L.sekv_noalloc_status.argtypes = [_c_vp, ctypes.POINTER(_c_i32), ctypes.POINTER(_c_i32)]
        L.sekv_build_spans.restype = _c_i32
        L.sekv_build_spans.argtypes = [ctypes.POINTER(SekvConfig), _c_i64, _c_vp, _c_vp, _c_vp,
                                       _c_vp, _c_vp, ctypes.POINTER(SekvCacheOut), _c_vp, _c_sz,
                                       _c_vp]
        L.sekv_status_string.restype = ctypes.c_char_p
        L.sekv_status_string.argtypes = [_c_i32]
        L.sekv_last_launch_count.restype = _c_i32
        L.sekv_last_launch_count.argtypes = []
        _LIB = L
    return _LIB


def _check(call: str, st: int):
    if st != 0:
        raise SekvError(call, st)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need(t: torch.Tensor, name: str, dtype, cuda: bool = True):
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if cuda and not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")


# ----------------------------------------------------------------------------
# configuration, cache, workspace
# ----------------------------------------------------------------------------

@dataclasses.dataclass
class Config:
    batch: int
    n_q_heads: int
    n_kv_heads: int
    n_sink: int
    n_recent: int
    max_spans: int
    rank_cap: int = 32
    len_min: int = 4
    len_max: int = 256
    tau: float = 5.2
    head_dim: int = 128
    route_dim: int = 64
    flags: int = 0

    def c(self) -> SekvConfig:
        return SekvConfig(self.batch, self.n_q_heads, self.n_kv_heads, self.head_dim,
                          self.route_dim, self.n_sink, self.n_recent, self.max_spans,
                          self.rank_cap, self.len_min, self.len_max, float(self.tau),
                          self.flags)


CACHE_FIELDS = ("n_spans", "body_len", "k_full", "v_full", "s_route", "k_sum", "v_sum",
                "rec_off", "rec_rank", "store")


class LayerCache:
    """One layer of the span cache as torch tensors in the C-ABI layout."""

    def __init__(self, tensors: Dict[str, torch.Tensor], store_on_host: bool = False):
        self.t = {k: tensors[k] for k in CACHE_FIELDS if k in tensors}
        self.store_on_host = store_on_host
        for k, dt in (("n_spans", torch.int32), ("body_len", torch.int32),
                      ("k_full", torch.bfloat16), ("v_full", torch.bfloat16),
                      ("s_route", torch.float32), ("k_sum", torch.bfloat16),
                      ("v_sum", torch.bfloat16), ("rec_off", torch.int64),
                      ("rec_rank", torch.int32)):
            _need(self.t[k], k, dt)
        st = self.t["store"]
        _need(st, "store", torch.uint8, cuda=not store_on_host)
        if store_on_host and not st.is_pinned():
            raise ValueError("store: host tier must be pinned memory")
        n_tail = tensors.get("n_tail")
        if n_tail is not None:
            _need(n_tail, "n_tail", torch.int32)
            self.t["n_tail"] = n_tail
        self._c = SekvLayerCache(*[_ptr(self.t[k]) for k in CACHE_FIELDS], int(store_on_host),
                                 _ptr(n_tail))

    @property
    def c(self) -> SekvLayerCache:
        return self._c


class Workspace:
    """Caller-owned scratch of sekv_workspace_size bytes, zeroed once."""

    def __init__(self, cfg: Config, device=None, which: int = SEKV_CALL_DECODE, ctx_len: int = 0):
        c = cfg.c()
        n = int(lib().sekv_workspace_size(ctypes.byref(c), which, ctx_len))
        if n == 0:
            raise SekvError("sekv_workspace_size", -1)
        self.nbytes = n
        self.buf = torch.empty(n, dtype=torch.uint8, device=device or "cuda")
        _check("sekv_workspace_init", lib().sekv_workspace_init(_ptr(self.buf), n, _stream()))

    def ptr(self):
        return _ptr(self.buf)

    def status(self) -> Tuple[int, int]:
        """Synchronise; return (device code, detail) and clear them."""
        code, detail = _c_i32(0), _c_i32(0)
        lib().sekv_workspace_status(self.ptr(), _stream(), ctypes.byref(code), ctypes.byref(detail))
        return code.value, detail.value

    def raise_on_error(self):
        code, detail = self.status()
        if code != 0:
            raise RuntimeError(f"libsekv device status {code} (detail {detail})")


def record_size(body: int, rank_k: int, rank_v: int) -> int:
    return int(lib().sekv_record_size(body, rank_k, rank_v))


def last_launch_count() -> int:
    return int(lib().sekv_last_launch_count())


# ----------------------------------------------------------------------------
# calls
# ----------------------------------------------------------------------------

def route(cfg: Config, cache: LayerCache, q, W_r, theta, ws: Workspace, want_z: bool = False,
          expanded=None, n_expanded=None, stream=None):
    _need(q, "q", torch.bfloat16); _need(W_r, "W_r", torch.float32)
    _need(theta, "theta", torch.float32)
    dev = q.device
    NG = cfg.batch * cfg.n_kv_heads
    if expanded is None:
        expanded = torch.empty(NG * cfg.max_spans, dtype=torch.int32, device=dev)
    if n_expanded is None:
        n_expanded = torch.empty(NG, dtype=torch.int32, device=dev)
    z = (torch.zeros(cfg.batch * cfg.n_q_heads * cfg.max_spans, dtype=torch.float32, device=dev)
         if want_z else None)
    c = cfg.c()
    _check("sekv_route", lib().sekv_route(ctypes.byref(c), ctypes.byref(cache.c), _ptr(q),
                                          _ptr(W_r), _ptr(theta), _ptr(expanded),
                                          _ptr(n_expanded), _ptr(z), ws.ptr(), ws.nbytes,
                                          _stream(stream)))
    return expanded, n_expanded, z


def decode_attention(cfg: Config, cache: LayerCache, q, expanded, n_expanded, scale: float,
                     ws: Workspace, staging=None, staged_off=None, out=None, lse=None,
                     stream=None):
    _need(q, "q", torch.bfloat16); _need(expanded, "expanded", torch.int32)
    _need(n_expanded, "n_expanded", torch.int32)
    dev = q.device
    if out is None:
        out = torch.empty(cfg.batch, cfg.n_q_heads, 128, dtype=torch.float32, device=dev)
    if lse is None:
        lse = torch.empty(cfg.batch, cfg.n_q_heads, dtype=torch.float32, device=dev)
    c = cfg.c()
    _check("sekv_decode_attention",
           lib().sekv_decode_attention(ctypes.byref(c), ctypes.byref(cache.c), _ptr(q),
                                       _ptr(expanded), _ptr(n_expanded), _ptr(staging),
                                       _ptr(staged_off), float(scale), _ptr(out), _ptr(lse),
                                       ws.ptr(), ws.nbytes, _stream(stream)))
    return out, lse


def decode_step(cfg: Config, cache: LayerCache, q, W_r, theta, scale: float, ws: Workspace,
                out=None, lse=None, want_list: bool = False, stream=None):
    _need(q, "q", torch.bfloat16); _need(W_r, "W_r", torch.float32)
    _need(theta, "theta", torch.float32)
    dev = q.device
    if out is None:
        out = torch.empty(cfg.batch, cfg.n_q_heads, 128, dtype=torch.float32, device=dev)
    if lse is None:
        lse = torch.empty(cfg.batch, cfg.n_q_heads, dtype=torch.float32, device=dev)
    NG = cfg.batch * cfg.n_kv_heads
    expanded = n_expanded = None
    if want_list:
        expanded = torch.zeros(NG * cfg.max_spans, dtype=torch.int32, device=dev)
        n_expanded = torch.zeros(NG, dtype=torch.int32, device=dev)
    c = cfg.c()
    _check("sekv_decode_step",
           lib().sekv_decode_step(ctypes.byref(c), ctypes.byref(cache.c), _ptr(q), _ptr(W_r),
                                  _ptr(theta), float(scale), _ptr(out), _ptr(lse),
                                  _ptr(expanded), _ptr(n_expanded), ws.ptr(), ws.nbytes,
                                  _stream(stream)))
    return out, lse, expanded, n_expanded


def query_blocks(cfg: Config, n_q: int) -> int:
    """sekv_query_blocks: launches (blocks of query tokens) of the multi-query step."""
    c = cfg.c()
    return int(lib().sekv_query_blocks(ctypes.byref(c), int(n_q)))


def decode_step_multi(cfg: Config, cache: LayerCache, q, W_r, theta, scale: float,
                      ws: Workspace, out=None, lse=None, want_list: bool = False, stream=None):
    """sekv_decode_step_multi: q [B][n_q][Hq][128] bf16, n_q query tokens per
    sequence over the same cache; returns out [B][n_q][Hq][128], lse, and, when
    want_list, per block of tokens the union expansion lists
    [blocks][B*Hkv][max_spans] and counts [blocks][B*Hkv]."""
    _need(q, "q", torch.bfloat16); _need(W_r, "W_r", torch.float32)
    _need(theta, "theta", torch.float32)
    B, n_q = q.shape[0], q.shape[1]
    dev = q.device
    if out is None:
        out = torch.empty(B, n_q, cfg.n_q_heads, 128, dtype=torch.float32, device=dev)
    if lse is None:
        lse = torch.empty(B, n_q, cfg.n_q_heads, dtype=torch.float32, device=dev)
    NG = cfg.batch * cfg.n_kv_heads
    expanded = n_expanded = None
    if want_list:
        nb = max(query_blocks(cfg, n_q), 1)
        expanded = torch.zeros(nb * NG * cfg.max_spans, dtype=torch.int32, device=dev)
        n_expanded = torch.zeros(nb * NG, dtype=torch.int32, device=dev)
    c = cfg.c()
    _check("sekv_decode_step_multi",
           lib().sekv_decode_step_multi(ctypes.byref(c), ctypes.byref(cache.c), _ptr(q), n_q,
                                        _ptr(W_r), _ptr(theta), float(scale), _ptr(out),
                                        _ptr(lse), _ptr(expanded), _ptr(n_expanded), ws.ptr(),
                                        ws.nbytes, _stream(stream)))
    return out, lse, expanded, n_expanded


def decode_step_noalloc(cfg: Config, cache: LayerCache, q, W_r, theta, scale: float, out=None,
                        lse=None, want_list: bool = False, stream=None):
    """sekv_decode_step_noalloc: the decode step with no workspace argument.

    For callers that cannot allocate device memory: the library's fixed 8 MiB
    device scratch array stands in for the workspace (shapes needing more
    raise SekvError with SEKV_ERR_CAPACITY).  Calls share that array, so they
    must not overlap on the GPU.  The outputs here are allocated by torch only
    when the caller passes none.
    """
    _need(q, "q", torch.bfloat16); _need(W_r, "W_r", torch.float32)
    _need(theta, "theta", torch.float32)
    dev = q.device
    if out is None:
        out = torch.empty(cfg.batch, cfg.n_q_heads, 128, dtype=torch.float32, device=dev)
    if lse is None:
        lse = torch.empty(cfg.batch, cfg.n_q_heads, dtype=torch.float32, device=dev)
    NG = cfg.batch * cfg.n_kv_heads
    expanded = n_expanded = None
    if want_list:
        expanded = torch.zeros(NG * cfg.max_spans, dtype=torch.int32, device=dev)
        n_expanded = torch.zeros(NG, dtype=torch.int32, device=dev)
    c = cfg.c()
    _check("sekv_decode_step_noalloc",
           lib().sekv_decode_step_noalloc(ctypes.byref(c), ctypes.byref(cache.c), _ptr(q),
                                          _ptr(W_r), _ptr(theta), float(scale), _ptr(out),
                                          _ptr(lse), _ptr(expanded), _ptr(n_expanded),
                                          _stream(stream)))
    return out, lse, expanded, n_expanded


def noalloc_status(stream=None):
    """(code, detail) of the no-alloc scratch array's status word on the
    current device (sekv_noalloc_status): synchronises, reads and clears it."""
    code, detail = _c_i32(0), _c_i32(0)
    lib().sekv_noalloc_status(_stream(stream), ctypes.byref(code), ctypes.byref(detail))
    return code.value, detail.value


def fetch_bases(cfg: Config, cache: LayerCache, expanded, n_expanded, staging, per_group: int,
                staged_off, ws: Workspace, stream=None):
    _need(staging, "staging", torch.uint8); _need(staged_off, "staged_off", torch.int64)
    c = cfg.c()
    _check("sekv_fetch_bases",
           lib().sekv_fetch_bases(ctypes.byref(c), ctypes.byref(cache.c), _ptr(expanded),
                                  _ptr(n_expanded), _ptr(staging), int(per_group),
                                  _ptr(staged_off), ws.ptr(), ws.nbytes, _stream(stream)))
    return staging, staged_off


def fetch_bases_copy(cfg: Config, cache: LayerCache, expanded_host, n_expanded_host,
                     rec_off_host, staging, per_group: int, staged_off_host, staged_off,
                     done_event, copy_stream) -> int:
    """sekv_fetch_bases_copy: the host-driven fetch (one cudaMemcpyAsync per
    run of adjacent records on `copy_stream`, then `done_event` recorded).
    The lists and record offsets are host tensors; returns the copies issued."""
    _need(expanded_host, "expanded_host", torch.int32, cuda=False)
    _need(n_expanded_host, "n_expanded_host", torch.int32, cuda=False)
    _need(rec_off_host, "rec_off_host", torch.int64, cuda=False)
    _need(staged_off_host, "staged_off_host", torch.int64, cuda=False)
    _need(staging, "staging", torch.uint8); _need(staged_off, "staged_off", torch.int64)
    if done_event.cuda_event == 0:
        done_event.record(copy_stream)  # torch creates the CUDA event at its first record
    n = _c_i32(0)
    c = cfg.c()
    _check("sekv_fetch_bases_copy",
           lib().sekv_fetch_bases_copy(ctypes.byref(c), ctypes.byref(cache.c), _ptr(expanded_host),
                                       _ptr(n_expanded_host), _ptr(rec_off_host), _ptr(staging),
                                       int(per_group), _ptr(staged_off_host), _ptr(staged_off),
                                       ctypes.byref(n), ctypes.c_void_p(copy_stream.cuda_stream),
                                       ctypes.c_void_p(done_event.cuda_event)))
    return n.value


class BasisCache:
    """Residency cache table of one layer (sekv_basis_cache_*): n_slots slots
    of slot_bytes per (sequence, KV head) group, living after the staging
    area of the caller's staging buffer (see staging_bytes)."""

    def __init__(self, cfg: Config, n_slots: int, slot_bytes: int, device=None):
        c = cfg.c()
        n = int(lib().sekv_basis_cache_bytes(ctypes.byref(c), n_slots))
        if n == 0:
            raise SekvError("sekv_basis_cache_bytes", -1)
        self.n_slots, self.slot_bytes = n_slots, slot_bytes
        self.table = torch.empty(n, dtype=torch.uint8, device=device or "cuda")
        _check("sekv_basis_cache_init", lib().sekv_basis_cache_init(ctypes.byref(c),
                                                                     _ptr(self.table), n_slots,
                                                                     _stream()))

    def staging_bytes(self, cfg: Config, per_group: int) -> int:
        return cfg.batch * cfg.n_kv_heads * (per_group + self.n_slots * self.slot_bytes)


def fetch_bases_cached(cfg: Config, cache: LayerCache, expanded, n_expanded, staging,
                       per_group: int, bcache: BasisCache, staged_off, ws: Workspace, hits=None,
                       copied=None, stream=None):
    _need(staging, "staging", torch.uint8); _need(staged_off, "staged_off", torch.int64)
    if staging.numel() < bcache.staging_bytes(cfg, per_group):
        raise ValueError("staging: smaller than the staging area plus the cache's slots")
    c = cfg.c()
    _check("sekv_fetch_bases_cached",
           lib().sekv_fetch_bases_cached(ctypes.byref(c), ctypes.byref(cache.c), _ptr(expanded),
                                         _ptr(n_expanded), _ptr(staging), int(per_group),
                                         _ptr(bcache.table), bcache.n_slots, bcache.slot_bytes,
                                         _ptr(staged_off), _ptr(hits), _ptr(copied), ws.ptr(),
                                         ws.nbytes, _stream(stream)))
    return staging, staged_off


def alloc_cache(cfg: Config, store_bytes: int, device=None) -> Dict[str, torch.Tensor]:
    """Zeroed tensors for one layer of the cache in the C-ABI layout."""
    dev = device or "cuda"
    B, Hkv, ms = cfg.batch, cfg.n_kv_heads, cfg.max_spans
    cap = cfg.n_sink + ms + cfg.n_recent
    z = lambda *shape, dt: torch.zeros(*shape, dtype=dt, device=dev)  # noqa: E731
    return dict(n_spans=z(B, dt=torch.int32), body_len=z(B, ms, dt=torch.int32),
                k_full=z(B, Hkv, cap, 128, dt=torch.bfloat16),
                v_full=z(B, Hkv, cap, 128, dt=torch.bfloat16),
                s_route=z(B, Hkv, ms, 64, dt=torch.float32),
                k_sum=z(B, Hkv, ms, 128, dt=torch.bfloat16),
                v_sum=z(B, Hkv, ms, 128, dt=torch.bfloat16),
                rec_off=z(B, Hkv, ms, dt=torch.int64), rec_rank=z(B, Hkv, ms, dt=torch.int32),
                store=z(store_bytes, dt=torch.uint8))


def build_spans(cfg: Config, K, V, H, W_r, gates, out: Dict[str, torch.Tensor], ws: Workspace,
                stream=None) -> Dict[str, torch.Tensor]:
    """Prefill build of one layer into `out` (tensors from alloc_cache)."""
    _need(K, "K", torch.bfloat16); _need(V, "V", torch.bfloat16)
    _need(H, "H", torch.float32); _need(W_r, "W_r", torch.float32)
    _need(gates, "gates", torch.float32)
    T = K.shape[2]
    o = SekvCacheOut(*[_ptr(out[k]) for k in CACHE_FIELDS], out["store"].numel())
    c = cfg.c()
    _check("sekv_build_spans",
           lib().sekv_build_spans(ctypes.byref(c), T, _ptr(K), _ptr(V), _ptr(H), _ptr(W_r),
                                  _ptr(gates), ctypes.byref(o), ws.ptr(), ws.nbytes,
                                  _stream(stream)))
    return out


def build_flops(ws: Workspace, stream=None) -> int:
    """fp32 operations the span SVDs of the builds on `ws` performed since the
    last read (sekv_build_flops); synchronises and clears the count."""
    v = _c_i64(0)
    _check("sekv_build_flops", lib().sekv_build_flops(ws.ptr(), _stream(stream), ctypes.byref(v)))
    return v.value


class Maintainer:
    """Decode-time maintenance of one layer's cache (sekv_maint_init,
    sekv_append_token): `out` is the dict of sekv_build_spans' output tensors;
    this object adds the per-sequence tail lengths (``n_tail``) and the state
    buffer, and keeps the sequence length.  ``layer_cache()`` gives the
    LayerCache (with n_tail) that the decode calls read."""

    def __init__(self, cfg: Config, out: Dict[str, torch.Tensor], K, V, H, ctx_len: int,
                 ws: Workspace, stream=None):
        self.cfg, self.out, self.ws, self.T = cfg, out, ws, int(ctx_len)
        dev = out["k_full"].device
        c = cfg.c()
        n = int(lib().sekv_maint_state_size(ctypes.byref(c)))
        self.state = torch.zeros(n, dtype=torch.uint8, device=dev)
        self.n_tail = torch.zeros(cfg.batch, dtype=torch.int32, device=dev)
        self._o = SekvCacheOut(*[_ptr(out[k]) for k in CACHE_FIELDS], out["store"].numel())
        _need(K, "K", torch.bfloat16); _need(V, "V", torch.bfloat16); _need(H, "H", torch.float32)
        _check("sekv_maint_init",
               lib().sekv_maint_init(ctypes.byref(c), self.T, _ptr(K), _ptr(V), _ptr(H),
                                     ctypes.byref(self._o), _ptr(self.n_tail), _ptr(self.state),
                                     self.state.numel(), ws.ptr(), ws.nbytes, _stream(stream)))

    def append(self, k_new, v_new, h_new, stream=None):
        """sekv_append_token: one token per sequence (lengths advance on the
        device; `T` here mirrors them for the caller).  Spans it closes wait
        at full resolution until `flush`."""
        _need(k_new, "k_new", torch.bfloat16); _need(v_new, "v_new", torch.bfloat16)
        _need(h_new, "h_new", torch.float32)
        c = self.cfg.c()
        _check("sekv_append_token",
               lib().sekv_append_token(ctypes.byref(c), _ptr(k_new), _ptr(v_new), _ptr(h_new),
                                       ctypes.byref(self._o), _ptr(self.n_tail), _ptr(self.state),
                                       self.state.numel(), self.ws.ptr(), self.ws.nbytes,
                                       _stream(stream)))
        self.T += 1

    def flush(self, W_r, gates, stream=None):
        """sekv_maint_flush: builds every closed span still waiting."""
        _need(W_r, "W_r", torch.float32); _need(gates, "gates", torch.float32)
        c = self.cfg.c()
        _check("sekv_maint_flush",
               lib().sekv_maint_flush(ctypes.byref(c), _ptr(W_r), _ptr(gates),
                                      ctypes.byref(self._o), _ptr(self.n_tail), _ptr(self.state),
                                      self.state.numel(), self.ws.ptr(), self.ws.nbytes,
                                      _stream(stream)))

    def layer_cache(self) -> LayerCache:
        return LayerCache({**{k: self.out[k] for k in CACHE_FIELDS}, "n_tail": self.n_tail})


def default_scale() -> float:
    return 1.0 / math.sqrt(128.0)
