"""Decode-step benchmark of the SeKV span-cache hot path on GB300.

One step = routing + mixed-resolution attention of every layer, in layer
order, for one decode token (Llama-3-8B shape at 128K context: 32 layers, 32
query / 8 KV heads, about 5% of spans expanded), inputs resident in HBM, all
32 fused launches captured in one CUDA graph.  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl sekv|reference]

N > 1 (torchrun): every rank runs an independent replica on its own GPU
(the path has no exchange step); value = steps of all ranks / max time.
--impl reference times the fp64 CPU oracle on a bounded sample of the same
workload (there is no other implementation of this method to run).
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402
from synth import gen  # noqa: E402

METRIC = "decode steps/s at 128K ctx; achieved HBM GB/s vs ~8 TB/s roofline"


def decode_metric(w) -> str:
    """The headline metric's name for the 128K workload; the same wording with
    the workload's own context length for the others."""
    if w.name == "llama3_8b_128k":
        return METRIC
    return f"decode steps/s at {w.ctx // 1024}K ctx ({w.name}); achieved HBM GB/s vs ~8 TB/s roofline"
UNIT = "steps/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="sekv", choices=["sekv", "reference"])
    ap.add_argument("--config", default="llama3_8b_128k")
    ap.add_argument("--layers", type=int, default=0, help="override layer count (tests only)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--traffic-from", default=None, metavar="CSV",
                    help="write profiles/decode_kernel_traffic.json from an ncu --csv capture of "
                         "dram__bytes_read.sum / dram__bytes_write.sum and exit")
    ap.add_argument("--traffic-workload", default="llama3_8b_128k")
    ap.add_argument("--traffic-scale", type=float, default=1.0)
    ap.add_argument("--traffic-command", default="")
    ap.add_argument("--path", default="decode",
                    choices=["decode", "build", "fullkv", "append", "multi", "e2e"],
                    help="decode: the headline decode step; build: the prefill cache build; "
                         "fullkv: the same decode step over a full-KV cache (comparator); "
                         "append: decode-time cache maintenance, one token per step; "
                         "multi: several query tokens per sequence over one cache; "
                         "e2e: the tiered end-to-end leg of the decode line alone")
    ap.add_argument("--query-tokens", type=int, default=2,
                    help="multi: query tokens per sequence (launched in blocks of 8 / hpg)")
    return ap.parse_args()


def dist_setup(args):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return ws, rank, local


def whole_job_rate(steps: int, ms_max: float, world: int) -> float:
    """Steps/s of the whole job: every rank runs `steps` steps of its own
    replica; the slowest rank's time counts."""
    return steps * world / (ms_max / 1000.0)


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, ws: int) -> float:
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------
# peaks and clocks
# ----------------------------------------------------------------------------

DECODE_SOURCES = ("decode_attn.cuh", "decode_consumer.cuh", "decode_kernel_impl.cuh",
                  "decode_ks1.cu", "decode_ks2.cu", "decode_ks3.cu", "decode_ks4.cu",
                  "sekv_common.cuh")
TRAFFIC_JSON = os.path.join(ROOT, "profiles", "decode_kernel_traffic.json")


def decode_source_hash() -> str:
    """sha256 over the decode kernel's sources (the kernel a capture covers)."""
    import hashlib
    h = hashlib.sha256()
    for f in DECODE_SOURCES:
        with open(os.path.join(ROOT, "decode_attention_span_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def profiled_traffic(workload: str):
    """DRAM bytes per decode launch (read + write) for `workload`, from the
    JSON that ``--traffic-from`` wrote out of an ncu capture, or None when the
    kernel sources changed since that capture or it covers another workload."""
    try:
        with open(TRAFFIC_JSON, encoding="utf-8") as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    e = d.get(workload)
    if not e or e.get("source_sha256") != decode_source_hash():
        return None
    return e.get("bytes_per_launch")


def write_traffic(csv_path: str, workload: str, launch_scale: float, command: str):
    """Parse an ncu --csv capture (metrics dram__bytes_read.sum and
    dram__bytes_write.sum of the decode kernel) and record the mean DRAM bytes
    per launch, times `launch_scale` (the capture's workload scaled to a full
    launch), in profiles/decode_kernel_traffic.json under `workload`."""
    import csv
    per = {}
    with open(csv_path, newline="", encoding="utf-8", errors="replace") as f:
        rows = [r for r in csv.reader(f)]
    head = None
    for i, r in enumerate(rows):
        if "Metric Name" in r and "Kernel Name" in r:
            head = i
            break
    if head is None:
        raise SystemExit(f"{csv_path}: no ncu metric table")
    cols = rows[head]
    ki, ii, mi, vi = (cols.index("Kernel Name"), cols.index("ID"), cols.index("Metric Name"),
                      cols.index("Metric Value"))
    unit_i = cols.index("Metric Unit") if "Metric Unit" in cols else None
    scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "KB": 1e3, "MB": 1e6,
             "GB": 1e9, "B": 1}
    for r in rows[head + 1:]:
        if len(r) <= max(ki, ii, mi, vi) or "decode_kernel" not in r[ki]:
            continue
        if r[mi] not in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            continue
        v = float(r[vi].replace(",", ""))
        if unit_i is not None:
            v *= scale.get(r[unit_i], 1)
        per[r[ii]] = per.get(r[ii], 0.0) + v
    if not per:
        raise SystemExit(f"{csv_path}: no decode_kernel DRAM metrics")
    mean = sum(per.values()) / len(per)
    try:
        with open(TRAFFIC_JSON, encoding="utf-8") as f:
            d = json.load(f)
    except (OSError, ValueError):
        d = {}
    d[workload] = {"bytes_per_launch": int(round(mean * launch_scale)), "launches": len(per),
                   "captured_bytes_per_launch": int(round(mean)), "launch_scale": launch_scale,
                   "source_sha256": decode_source_hash(), "command": command}
    with open(TRAFFIC_JSON, "w", encoding="utf-8") as f:
        json.dump(d, f, indent=1, sort_keys=True)
        f.write("\n")
    print(json.dumps({workload: d[workload]}))


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        self.proc.wait()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ----------------------------------------------------------------------------
# workload
# ----------------------------------------------------------------------------

def algorithmic_bytes(d, lst, cnt, cfg) -> int:
    """Bytes the method must touch for one layer (one launch of the kernel).

    Per (sequence, KV head): 512 B per full-resolution row (K + V bf16),
    256 + 16 B per span (routing summary fp32 + body length, ranks and record
    offset), 512 B per unexpanded non-empty span (summary K + V bf16), and per
    expanded span its factors: U_K, U_V (b x r bf16), Vt_K, Vt_V (r x 128 bf16),
    sigma and g (r fp32 each), for keys and values.  Padding, record headers and
    the masked summary rows of expanded spans are not counted.
    """
    B, Hkv, ms = cfg.batch, cfg.n_kv_heads, cfg.max_spans
    n_sp = d["n_spans"].long()                                        # [B]
    body = d["body_len"].long()                                       # [B][ms]
    nonempty = (body > 0).sum(1)                                      # [B]
    n_full = cfg.n_sink + n_sp + cfg.n_recent
    cnt = cnt.view(B, Hkv).long()
    fixed = (512 * n_full[:, None] + 272 * n_sp[:, None] + 512 * (nonempty[:, None] - cnt)).sum()
    lst = lst.view(B, Hkv, ms).long()
    idx = torch.arange(ms, device=lst.device)[None, None, :]
    valid = idx < cnt[:, :, None]
    k = torch.where(valid, lst, torch.zeros_like(lst))
    bb = torch.gather(body[:, None, :].expand(B, Hkv, ms), 2, k)
    rr = torch.gather(d["rec_rank"].long(), 2, k)
    r_sum = (rr & 0xFFFF) + ((rr >> 16) & 0xFFFF)
    fac = (2 * bb * r_sum + 264 * r_sum) * valid
    return int((fixed + fac.sum()).item())


def record_bytes_fetched(d, lst, cnt, cfg) -> int:
    B, Hkv, ms = cfg.batch, cfg.n_kv_heads, cfg.max_spans
    cnt = cnt.view(B, Hkv).long()
    lst = lst.view(B, Hkv, ms).long()
    idx = torch.arange(ms, device=lst.device)[None, None, :]
    valid = idx < cnt[:, :, None]
    k = torch.where(valid, lst, torch.zeros_like(lst))
    bb = torch.gather(d["body_len"].long()[:, None, :].expand(B, Hkv, ms), 2, k)
    rr = torch.gather(d["rec_rank"].long(), 2, k)
    return int((gen.record_size(bb, rr & 0xFFFF, (rr >> 16) & 0xFFFF) * valid).sum().item())


def build_workload(sk, w, dev, n_layers):
    ms = gen.max_spans_for(w)
    cfg = sk.Config(w.batch, w.n_q_heads, w.n_kv_heads, w.n_sink, w.n_recent, ms, w.rank_cap,
                    w.len_min, w.len_max, w.tau, flags=sk.sekv.FLAG_OVERLAP_PREVIOUS)
    ws = sk.Workspace(cfg, dev)
    p_head = gen.per_head_fraction(w.expand_frac, w.group)
    layers = []
    for l in range(n_layers):
        d = gen.decode_cache(w, l, device=dev, max_spans=ms)
        tens = {k: v for k, v in d.items() if isinstance(v, torch.Tensor)}
        cache = sk.LayerCache(tens)
        g = gen._gen(w.seed * 7919 + 101 * l + 1, dev)
        q = gen.query(g, w.batch, w.n_q_heads, dev)
        W = gen.routing_weights(g, w.n_kv_heads, dev).contiguous()
        inf = torch.full((w.n_q_heads,), float("inf"), device=dev)
        _, _, z = sk.route(cfg, cache, q, W, inf, ws, want_z=True)
        z = z.view(w.batch, w.n_q_heads, ms).cpu().numpy()
        nsp = d["n_spans"].cpu().numpy()
        theta = np.array([gen.pick_threshold(np.concatenate([z[b, h, :nsp[b]]
                                                             for b in range(w.batch)]), p_head)
                          for h in range(w.n_q_heads)], np.float32)
        theta_t = torch.from_numpy(theta).to(dev)
        lst, cnt, _ = sk.route(cfg, cache, q, W, theta_t, ws)
        nbytes = algorithmic_bytes(tens, lst, cnt, cfg)
        fetched = record_bytes_fetched(tens, lst, cnt, cfg)
        n_ne = int((d["body_len"] > 0).sum().item()) * w.n_kv_heads
        layers.append(dict(t=tens, cache=cache, q=q, W=W, theta=theta_t, theta_np=theta,
                           out=torch.empty(w.batch, w.n_q_heads, 128, device=dev),
                           lse=torch.empty(w.batch, w.n_q_heads, device=dev),
                           bytes=nbytes, fetched=fetched, n_exp=int(cnt.sum().item()),
                           n_nonempty=n_ne))
    torch.cuda.synchronize()
    ws.raise_on_error()
    return cfg, ws, layers


# ----------------------------------------------------------------------------
# timed runs
# ----------------------------------------------------------------------------

def time_graph(step_fn, steps, warmup, stream, ws_n, clocks=None):
    with torch.cuda.stream(stream):
        step_fn()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            step_fn()
    for _ in range(max(warmup, 3)):
        with torch.cuda.stream(stream):
            graph.replay()
    torch.cuda.synchronize()
    barrier(ws_n)
    torch.cuda.synchronize()
    if clocks:
        clocks.start()
        time.sleep(0.3)
        # the GPU idled while the sampler started: warm it up again so that the
        # timed replays do not include its clock ramp
        with torch.cuda.stream(stream):
            for _ in range(max(warmup, 3)):
                graph.replay()
        torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            graph.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    barrier(ws_n)
    torch.cuda.synchronize()
    ck = clocks.stop() if clocks else None
    return e0.elapsed_time(e1), ck


def run_resident(sk, cfg, ws, layers, steps, warmup, ws_n, clocks):
    scale = sk.default_scale()

    def step():
        for L in layers:
            sk.decode_step(cfg, L["cache"], L["q"], L["W"], L["theta"], scale, ws,
                           out=L["out"], lse=L["lse"])

    stream = torch.cuda.Stream()
    ms, ck = time_graph(step, steps, warmup, stream, ws_n, clocks)
    code, detail = ws.status()
    if code:
        raise RuntimeError(f"device status {code} ({detail}) after the timed run")
    return ms, ck


def h2d_peak_gbs(dev, nbytes: int = 1 << 30) -> float:
    """Host-link peak: one large pinned host -> device copy, best of 6, timed
    with CUDA events."""
    src = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    dst = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    best = 0.0
    for _ in range(6):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        dst.copy_(src, non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        best = max(best, nbytes / (e0.elapsed_time(e1) / 1e3) / 1e9)
    del src, dst
    return best


QUERY_SETS = 8        # distinct queries per layer, used in turn by successive steps
QUERY_DRIFT = 0.3     # q_s = sqrt(1 - d^2) q_(s-1) + d n, n ~ N(0, 1)
SIDE_STREAMS = 3         # tiered mode: streams that route and fetch ahead of attention
CACHE_SLOTS = 256     # residency cache slots per (sequence, KV head), 20 KB each
CACHE_SLOT_BYTES = 20480
STAGING_PER_GROUP = 8 << 20


def drifting_queries(layers, seed: int):
    """QUERY_SETS query sets per layer: set 0 is the layer's query; each next
    set moves away from the previous one by QUERY_DRIFT (successive decode
    tokens' queries are correlated, so their expansion sets overlap)."""
    g = torch.Generator().manual_seed(seed)
    sets = [torch.stack([L["q"].cpu() for L in layers])]
    c = math.sqrt(1.0 - QUERY_DRIFT ** 2)
    for _ in range(QUERY_SETS - 1):
        prev = sets[-1].float()
        nxt = c * prev + QUERY_DRIFT * torch.randn(prev.shape, generator=g)
        sets.append(nxt.to(torch.bfloat16))
    return [x.pin_memory() for x in sets]


def run_tiered(sk, cfg, w, layers, steps, warmup, ws_n, dev):
    """End to end through the C ABI with host buffers.  Each step copies every
    layer's query from pinned host memory, routes it, fetches the expanded
    spans' bases through the residency cache (misses over the host link from
    the pinned host store), attends, and reads every layer's output back.
    Routing and fetch of a layer run on a side stream that runs ahead of the
    attention stream, so the fetch of layer l+1 overlaps the attention of
    layer l (every layer's query is an input of the step).  Successive steps
    use drifting query sets (drifting_queries), so the cache sees the partial
    reuse of consecutive tokens."""
    scale = sk.default_scale()
    cfg_t = sk.Config(**{**cfg.__dict__, "flags": 0})
    ws_main = sk.Workspace(cfg_t, dev)
    ws_sides = [sk.Workspace(cfg_t, dev) for _ in range(SIDE_STREAMS)]
    L_n, B, Hq = len(layers), cfg.batch, cfg.n_q_heads
    NG, ms = B * cfg.n_kv_heads, cfg.max_spans
    q_sets = drifting_queries(layers, w.seed * 31 + 5)
    q_dev = torch.empty_like(q_sets[0], device=dev)
    out_dev = torch.empty(L_n, B, Hq, 128, device=dev)
    out_host = torch.empty(L_n, B, Hq, 128).pin_memory()
    per = []
    for L in layers:
        host = dict(L["t"])
        host["store"] = L["t"]["store"].cpu().pin_memory()
        bc = sk.BasisCache(cfg_t, CACHE_SLOTS, CACHE_SLOT_BYTES, dev)
        per.append(dict(cache=sk.LayerCache(host, store_on_host=True), bc=bc,
                        staging=torch.empty(bc.staging_bytes(cfg_t, STAGING_PER_GROUP),
                                            dtype=torch.uint8, device=dev),
                        staged_off=torch.empty(NG * ms, dtype=torch.int64, device=dev),
                        lst=torch.empty(NG * ms, dtype=torch.int32, device=dev),
                        cnt=torch.empty(NG, dtype=torch.int32, device=dev),
                        hits=torch.zeros(NG, dtype=torch.int32, device=dev),
                        copied=torch.zeros(NG, dtype=torch.int64, device=dev),
                        ev=torch.cuda.Event()))
    # side streams take the layers in turn, so that one layer's routing and
    # planning overlap the previous layers' copies over the host link
    sides = [torch.cuda.Stream() for _ in range(SIDE_STREAMS)]
    ev_q, ev_end = torch.cuda.Event(), [torch.cuda.Event() for _ in range(SIDE_STREAMS)]
    launches = [0]

    def step(s):
        main = torch.cuda.current_stream()
        n = 0
        q_dev.copy_(q_sets[s], non_blocking=True)
        ev_q.record(main)
        for sd in sides:
            sd.wait_event(ev_q)
        for i, L in enumerate(layers):
            X = per[i]
            side, ws_side = sides[i % SIDE_STREAMS], ws_sides[i % SIDE_STREAMS]
            sk.route(cfg_t, X["cache"], q_dev[i], L["W"], L["theta"], ws_side, expanded=X["lst"],
                     n_expanded=X["cnt"], stream=side)
            n += sk.last_launch_count()
            sk.fetch_bases_cached(cfg_t, X["cache"], X["lst"], X["cnt"], X["staging"],
                                  STAGING_PER_GROUP, X["bc"], X["staged_off"], ws_side,
                                  hits=X["hits"], copied=X["copied"], stream=side)
            n += sk.last_launch_count()
            X["ev"].record(side)
            main.wait_event(X["ev"])
            sk.decode_attention(cfg_t, X["cache"], q_dev[i], X["lst"], X["cnt"], scale, ws_main,
                                staging=X["staging"], staged_off=X["staged_off"],
                                out=out_dev[i], stream=main)
            n += sk.last_launch_count()
        for sd, ev in zip(sides, ev_end):
            ev.record(sd)
            main.wait_event(ev)
        out_host.copy_(out_dev, non_blocking=True)
        launches[0] = n

    stream = torch.cuda.Stream()
    graphs = []
    with torch.cuda.stream(stream):
        for s in range(QUERY_SETS):
            step(s)
        torch.cuda.synchronize()
        for s in range(QUERY_SETS):
            gph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gph, stream=stream):
                step(s)
            graphs.append(gph)
    for i in range(max(warmup, 3) + QUERY_SETS):
        with torch.cuda.stream(stream):
            graphs[i % QUERY_SETS].replay()
    torch.cuda.synchronize()
    barrier(ws_n)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(steps):
            graphs[i % QUERY_SETS].replay()
        e1.record(stream)
    torch.cuda.synchronize()
    barrier(ws_n)
    torch.cuda.synchronize()
    ms_total = e0.elapsed_time(e1)
    for W_ in (*ws_sides, ws_main):
        code, detail = W_.status()
        if code:
            raise RuntimeError(f"device status {code} ({detail}) after the tiered run")
    last = (steps - 1) % QUERY_SETS
    n_exp = sum(int(X["cnt"].sum()) for X in per)
    hits = sum(int(X["hits"].sum()) for X in per)
    copied = sum(int(X["copied"].sum()) for X in per)
    # the last step's outputs against the resident path on the same queries
    ws_r = sk.Workspace(cfg_t, dev)
    err = 0.0
    for i, L in enumerate(layers):
        o, _, _, _ = sk.decode_step(cfg_t, L["cache"], q_sets[last][i].to(dev), L["W"], L["theta"],
                                    scale, ws_r)
        err = max(err, float((out_host[i] - o.cpu()).abs().max()))
    h2d = q_sets[0].numel() * 2 + copied
    d2h = out_host.numel() * 4
    return dict(ms=ms_total, steps=steps, h2d=h2d, d2h=d2h, launches=launches[0], err=err,
                hit_frac=hits / max(1, n_exp), copied=copied, n_exp=n_exp,
                fetch_paths=fetch_path_times(sk, cfg_t, layers, per, q_sets, dev))


def e2e_leg(sk, cfg, w, layers, steps, warmup, ws_n, dev):
    """The tiered end-to-end measurement (run_tiered) as the bench line's
    `e2e` object; also returns the library launches of one step."""
    peak_h2d = h2d_peak_gbs(dev)
    r = run_tiered(sk, cfg, w, layers, steps, warmup, ws_n, dev)
    ms_e = max_over_ranks(r["ms"], ws_n)
    step_s = ms_e / steps / 1e3
    e2e = {"value": ws_n * steps / (ms_e / 1e3), "unit": UNIT,
           "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"],
           "path": f"tiered: q H2D; per layer route + residency-cached fetch of the bases from "
                   f"pinned host memory on one of {SIDE_STREAMS} side streams running ahead of "
                   f"attention; out D2H; one CUDA graph per step",
           "queries": f"{QUERY_SETS} drifting query sets in turn (drift {QUERY_DRIFT} per step)",
           "cache": {"slots_per_group": CACHE_SLOTS, "slot_bytes": CACHE_SLOT_BYTES,
                     "hit_frac": r["hit_frac"], "expanded_per_step": r["n_exp"],
                     "record_bytes_copied_per_step": r["copied"]},
           "h2d_gbs": r["h2d"] / step_s / 1e9, "h2d_peak_gbs": peak_h2d,
           "h2d_frac_of_peak": r["h2d"] / step_s / 1e9 / peak_h2d,
           "fetch_paths": r["fetch_paths"],
           "steps": steps, "max_abs_vs_resident": r["err"]}
    return e2e, r["launches"]


def run_e2e_bench(args, ws_n, rank, local):
    """The tiered end-to-end leg alone (bases in pinned host memory, residency
    cache, routing and fetch on side streams ahead of attention): the decode
    line's `e2e` object as a line of its own, for profiling the pipeline."""
    import decode_attention_span_gb300 as sk
    if not torch.cuda.is_available():
        raise SystemExit("bench.py (e2e) needs a CUDA device")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = synth.get_config(args.config, **({"layers": args.layers} if args.layers else {}))
    cfg, _, layers = build_workload(sk, w, dev, w.layers)
    e2e, launches = e2e_leg(sk, cfg, w, layers, args.steps, args.warmup, ws_n, dev)
    if rank != 0:
        return
    line = {"metric": "tiered " + decode_metric(w).split(";")[0] + " (bases in pinned host memory)",
            "value": e2e["value"], "unit": UNIT, "n_gpus": ws_n, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 / e2e["value"] * ws_n,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": decode_config(w, ws_n), "e2e": e2e,
            "gpu_launches": args.steps * launches}
    print(json.dumps(line), flush=True)


def fetch_path_times(sk, cfg, layers, per, q_sets, dev):
    """One step's fetch of every layer's expanded bases (query set 0) by the
    three forms, timed on their own: the gather kernel over mapped pinned
    memory, the host-driven copies (lists back to the host, one
    cudaMemcpyAsync per run of adjacent records, an event), and the warm
    residency cache."""
    ws = sk.Workspace(cfg, dev)
    NG, ms = cfg.batch * cfg.n_kv_heads, cfg.max_spans
    q = q_sets[0].to(dev)
    lists = []
    for i, L in enumerate(layers):
        lst, cnt, _ = sk.route(cfg, per[i]["cache"], q[i], L["W"], L["theta"], ws)
        lists.append((lst, cnt))
    torch.cuda.synchronize()
    staging = torch.empty(NG * STAGING_PER_GROUP, dtype=torch.uint8, device=dev)
    staged_off = torch.empty(NG * ms, dtype=torch.int64, device=dev)
    # gather kernel
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(len(layers)):
        sk.fetch_bases(cfg, per[i]["cache"], lists[i][0], lists[i][1], staging, STAGING_PER_GROUP,
                       staged_off, ws)
    e1.record()
    torch.cuda.synchronize()
    gather_ms = e0.elapsed_time(e1)
    # host-driven copies, including the lists' trip to the host
    side = torch.cuda.Stream()
    done = torch.cuda.Event()
    lst_h = torch.empty(NG * ms, dtype=torch.int32).pin_memory()
    cnt_h = torch.empty(NG, dtype=torch.int32).pin_memory()
    off_h = torch.empty(NG * ms, dtype=torch.int64).pin_memory()
    rec_off_h = [L["t"]["rec_off"].cpu().contiguous() for L in layers]
    copies = 0
    t0 = time.perf_counter()
    for i in range(len(layers)):
        lst_h.copy_(lists[i][0], non_blocking=True)
        cnt_h.copy_(lists[i][1], non_blocking=True)
        torch.cuda.current_stream().synchronize()
        copies += sk.fetch_bases_copy(cfg, per[i]["cache"], lst_h, cnt_h, rec_off_h[i], staging,
                                      STAGING_PER_GROUP, off_h, staged_off, done, side)
        done.synchronize()
    copy_ms = (time.perf_counter() - t0) * 1e3
    # residency cache, warm (the tables hold the timed run's last state)
    e0.record()
    for i in range(len(layers)):
        X = per[i]
        sk.fetch_bases_cached(cfg, X["cache"], lists[i][0], lists[i][1], X["staging"],
                              STAGING_PER_GROUP, X["bc"], X["staged_off"], ws, hits=X["hits"],
                              copied=X["copied"])
    e1.record()
    torch.cuda.synchronize()
    cached_ms = e0.elapsed_time(e1)
    rec_bytes = sum(L["fetched"] for L in layers)
    return {"record_bytes_per_step": rec_bytes,
            "gather_kernel_ms_per_step": gather_ms,
            "gather_kernel_gbs": rec_bytes / (gather_ms / 1e3) / 1e9,
            "memcpy_per_run_ms_per_step": copy_ms, "memcpy_copies_per_step": copies,
            "memcpy_per_run_gbs": rec_bytes / (copy_ms / 1e3) / 1e9,
            "cached_ms_per_step": cached_ms,
            "note": "query set 0 of every layer; the memcpy form is host wall time including "
                    "the lists' device-to-host trip and a synchronisation per layer"}


# ----------------------------------------------------------------------------
# CPU oracle (bench's cpu_baseline leg and the --impl reference arm)
# ----------------------------------------------------------------------------

def _group_arrays(arr, b, c):
    """ABI arrays of one (sequence, KV head) as a batch-1, one-KV-head layer."""
    out = dict(arr)
    out["n_spans"] = arr["n_spans"][b:b + 1]
    out["body_len"] = arr["body_len"][b:b + 1]
    for k in ("k_full", "v_full", "s_route", "k_sum", "v_sum", "rec_off", "rec_rank"):
        out[k] = arr[k][b:b + 1, c:c + 1]
    return out


UNITS_PER_STEP_DOC = ("one timed sample is one (layer, sequence, KV head) unit: the oracle's "
                      "routing + mixed-resolution attention of one group")


def decode_config(w, ws_n: int) -> dict:
    """The workload a decode line is quoted on (the same on both arms)."""
    return {"workload": w.name, "layers": w.layers, "batch": w.batch, "ctx": w.ctx,
            "q_heads": w.n_q_heads, "kv_heads": w.n_kv_heads,
            "expand_frac_target": w.expand_frac, "bases": "hbm-resident",
            "l2": "inputs larger than L2 (distinct buffers per layer)",
            "parallelism": f"replicas x{ws_n}",
            "graph": "one CUDA graph per step, programmatic dependent launch"}


def oracle_units(w, n: int):
    """The oracle's inputs for the first n (sequence, KV head) groups of layer
    0 of the workload, drawn on the CPU: the one unit sample both oracle legs
    time (the cpu_baseline leg and --impl reference).  Thresholds come from
    the oracle's own logits (per-head quantile, 1e-3 margin)."""
    import oracle
    from oracle import layout
    G = w.group
    p_head = gen.per_head_fraction(w.expand_frac, G)
    arr = gen.abi_to_numpy(gen.decode_cache(w, 0, device="cpu"))
    g = gen._gen(w.seed * 7919 + 1)
    q = gen.query(g, w.batch, w.n_q_heads).float().numpy()
    W = gen.routing_weights(g, w.n_kv_heads).numpy()
    units = []
    for b in range(w.batch):
        for c in range(w.n_kv_heads):
            if len(units) >= n:
                return units
            cache = layout.unpack_layer(_group_arrays(arr, b, c), w.n_sink, w.n_recent)
            qg, Wg = q[b:b + 1, c * G:(c + 1) * G], W[c:c + 1]
            z = oracle.route_logits(qg, Wg, cache)
            theta = np.array([gen.pick_threshold(z[0][h], p_head) for h in range(G)])
            units.append((cache, qg, Wg, theta))
    return units


def time_units(units, n_warm: int, n_timed: int):
    """Seconds per unit of the oracle's routing + attention, cycling over
    `units`."""
    import oracle
    times = []
    for i in range(n_warm + n_timed):
        cache, qg, Wg, theta = units[i % len(units)]
        t0 = time.perf_counter()
        E, _ = oracle.route(qg, Wg, cache, theta)
        oracle.decode_attention(qg, cache, E, 1.0 / math.sqrt(128.0))
        if i >= n_warm:
            times.append(time.perf_counter() - t0)
    return times


def cpu_baseline_leg(w, seconds: float) -> dict:
    """The oracle on the host cores: the shared unit sample, about `seconds`
    of timed work, scaled to steps/s."""
    units = oracle_units(w, 8)
    est = float(np.mean(time_units(units, 1, 1)))
    n = max(2, int(seconds / max(est, 1e-6)))
    times = time_units(units, 0, n)
    units_per_step = w.batch * w.n_kv_heads * w.layers
    value = 1.0 / (float(np.mean(times)) * units_per_step)
    return {"value": value, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
            "sample": f"{UNITS_PER_STEP_DOC}; {n} units timed, cycling over the first "
                      f"{len(units)} groups of layer 0 (drawn on the CPU); steps/s = 1 / (mean "
                      f"unit time x {units_per_step} units per step)",
            "units_timed": n, "units_per_step": units_per_step}


def parity_check(sk, cfg, ws, L, w) -> dict:
    """The bench's own layer 0 against the oracle: sequence 0, KV head 0, at
    the full workload size and in the timed launch configuration.  The
    group's thresholds come from the oracle's own logits (1e-3 margin); the
    GPU step is run again with them, outside the timed region."""
    import oracle
    from oracle import layout
    G = w.group
    arr = gen.abi_to_numpy(L["t"])
    cache = layout.unpack_layer(_group_arrays(arr, 0, 0), w.n_sink, w.n_recent)
    qg = L["q"].float().cpu().numpy()[0:1, 0:G]
    Wg = L["W"].cpu().numpy()[0:1]
    z = oracle.route_logits(qg, Wg, cache)
    p_head = gen.per_head_fraction(w.expand_frac, G)
    th = np.array([gen.pick_threshold(z[0][h], p_head) for h in range(G)], np.float32)
    E, _ = oracle.route(qg, Wg, cache, th)
    scale = 1.0 / math.sqrt(128.0)
    o_ref, lse_ref = oracle.decode_attention(qg, cache, E, scale)
    theta = L["theta"].clone()
    theta[:G] = torch.from_numpy(th).to(theta.device)
    out, lse, lst, cnt = sk.decode_step(cfg, L["cache"], L["q"], L["W"], theta, scale, ws,
                                        want_list=True)
    torch.cuda.synchronize()
    o = out[0, :G].double().cpu().numpy()
    err = float(np.abs(o - o_ref[0]).max())
    rel = float(np.linalg.norm(o - o_ref[0]) / max(np.linalg.norm(o_ref[0]), 1e-30))
    n = int(cnt[0])
    same = n == len(E[0][0]) and bool(np.array_equal(lst[:n].cpu().numpy(), E[0][0]))
    return {"sample": "layer 0, sequence 0, KV head 0 (its query heads), full size, timed "
                      "launch configuration, thresholds from the oracle's logits",
            "max_abs": err, "rel_l2": rel, "expansion_set_equal": same, "expanded": n,
            "tolerance": {"max_abs": 1e-2, "rel_l2": 5e-3},
            "ok": bool(same and err <= 1e-2 and rel <= 5e-3)}


def cpu_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info()]
        return max(n) if n else 1
    except Exception:
        return len(os.sched_getaffinity(0))


def run_reference(args, w, ws_n, rank):
    """The oracle, as it stands, on the host cores.  Each timed sample is one
    (layer, sequence, KV head) unit of the workload (the shared unit sample);
    ms_per_step is the time of one sample, and the value is steps/s of the
    whole workload, extrapolated from the mean unit time."""
    if rank != 0:
        return
    units = oracle_units(w, min(8, args.steps + args.warmup))
    times = time_units(units, args.warmup, args.steps)
    units_per_step = w.batch * w.n_kv_heads * w.layers
    mean = float(np.mean(times))
    value = 1.0 / (mean * units_per_step)
    desc = (f"{UNITS_PER_STEP_DOC}; {args.steps} units timed after {args.warmup} warm-up, "
            f"cycling over the first {len(units)} groups of layer 0 (drawn on the CPU); steps/s "
            f"= 1 / (mean unit time x {units_per_step} units per step)")
    line = {"metric": decode_metric(w), "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean * 1e3,
            "step_is": "one (layer, sequence, KV head) unit", "units_per_step": units_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference", "config": decode_config(w, ws_n),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_threads(),
                             "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------
# main
# ----------------------------------------------------------------------------

def build_bytes(w, inp, out) -> int:
    """HBM bytes the prefill build of one layer must move: read K, V (bf16),
    the surprisal, W_r and the gates; write the full-resolution rows, the
    routing summaries, the summary keys/values, the per-span metadata and the
    basis records actually packed."""
    B, Hkv, T = w.batch, w.n_kv_heads, w.ctx
    ms = inp["max_spans"]
    n_sp = out["n_spans"].long()
    rd = 2 * B * Hkv * T * 128 * 2 + 4 * B * T + inp["W_r"].numel() * 4 + inp["gates"].size * 4
    n_full = (w.n_sink + n_sp + w.n_recent).sum().item()
    wr = Hkv * (512 * n_full + (256 + 512 + 8 + 4) * n_sp.sum().item()) + 4 * B * (1 + ms)
    rec = out["rec_rank"].long()
    body = out["body_len"].long()[:, None, :].expand_as(rec)
    valid = torch.arange(ms, device=rec.device)[None, None, :] < n_sp[:, None, None]
    recb = (gen.record_size(body, rec & 0xFFFF, (rec >> 16) & 0xFFFF) * (valid & (body > 0))).sum()
    return int(rd + wr + recb.item())


def fp32_peak_tflops(dev) -> dict:
    """fp32 arithmetic rate: a cuBLAS SGEMM (8192^3, TF32 off) timed with CUDA
    events, best of 5, and the nominal 152 SMs x 128 fma/clock x 2 x max clock."""
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    n = 8192
    a = torch.randn(n, n, device=dev)
    b = torch.randn(n, n, device=dev)
    best = 0.0
    for _ in range(5):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        torch.mm(a, b)
        e1.record()
        torch.cuda.synchronize()
        best = max(best, 2.0 * n ** 3 / (e0.elapsed_time(e1) / 1e3) / 1e12)
    torch.backends.cuda.matmul.allow_tf32 = prev
    props = torch.cuda.get_device_properties(dev)
    mhz = 2070.0
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            mhz = float(json.load(f).get("sm_max_mhz", mhz))
    except (OSError, ValueError):
        pass
    return {"measured": best,
            "nominal": props.multi_processor_count * 128 * 2 * mhz * 1e6 / 1e12}


def run_append_bench(args, ws_n, rank, local):
    """Decode-time cache maintenance at 128K (Mistral-7B shape, one layer): the
    prefill build of the first 131,072 - 1,024 tokens, then one appended token
    per step (sekv_append_token: the token joins the tail, the token leaving
    the recent window continues the segmentation walk; about one step in 32
    closes a span of every KV head) and a flush (sekv_maint_flush: the closed
    spans' summaries and gated SVD bases, their body rows leave full
    resolution) every FLUSH_EVERY steps.  Appends and flushes are CUDA graphs
    over fixed input buffers, as in a decode loop."""
    import decode_attention_span_gb300 as sk
    if not torch.cuda.is_available():
        raise SystemExit("bench.py (append) needs a CUDA device")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = synth.get_config("mistral_7b_build_128k")
    n_app, every = 1024, 64
    T0 = w.ctx - n_app
    n_sp = len(gen.sequence_spans(w, 0))
    ms = (n_sp + w.len_max + 63) // 64 * 64
    inp = gen.build_inputs(w, 0, device="cpu", max_spans=ms)
    K, V = inp["K"].to(dev), inp["V"].to(dev)
    H = torch.from_numpy(inp["H"]).to(dev)
    W = inp["W_r"].to(dev)
    gates = torch.from_numpy(inp["gates"]).to(dev)
    cfg = sk.Config(w.batch, w.n_q_heads, w.n_kv_heads, w.n_sink, w.n_recent, ms, w.rank_cap,
                    w.len_min, w.len_max, w.tau)
    ws = sk.Workspace(cfg, which=sk.sekv.SEKV_CALL_BUILD, ctx_len=w.ctx)
    out = sk.alloc_cache(cfg, 1 << 30, dev)
    K0, V0, H0 = K[:, :, :T0].contiguous(), V[:, :, :T0].contiguous(), H[:, :T0].contiguous()
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        sk.build_spans(cfg, K0, V0, H0, W, gates, out, ws, stream=stream)
        mt = sk.Maintainer(cfg, out, K0, V0, H0, T0, ws, stream=stream)
    del K0, V0
    kv = [(K[:, :, t].contiguous(), V[:, :, t].contiguous(), H[:, t].contiguous())
          for t in range(T0, w.ctx)]
    # the appends of each chunk of tokens, and the flush that closes the chunk,
    # captured as one CUDA graph (each token's inputs at their own address, as
    # a decode loop's projection would write them); the timed region replays
    # the chunks' graphs back to back
    warm = max(args.warmup, 3)
    with torch.cuda.stream(stream):
        for i in range(warm):
            mt.append(*kv[i], stream=stream)
        mt.flush(W, gates, stream=stream)
    torch.cuda.synchronize()

    def chunk_graph(i0, n, flush_every):
        gph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gph, stream=stream):
            for i in range(i0, i0 + n):
                mt.append(*kv[i], stream=stream)
                if flush_every and (i - i0 + 1) % flush_every == 0:
                    mt.flush(W, gates, stream=stream)
        return gph

    def timed(graphs):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        s0 = int(out["n_spans"][0])
        with torch.cuda.stream(stream):
            e0.record(stream)
            for gph in graphs:
                gph.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1), int(out["n_spans"][0]) - s0

    steps = min(args.steps, 512)
    steps -= steps % every
    main = [chunk_graph(warm + i0, every, every) for i0 in range(0, steps, every)]
    i = warm + steps
    g_warm = chunk_graph(i, every, every)  # replayed right before the timed region
    i += every
    g_app = chunk_graph(i, 32, 0)            # 32 appends alone (their spans wait)
    g_fl = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_fl, stream=stream):
        mt.flush(W, gates, stream=stream)   # the flush of those 32 appends
    g_imm = chunk_graph(i + 32, 128, 1)     # a flush after every append
    ws.raise_on_error()
    sk.build_flops(ws)
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    barrier(ws_n)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    timed([g_warm])  # the GPU idled while the sampler started
    ms_total, closed = timed(main)
    ck = clocks.stop()
    barrier(ws_n)
    ws.raise_on_error()
    flops = sk.build_flops(ws)
    ms_total = max_over_ranks(ms_total, ws_n)
    ms_app, _ = timed([g_app])
    ms_fl1, _ = timed([g_fl])
    ms_imm, closed_imm = timed([g_imm])
    ws.raise_on_error()
    us = ms_total * 1e3 / steps
    if rank != 0:
        return
    fp32 = fp32_peak_tflops(dev)
    alu = flops / (ms_total / 1e3) / 1e12
    line = {"metric": "decode-time cache maintenance: us per appended token (one 128K layer, "
                      "8 KV heads, a flush every 64 tokens)",
            "value": us, "unit": "us/token", "n_gpus": ws_n, "steps": steps, "warmup": warm,
            "ms_per_step": ms_total / steps, "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16 in, fp32 compute", "data": "synthetic",
            "config": {"workload": w.name, "batch": w.batch, "ctx_before": T0 + warm,
                       "kv_heads": w.n_kv_heads, "rank_cap": w.rank_cap,
                       "flush_every": every, "spans_built": closed,
                       "graph": "each chunk of 64 appends and its flush captured as one CUDA "
                                "graph; the chunks' graphs replayed back to back"},
            "append_us": ms_app * 1e3 / 32,
            "flush_us_after_32_appends": ms_fl1 * 1e3,
            "flush_after_every_append_us_per_token": ms_imm * 1e3 / 128,
            "spans_built_flushing_every_append": closed_imm,
            "roofline": {"bound": "alu", "achieved": alu, "peak": fp32["measured"],
                         "unit": "TFLOP/s", "frac": alu / fp32["measured"], "traffic": None,
                         "peak_kind": "measured fp32 (cuBLAS SGEMM, TF32 off)",
                         "flops_per_token": flops / steps,
                         "note": "latency-bound: a flush is a few short launches and one wave of "
                                 "span SVDs (16 per span: 8 KV heads x keys and values)"},
            "clocks": ck, "gpu_launches": steps + 9 * (steps // every)}
    print(json.dumps(line), flush=True)


def run_build_bench(args, ws_n, rank, local):
    """Prefill cache build at 128K (Mistral-7B shape): segmentation, summaries
    and the batched gated span SVD of every span, one layer per call.  Two
    layers of distinct inputs (1 GB of K/V) alternate, so every call streams
    from HBM."""
    import decode_attention_span_gb300 as sk
    if not torch.cuda.is_available():
        raise SystemExit("bench.py (build) needs a CUDA device")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = synth.get_config("mistral_7b_build_128k")
    inps = [gen.build_inputs(w, l, device="cpu") for l in range(2)]
    ms = max(i["max_spans"] for i in inps)
    cfg = sk.Config(w.batch, w.n_q_heads, w.n_kv_heads, w.n_sink, w.n_recent, ms, w.rank_cap,
                    w.len_min, w.len_max, w.tau)
    ws = sk.Workspace(cfg, which=sk.sekv.SEKV_CALL_BUILD, ctx_len=w.ctx)
    layers = []
    for inp in inps:
        gates = np.zeros((w.batch, w.n_kv_heads, 2, ms, w.rank_cap), np.float32)
        gates[:, :, :, :inp["gates"].shape[3]] = inp["gates"]
        layers.append(dict(K=inp["K"].to(dev), V=inp["V"].to(dev),
                           H=torch.from_numpy(inp["H"]).to(dev), W=inp["W_r"].to(dev),
                           g=torch.from_numpy(gates).to(dev), inp=inp,
                           out=sk.alloc_cache(cfg, 1 << 30, dev)))
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            L = layers[i % 2]
            sk.build_spans(cfg, L["K"], L["V"], L["H"], L["W"], L["g"], L["out"], ws, stream=stream)
    torch.cuda.synchronize()
    ws.raise_on_error()
    sk.build_flops(ws)  # clear the warm-up calls' count
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    barrier(ws_n)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(args.steps):
            L = layers[i % 2]
            sk.build_spans(cfg, L["K"], L["V"], L["H"], L["W"], L["g"], L["out"], ws, stream=stream)
        e1.record(stream)
    torch.cuda.synchronize()
    ck = clocks.stop()
    barrier(ws_n)
    ws.raise_on_error()
    flops = sk.build_flops(ws) / args.steps
    ms_total = max_over_ranks(e0.elapsed_time(e1), ws_n)
    per_call = ms_total / 1e3 / args.steps
    tokens = w.batch * w.ctx
    nbytes = sum(build_bytes(w, L["inp"], L["out"]) for L in layers) / 2
    peak, peak_kind = measured_peaks()
    achieved = nbytes / per_call / 1e9
    fp32 = fp32_peak_tflops(dev)
    alu = flops / per_call / 1e12
    if rank != 0:
        return
    line = {"metric": "prefill cache build tokens/s at 128K ctx (one layer per call)",
            "value": whole_job_rate(args.steps, ms_total, ws_n) * tokens, "unit": "tokens/s",
            "n_gpus": ws_n, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms_total / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16 in, fp32 compute", "data": "synthetic",
            "config": {"workload": w.name, "batch": w.batch, "ctx": w.ctx,
                       "kv_heads": w.n_kv_heads, "rank_cap": w.rank_cap,
                       "spans_per_head": int(np.mean([int(L["out"]["n_spans"][0]) for L in layers])),
                       "l2": "two layers of distinct inputs alternate (1 GB of K/V)"},
            "roofline": {"bound": "alu", "achieved": alu, "peak": fp32["measured"],
                         "unit": "TFLOP/s", "frac": alu / fp32["measured"], "traffic": None,
                         "peak_kind": "measured fp32 (cuBLAS SGEMM, TF32 off)",
                         "flops_per_call": flops,
                         "flops_counted": "fp32 operations the span SVDs performed (fma = 2): "
                                          "Gram matrices, the Jacobi sweeps actually run, "
                                          "projections (counted by the kernel)",
                         "fp32_nominal_tflops": fp32["nominal"],
                         "frac_of_nominal": alu / fp32["nominal"]},
            "hbm": {"achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                    "peak_kind": peak_kind, "bytes_per_call": nbytes},
            "clocks": ck, "gpu_launches": None}
    print(json.dumps(line), flush=True)


def run_multi_bench(args, ws_n, rank, local):
    """Multi-query decode at 128K (Llama-3-8B shape): --query-tokens query
    tokens per sequence over the same cache (sekv_decode_step_multi: each
    token routes and attends on its own; each (token, head) pair is a column
    of the tensor-core tiles, eight per launch, so the tokens go in blocks of
    8 / hpg, and the union of a block's expansion sets is loaded once), 32
    layers in one CUDA graph.  Reported as query tokens/s, with the one-query
    step of the same run beside it."""
    import decode_attention_span_gb300 as sk
    if not torch.cuda.is_available():
        raise SystemExit("bench.py (multi) needs a CUDA device")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = synth.get_config(args.config, **({"layers": args.layers} if args.layers else {}))
    nq = args.query_tokens
    cfg, ws, layers = build_workload(sk, w, dev, w.layers)
    B, Hkv, ms = cfg.batch, cfg.n_kv_heads, cfg.max_spans
    tpb = 8 // (w.n_q_heads // w.n_kv_heads)
    nblk = sk.query_blocks(cfg, nq)
    for l, L in enumerate(layers):
        g = gen._gen(w.seed * 4099 + 17 * l + 3, dev)
        qs = [L["q"]] + [gen.query(g, w.batch, w.n_q_heads, dev) for _ in range(nq - 1)]
        L["qm"] = torch.stack(qs, 1).contiguous()
        L["outm"] = torch.empty(w.batch, nq, w.n_q_heads, 128, device=dev)
        L["lsem"] = torch.empty(w.batch, nq, w.n_q_heads, device=dev)
        sets = []
        for i in range(nq):
            lst, cnt, _ = sk.route(cfg, L["cache"], L["qm"][:, i].contiguous(), L["W"], L["theta"], ws)
            lst, cnt = lst.view(B * Hkv, ms).cpu().numpy(), cnt.cpu().numpy()
            sets.append([set(lst[gi, :cnt[gi]].tolist()) for gi in range(B * Hkv)])
        # per launch (block of tokens): the union's factors, and the summaries
        # of every span that some token of the block does not expand
        L["bytes_m"], ucount = 0, 0
        for k in range(nblk):
            bs = sets[k * tpb:(k + 1) * tpb]
            union = [sorted(set().union(*[st[gi] for st in bs])) for gi in range(B * Hkv)]
            both = sum(len(set.intersection(*[st[gi] for st in bs])) for gi in range(B * Hkv))
            ulst = torch.zeros(B * Hkv, ms, dtype=torch.int32)
            ucnt = torch.zeros(B * Hkv, dtype=torch.int32)
            for gi, u in enumerate(union):
                ulst[gi, :len(u)] = torch.tensor(u, dtype=torch.int32)
                ucnt[gi] = len(u)
            L["bytes_m"] += (algorithmic_bytes(L["t"], ulst.to(dev), ucnt.to(dev), cfg)
                             + 512 * (int(ucnt.sum()) - both))
            ucount += int(ucnt.sum())
        L["union_frac"] = ucount / nblk / max(L["n_nonempty"], 1)
    scale = sk.default_scale()

    def step_m():
        for L in layers:
            sk.decode_step_multi(cfg, L["cache"], L["qm"], L["W"], L["theta"], scale, ws,
                                 out=L["outm"], lse=L["lsem"])

    def step_1():
        for L in layers:
            sk.decode_step(cfg, L["cache"], L["q"], L["W"], L["theta"], scale, ws,
                           out=L["out"], lse=L["lse"])

    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    ms_m, ck = time_graph(step_m, args.steps, args.warmup, torch.cuda.Stream(), ws_n, clocks)
    ms_1, _ = time_graph(step_1, args.steps, args.warmup, torch.cuda.Stream(), ws_n, None)
    ws.raise_on_error()
    ms_m = max_over_ranks(ms_m, ws_n)
    ms_1 = max_over_ranks(ms_1, ws_n)
    if rank != 0:
        return
    per_launch = ms_m / 1e3 / args.steps / (len(layers) * nblk)
    nbytes = sum(L["bytes_m"] for L in layers) / (len(layers) * nblk)
    peak, peak_kind = measured_peaks()
    achieved = nbytes / per_launch / 1e9
    line = {"metric": f"multi-query decode: query tokens/s at 128K ctx ({nq} tokens per sequence "
                      f"over one cache, {nblk} launch{'es' if nblk > 1 else ''} per layer)",
            "value": whole_job_rate(args.steps, ms_m, ws_n) * nq * w.batch, "unit": "tokens/s",
            "n_gpus": ws_n, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms_m / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "layers": len(layers), "batch": w.batch,
                       "ctx": w.ctx, "q_heads": w.n_q_heads, "kv_heads": w.n_kv_heads,
                       "query_tokens": nq, "columns": nq * w.n_q_heads // w.n_kv_heads,
                       "launches_per_layer": nblk, "tokens_per_launch": tpb,
                       "union_expand_frac": float(np.mean([L["union_frac"] for L in layers])),
                       "graph": "one CUDA graph per step, programmatic dependent launch"},
            "one_query_ms_per_step": ms_1 / args.steps,
            "one_query_tokens_per_s": whole_job_rate(args.steps, ms_1, ws_n) * w.batch,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": None, "peak_kind": peak_kind,
                         "kernel": "sekv::decode_kernel", "bytes_per_launch": nbytes,
                         "avg_launch_us": per_launch * 1e6},
            "clocks": ck, "gpu_launches": args.steps * len(layers) * nblk}
    print(json.dumps(line), flush=True)


def run_fullkv_bench(args, ws_n, rank, local):
    """Full-KV comparator at the headline shape: the same decode step over a
    cache with no spans, every one of the 128K context tokens a full-resolution
    row (n_sink = 0, n_recent = T), so one step is plain softmax attention over
    all tokens in every layer.  Layers hold distinct caches (16 GB), so every
    step streams from HBM."""
    import decode_attention_span_gb300 as sk
    if not torch.cuda.is_available():
        raise SystemExit("bench.py (fullkv) needs a CUDA device")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = synth.get_config(args.config)
    if args.layers:
        w = synth.get_config(args.config, layers=args.layers)
    T = w.ctx
    layers = []
    for l in range(w.layers):
        d = gen.full_kv_cache(w, l, T, device=dev)
        g = gen._gen(w.seed * 7919 + 101 * l + 1, dev)
        q = gen.query(g, w.batch, w.n_q_heads, dev)
        layers.append(dict(cache=sk.LayerCache({k: v for k, v in d.items()
                                                 if isinstance(v, torch.Tensor)}),
                           t=d, q=q, W=gen.routing_weights(g, w.n_kv_heads, dev).contiguous(),
                           theta=torch.zeros(w.n_q_heads, device=dev),
                           out=torch.empty(w.batch, w.n_q_heads, 128, device=dev),
                           lse=torch.empty(w.batch, w.n_q_heads, device=dev)))
    cfg = sk.Config(w.batch, w.n_q_heads, w.n_kv_heads, 0, T, layers[0]["t"]["max_spans"],
                    w.rank_cap, w.len_min, w.len_max, w.tau,
                    flags=sk.sekv.FLAG_OVERLAP_PREVIOUS)
    ws = sk.Workspace(cfg, dev)
    torch.cuda.synchronize()
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    ms_total, ck = run_resident(sk, cfg, ws, layers, args.steps, args.warmup, ws_n, clocks)
    ms_total = max_over_ranks(ms_total, ws_n)
    launch_s = ms_total / 1e3 / args.steps / w.layers
    per_launch = float(w.batch * w.n_kv_heads * T * 2 * 128 * 2)  # K and V rows, bf16
    peak, peak_kind = measured_peaks()
    achieved = per_launch / launch_s / 1e9
    if rank != 0:
        return
    line = {"metric": "full-KV decode steps/s at 128K ctx (comparator: every token a "
                      "full-resolution row)",
            "value": whole_job_rate(args.steps, ms_total, ws_n), "unit": "steps/s",
            "n_gpus": ws_n, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms_total / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name + "_fullkv", "layers": w.layers, "batch": w.batch,
                       "ctx": T, "q_heads": w.n_q_heads, "kv_heads": w.n_kv_heads,
                       "l2": "inputs larger than L2 (distinct caches per layer)",
                       "graph": "one CUDA graph per step, programmatic dependent launch"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": None, "peak_kind": peak_kind,
                         "kernel": "sekv::decode_kernel", "bytes_per_launch": per_launch,
                         "avg_launch_us": launch_s * 1e6},
            "clocks": ck, "gpu_launches": args.steps * w.layers}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.traffic_from:
        write_traffic(args.traffic_from, args.traffic_workload, args.traffic_scale,
                      args.traffic_command)
        return
    ws_n, rank, local = dist_setup(args)
    if args.impl == "reference" and args.path != "decode":
        if rank == 0:
            print(json.dumps({"impl": "reference", "unavailable": "the reference arm (the oracle) "
                              "is timed on the decode path only"}), flush=True)
        return
    if args.path == "append":
        return run_append_bench(args, ws_n, rank, local)
    if args.path == "multi":
        return run_multi_bench(args, ws_n, rank, local)
    if args.path == "build":
        run_build_bench(args, ws_n, rank, local)
        return
    if args.path == "fullkv":
        run_fullkv_bench(args, ws_n, rank, local)
        return
    if args.path == "e2e":
        return run_e2e_bench(args, ws_n, rank, local)
    w = synth.get_config(args.config)
    if args.layers:
        w = synth.get_config(args.config, layers=args.layers)
    if args.impl == "reference":
        run_reference(args, w, ws_n, rank)
        return
    import decode_attention_span_gb300 as sk
    if not torch.cuda.is_available():
        raise SystemExit("bench.py (sekv) needs a CUDA device")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    cfg, ws, layers = build_workload(sk, w, dev, w.layers)
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    ms_total, ck = run_resident(sk, cfg, ws, layers, args.steps, args.warmup, ws_n, clocks)
    ms_total = max_over_ranks(ms_total, ws_n)
    ms_step = ms_total / args.steps
    value = whole_job_rate(args.steps, ms_total, ws_n)
    bytes_step = sum(L["bytes"] for L in layers)
    per_launch = bytes_step / len(layers)
    launch_s = ms_total / 1e3 / (args.steps * len(layers))
    peak, peak_kind = measured_peaks()
    achieved = per_launch / launch_s / 1e9
    line = {"metric": decode_metric(w), "value": value, "unit": UNIT, "n_gpus": ws_n,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": decode_config(w, ws_n),
            "workload_stats": {"expand_frac": sum(L["n_exp"] for L in layers) /
                               max(1, sum(L["n_nonempty"] for L in layers)),
                               "gb_touched_per_step": bytes_step / 1e9},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": profiled_traffic(w.name),
                         "peak_kind": peak_kind, "kernel": "sekv::decode_kernel",
                         "bytes_per_launch": per_launch,
                         "avg_launch_us": launch_s * 1e6},
            "clocks": ck, "gpu_launches": args.steps * len(layers)}
    if not args.no_e2e:
        e_steps = max(16, args.steps // 4)
        line["e2e"], launches = e2e_leg(sk, cfg, w, layers, e_steps, args.warmup, ws_n, dev)
        line["gpu_launches"] += e_steps * launches
    if not args.no_cpu_baseline and rank == 0:
        line["cpu_baseline"] = cpu_baseline_leg(w, args.cpu_seconds)
        line["parity"] = parity_check(sk, cfg, ws, layers[0], w)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws_n > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
