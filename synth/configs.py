"""The synthetic workloads (shapes of the backbones the SeKV pages evaluate).

The pages evaluate on LongBench, RULER, InfiniteBench and needle-in-a-haystack
with Llama-3, Mistral and Qwen backbones; none of those suites or weights is
used.  Seeded synthetic inputs with the same context lengths and attention
shapes stand in for them.
"""

from __future__ import annotations

import dataclasses


@dataclasses.dataclass(frozen=True)
class WorkloadConfig:
    name: str
    layers: int
    batch: int
    n_q_heads: int
    n_kv_heads: int
    ctx: int
    n_sink: int
    n_recent: int
    tau: float
    len_min: int
    len_max: int
    rank_cap: int
    rank_lo: int
    expand_frac: float       # target union expansion fraction per KV head
    seed: int
    unit_gates: bool = False  # g == 1 (rank = min(rank_cap, body))
    true_rank: int = 0        # fixed generator rank (0: per-span U{rank_lo..rank_cap})
    head_dim: int = 128
    route_dim: int = 64

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads


CONFIGS = {
    # one layer, 4K context, full pipeline (tokens -> build -> route -> attend)
    "pr1": WorkloadConfig("pr1", layers=1, batch=1, n_q_heads=32, n_kv_heads=8,
                          ctx=4096, n_sink=4, n_recent=64, tau=4.0, len_min=4,
                          len_max=256, rank_cap=16, rank_lo=16, expand_frac=0.10,
                          seed=0, unit_gates=True, true_rank=8),
    # Llama-3-8B decode shape at 32K
    "llama3_8b_32k": WorkloadConfig("llama3_8b_32k", layers=32, batch=1, n_q_heads=32,
                                    n_kv_heads=8, ctx=32768, n_sink=4, n_recent=128,
                                    tau=5.2, len_min=4, len_max=256, rank_cap=32,
                                    rank_lo=4, expand_frac=0.10, seed=1),
    # headline: same shape at 128K, about 5% of spans expanded
    "llama3_8b_128k": WorkloadConfig("llama3_8b_128k", layers=32, batch=1, n_q_heads=32,
                                     n_kv_heads=8, ctx=131072, n_sink=4, n_recent=128,
                                     tau=5.2, len_min=4, len_max=256, rank_cap=32,
                                     rank_lo=4, expand_frac=0.05, seed=2),
    # Qwen2-7B-shaped stress: group 7, batch 16, heavier span tail, 30% expanded
    "qwen2_7b_stress": WorkloadConfig("qwen2_7b_stress", layers=28, batch=16,
                                      n_q_heads=28, n_kv_heads=4, ctx=65536, n_sink=4,
                                      n_recent=128, tau=6.1, len_min=4, len_max=512,
                                      rank_cap=64, rank_lo=4, expand_frac=0.30, seed=3),
    # prefill cache build at 128K, Mistral-7B shape
    "mistral_7b_build_128k": WorkloadConfig("mistral_7b_build_128k", layers=32, batch=1,
                                            n_q_heads=32, n_kv_heads=8, ctx=131072,
                                            n_sink=4, n_recent=128, tau=5.2, len_min=4,
                                            len_max=256, rank_cap=32, rank_lo=4,
                                            expand_frac=0.05, seed=4),
}


def get_config(name: str, **overrides) -> WorkloadConfig:
    cfg = CONFIGS[name]
    return dataclasses.replace(cfg, **overrides) if overrides else cfg
