"""Plain, slow, fp64 CPU oracle for the SeKV span-cache decode path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product package imports this
package; only the test-suite, the smoke check in ``__graft_entry__`` and the
CPU-baseline leg of ``bench.py`` may call it.  It shares no code with the CUDA
path: it has its own reader and writer of the C-ABI byte layouts
(``oracle.layout``) and does every step with numpy in float64.

Sources (cited in every function as "page, section"):

* [DE] "SeKV: Resolution-Adaptive KV Cache with Hierarchical Semantic Memory
  for Long-Context LLM Inference", gist.science (German explainer),
  section "Technisches Resuemee": Methodik 1 (segmentation), 2 (dual
  representation), 3 (zoom-in and mixed-resolution attention); and its lay
  explainer, part 2 ("Der Zwei-Ebenen-Speicher").
* [ZH] the same paper on gist.science (Chinese explainer), section
  "技术摘要": 方法论 1, 2, 3; and its lay explainer, part 2 ("两层记忆").
* [EN] the paper's English abstract (chatpaper.ai page).

Parity status per function is listed in each docstring; every function here is
pinned by a CPU test in ``tests/test_oracle_*.py`` against a property that
the pages or the mathematics fix (brute force, closed forms, reductions to
textbook attention), never against a retyped copy of itself.
"""

from .sekv_oracle import (  # noqa: F401
    bf16_round,
    regions,
    segment,
    routing_summary,
    attention_summary,
    span_svd,
    build_span,
    build_layer,
    route,
    route_logits,
    decode_attention,
    full_attention,
    reconstruct,
    LayerCache,
    SpanFactors,
)
