"""GB300 (sm_103a) implementation of SeKV's span-cache decode path.

The compute runs in libsekv (CUDA kernels behind a C ABI, ``include/sekv.h``);
``decode_attention_span_gb300.sekv`` is its ctypes binding.
"""

from . import sekv  # noqa: F401
from .sekv import (  # noqa: F401
    Config,
    LayerCache,
    Workspace,
    SekvError,
    route,
    decode_attention,
    decode_step,
    decode_step_multi,
    query_blocks,
    decode_step_noalloc,
    fetch_bases,
    fetch_bases_copy,
    fetch_bases_cached,
    BasisCache,
    build_spans,
    build_flops,
    Maintainer,
    alloc_cache,
    record_size,
    last_launch_count,
    default_scale,
)
