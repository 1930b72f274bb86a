"""GB300-native per-layer n-gram embedding (PLE / Engram) lookup path.

The compute path is libple.so (hand-written CUDA for sm_103a, C ABI in
include/ple.h); this package holds its build script, a ctypes binding with
the C names, the PLELayer convenience wrapper (and PLEHostPipeline, which
runs it over pinned host buffers with transfers overlapping compute; PLEChain,
several layers with the next layers' lookups prefetched), the sharded lookups
over a group of ranks (HeadShardedLookup, RowShardedLookup) and the seeded
synthetic workloads used by the tests and the benchmark.
"""

from ._lib import (  # noqa: F401
    PleError,
    ple_ngram_ids,
    ple_lookup,
    ple_lookup_prefetch,
    ple_lookup_ordered,
    ple_lookup_ordered_workspace,
    ple_lookup_ordered_static,
    ple_wait,
    ple_kv_proj,
    ple_gate,
    ple_conv,
    ple_gate_conv,
    ple_lookup_shard,
    ple_select_rows,
    ple_version,
    PLE_DEVERR_BOUNDS,
    PLE_DEVERR_QSL,
    PLE_DEVERR_TIMEOUT,
    PLE_HBM,
    PLE_HOST_UVA,
    PLE_SHARD_HEADS,
    PLE_SHARD_ROWS,
)
from .layer import PLELayer, PLEHostPipeline, PLEChain  # noqa: F401
from .sharded import HeadShardedLookup, RowShardedLookup  # noqa: F401
