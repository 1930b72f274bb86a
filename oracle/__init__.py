"""Plain CPU oracle of the per-layer n-gram embedding (PLE / Engram) path.

TEST INFRASTRUCTURE, NOT PRODUCT CODE. Only the test-suite, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import it. The
CUDA library never links, imports or calls anything here, and nothing here
imports the CUDA library or its Python binding: the two sides share no code.

What it computes, step by step, and where the pages fix it (page titles are
abbreviated as "PR#<number> report" / "PR#53899 page"):

* ``ngram_ids``   -- ragged n-gram hash IDs. PR#54517 report ("Fuse Qwen4Exp
  PLE kernels"), section 关键源码片段: the CPU branch of ``compute_ngram_ids``
  (EOS-filled per-request rows, request found by a right-sided search of
  ``query_start_loc``, both clamps) and the skeleton of
  ``_ple_ngram_ids_kernel`` (walk back over the context, EOS crossing, XOR mix
  of token*multiplier, per-head reduction, int64 semantics of
  ``torch.remainder``).
* ``lookup_bf16`` / ``lookup_fp8`` -- the multi-head row gather, PR#54371
  report ("Support UVA PLE-offload ..."), section 实现拆解 item 1 and the
  ``start_prefetch`` snippet (``F.embedding(ngram_ids, weight)``); fp8 rows
  with a scale, same section (BF16 / FP8 weight methods) and PR#53899 page
  (FP8 PLE table with ``weight_scale``).
* ``kv_proj`` -- the merged key/value projection, PR#54517 report, 实现拆解
  item 1 (``key_proj`` and ``value_proj`` merged into ``kv_proj``).
* ``gate`` -- RMSNorm + sigmoid gate ("PLE gating and normalisation"),
  PR#54517 report, 实现拆解 item 2.
* ``conv`` / ``gate_conv`` -- the dilated causal depthwise short conv,
  PR#54517 report, 实现拆解 items 2 and 5.

Precision: integers are Python ints (exact), reduced to int64 wrap-around only
where the method's int64 arithmetic wraps. Floating point is float64; bf16
values are carried as uint16 bit patterns and decoded exactly.

Parity pins: every function is pinned by ``tests/test_oracle_*.py`` to things
other than itself (hand-worked golden values, brute force, closed forms,
library routines on the CPU). Functions without such a pin say
"parity unpinned" in their docstring; the gate formula's choice of reading and
the conv orientation are the pages' silent points (see the docstrings).
"""

from .numerics import (
    bf16_bits_to_f64,
    f64_to_bf16_bits,
    e4m3_code_to_float,
    E4M3_VALUES,
)
from .ngram_ids import request_spans, ngram_ids
from .lookup import lookup_bf16, lookup_fp8
from .layer import kv_proj, gate, conv, gate_conv, layer_forward

__all__ = [
    "bf16_bits_to_f64",
    "f64_to_bf16_bits",
    "e4m3_code_to_float",
    "E4M3_VALUES",
    "request_spans",
    "ngram_ids",
    "lookup_bf16",
    "lookup_fp8",
    "kv_proj",
    "gate",
    "conv",
    "gate_conv",
    "layer_forward",
]
