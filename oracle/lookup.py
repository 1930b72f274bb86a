"""Oracle for the multi-head row gather (``F.embedding`` over the PLE table).

TEST INFRASTRUCTURE (see the package docstring).

Source: PR#54371 report ("Support UVA PLE-offload ..."), section 关键源码片段,
``Qwen4ExpPLEPinnedHostEmbedding.start_prefetch``: the rows of the table named
by ``ngram_ids`` are gathered with ``F.embedding``; the device-resident and
the pinned-host (UVA) backends read the same rows and differ only in where the
table lives, so one oracle serves both. The table is one concatenated
``[sum_h V_h, D]`` array and the ids already carry the head offsets
(PR#54517 report, skeleton of ``_ple_ngram_ids_kernel``: "map into the
embedding-table partition"). Head h of token t fills columns
``[h*D, (h+1)*D)`` of output row t.

fp8 tables (PR#54371 report 实现拆解 item 1, BF16/FP8 weight methods; PR#53899
page, FP8 table with ``weight_scale``): each e4m3 code is decoded exactly,
multiplied in float32 by its row's float32 scale (one IEEE product, nearest
even), and the product is rounded to bf16 (nearest even). The pages show one
global ``weight_scale``; a per-row scale is the general case (a global scale is
every row carrying the same value).
"""

import numpy as np

from .numerics import E4M3_VALUES, f64_to_bf16_bits


def lookup_bf16(ids, table_bits):
    """Gather bf16 rows.

    Args:
      ids: [T, H] integer row indices into ``table_bits``.
      table_bits: [rows, D] uint16 (bf16 bit patterns).
    Returns:
      [T, H*D] uint16, a bit-exact copy of the named rows.
    """
    ids = np.asarray(ids, dtype=np.int64)
    T, H = ids.shape
    rows, D = table_bits.shape
    out = np.empty((T, H * D), dtype=np.uint16)
    for t in range(T):
        for h in range(H):
            row = int(ids[t, h])
            assert 0 <= row < rows, "id out of range"
            out[t, h * D:(h + 1) * D] = table_bits[row]
    return out


def lookup_fp8(ids, table_codes, row_scale):
    """Gather fp8 e4m3 rows and dequantise them to bf16.

    Args:
      ids: [T, H] integer row indices.
      table_codes: [rows, D] uint8 e4m3 codes.
      row_scale: [rows] float32 scale of each row.
    Returns:
      [T, H*D] uint16 bf16 bits of round_bf16(float32(value) * scale[row]).
    """
    ids = np.asarray(ids, dtype=np.int64)
    T, H = ids.shape
    rows, D = table_codes.shape
    scale = np.asarray(row_scale, dtype=np.float32)
    out = np.empty((T, H * D), dtype=np.uint16)
    for t in range(T):
        for h in range(H):
            row = int(ids[t, h])
            assert 0 <= row < rows, "id out of range"
            values = E4M3_VALUES[table_codes[row]]          # float32, exact
            product = values * np.float32(scale[row])       # one float32 product
            out[t, h * D:(h + 1) * D] = f64_to_bf16_bits(product.astype(np.float64))
    return out
