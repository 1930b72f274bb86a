"""The C ABI: libple builds, loads and exports what include/ple.h declares;
host-side argument checks reject bad calls before any CUDA work (no GPU)."""

import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ple.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ple_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from hashed_gram_embedding_gb300 import build, _lib
    build.build()
    return _lib.lib()


def test_header_declares_the_path():
    names = declared_functions()
    for required in ["ple_ngram_ids", "ple_lookup", "ple_lookup_prefetch", "ple_wait",
                     "ple_kv_proj", "ple_gate", "ple_conv", "ple_gate_conv",
                     "ple_last_error", "ple_version"]:
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    from hashed_gram_embedding_gb300 import _lib
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, f"binding lacks {name}"


def test_version_string(lib):
    assert b"libple" in lib.ple_version()


def _ngram(lib, **kw):
    args = dict(input_ids=None, T=4, qsl=None, R=1, ctx=None, ctx_len=2, mult=[1, 2, 3],
                V=[7, 11], O=[0, 7], eos=2, hpn=1, out=None, ctx_out=None, err=None)
    args.update(kw)
    I64P = ctypes.POINTER(ctypes.c_int64)
    keep = [np.asarray(args[k], dtype=np.int64) for k in ("mult", "V", "O")]
    return lib.ple_ngram_ids(args["input_ids"], args["T"], args["qsl"], args["R"], args["ctx"],
                             args["ctx_len"], *(a.ctypes.data_as(I64P) for a in keep),
                             args["eos"], args["hpn"], args["out"], args["ctx_out"], args["err"],
                             None)


def test_ngram_ids_rejects_empty_head_shard(lib):
    assert _ngram(lib, hpn=0) == 1
    assert b"empty head" in lib.ple_last_error()


def test_ngram_ids_rejects_bad_sizes(lib):
    assert _ngram(lib, ctx_len=0, mult=[1]) == 1
    assert _ngram(lib, ctx_len=8, mult=[1] * 9, V=[7] * 8, O=[0] * 8) == 1
    assert _ngram(lib, R=0) == 1                       # tokens but no request
    assert _ngram(lib, V=[7, 0]) == 1                  # empty vocab
    assert _ngram(lib, hpn=40, V=[7] * 80, O=[0] * 80) == 1  # too many heads
    assert _ngram(lib, T=-1) == 1


def test_ngram_ids_zero_tokens_is_a_noop(lib):
    assert _ngram(lib, T=0) == 0


def test_ngram_ids_rejects_overlapping_context_buffers(lib):
    buf = (ctypes.c_int32 * 8)()
    p = ctypes.addressof(buf)
    assert _ngram(lib, ctx=p, ctx_out=p + 4, R=2, T=0) == 1
    assert b"overlaps" in lib.ple_last_error()


def test_lookup_rejects_unaligned_rows_and_bad_enums(lib):
    # 12 bf16 = 24 bytes per row: not a multiple of 16
    assert lib.ple_lookup(None, 1, 1, None, 10, 12, 0, None, 0, None, 0, None, None) == 2
    assert lib.ple_lookup(None, 1, 1, None, 10, 64, 7, None, 0, None, 0, None, None) == 1
    assert lib.ple_lookup(None, 1, 1, None, 10, 64, 0, None, 9, None, 0, None, None) == 1
    assert lib.ple_lookup(None, 1, 0, None, 10, 64, 0, None, 0, None, 0, None, None) == 1
    assert lib.ple_lookup(None, 0, 1, None, 10, 64, 0, None, 0, None, 0, None, None) == 0
    # fp8 without scales
    assert lib.ple_lookup(ctypes.c_void_p(16), 1, 1, ctypes.c_void_p(16), 10, 64, 1, None, 0,
                          ctypes.c_void_p(16), 0, None, None) == 1


def test_kv_proj_rejects_unsupported_shapes(lib):
    assert lib.ple_kv_proj(None, None, 4, 12, 64, None, None, None) == 2   # E % 8
    assert lib.ple_kv_proj(None, None, 4, 64, 24, None, None, None) == 2   # C % 16
    assert lib.ple_kv_proj(None, None, 0, 64, 64, None, None, None) == 0


def test_conv_and_gate_reject_bad_shapes(lib):
    assert lib.ple_gate(None, None, None, None, 1e-6, 4, 12, None, None, None) == 1
    assert lib.ple_conv(None, None, 1, 4, 64, None, 9, 1, None, None, None, None, None) == 1
    assert lib.ple_conv(None, None, 1, 4, 64, None, 4, 30, None, None, None, None, None) == 1
    assert lib.ple_gate_conv(None, None, None, None, 1e-6, None, 0, 4, 64, None, 4, 3, None,
                             None, None, None, None, None) == 1


def test_gate_rejects_hidden_above_limit(lib):
    assert lib.ple_gate(None, None, None, None, 1e-6, 4, 16392, None, None, None) == 2
    assert b"16384" in lib.ple_last_error()


def test_ordered_gather_workspace_size(lib):
    # 32 GiB bf16 table, D = 128 (256-byte rows): one bucket per 2 MiB span =
    # 8192 rows, ceil(134219512 / 8192) = 16385 spans + 1 bucket for ids outside
    # the table; counts and cursors (4 bytes per bucket) and the walk order
    # (4 bytes per item), each rounded up to 256 bytes.
    up = lambda x: (x + 255) // 256 * 256
    buckets = 16385 + 1
    want = 2 * up(4 * buckets) + up(4 * 8192 * 16)
    assert lib.ple_lookup_ordered_workspace(8192, 16, 134219512, 128, 0) == want
    # fp8 rows of 128 bytes: 16384 rows per 2 MiB span
    buckets = -(-67110742 // 16384) + 1
    assert lib.ple_lookup_ordered_workspace(100, 16, 67110742, 128, 1) == \
        2 * up(4 * buckets) + up(4 * 1600)
    assert lib.ple_lookup_ordered_workspace(-1, 16, 10, 128, 0) == 0
    # one scale for the whole fp8 table: the same 128-byte rows as per-row fp8
    assert lib.ple_lookup_ordered_workspace(100, 16, 67110742, 128, 2) == \
        lib.ple_lookup_ordered_workspace(100, 16, 67110742, 128, 1)
    assert lib.ple_lookup_ordered_workspace(100, 16, 67110742, 128, 3) == 0  # no such dtype


def test_wait_rejects_null_event(lib):
    assert lib.ple_wait(None, None, 0) == 1


def test_gate_conv_requires_gate_out(lib):
    p = ctypes.c_void_p(256)  # never dereferenced: the call fails on the host first
    assert lib.ple_gate_conv(p, p, p, p, 1e-6, p, 1, 4, 64, p, 4, 3, None, None, p, None, None,
                             None) == 1
    assert b"gate_out" in lib.ple_last_error()


def test_host_table_rejects_zero_bytes(lib):
    out = ctypes.c_void_p()
    assert lib.ple_host_table_alloc(0, ctypes.byref(out)) == 1
    assert lib.ple_host_table_free(None, 0) == 0


def test_kv_proj_gate_workspace_size(lib):
    # partial sums: 16 bytes per token and 128-channel key block; counters at
    # the end: 4 bytes per 32 of the B/16 tokens a B-byte buffer could ever
    # hold; B the smallest multiple of 256 with room for both. 8192 x 4096:
    # 4 MiB of partials; B = 4227584 holds 8257 counters (33028 bytes) and
    # 4194304 + 33028 <= 4227584 < 4194304 + 33028 + 256.
    assert lib.ple_kv_proj_gate_workspace(8192, 4096) == 4227584
    assert lib.ple_kv_proj_gate_workspace(1, 256) == 256      # 32 + 4 bytes
    assert lib.ple_kv_proj_gate_workspace(33, 768) == 3328    # 3168 + 7 * 4
    counters = lambda B: (B // 16 + 31) // 32 * 4
    prev = 0
    for M in (1, 2, 31, 32, 33, 100, 1000, 4097, 65536):
        for C in (256, 1024, 4096):
            B = lib.ple_kv_proj_gate_workspace(M, C)
            part = C // 128 * M * 16
            assert B % 256 == 0 and part + counters(B) <= B < part + counters(B) + 256
        assert B >= prev
        prev = B
    for bad in ((100, 264), (100, 0), (0, 256), (-5, 256)):
        assert lib.ple_kv_proj_gate_workspace(*bad) == 0


def test_kv_proj_gate_host_checks(lib):
    p = ctypes.c_void_p(256)  # never dereferenced: every call fails on the host first
    ws = lib.ple_kv_proj_gate_workspace(64, 512)
    # hidden not a multiple of 256
    assert lib.ple_kv_proj_gate(p, p, 64, 64, 264, p, p, p, 1e-6, p, p, p, 1 << 20, None,
                                None) == 2
    # room for the partial sums but not the counters, then misaligned
    assert lib.ple_kv_proj_gate(p, p, 64, 64, 512, p, p, p, 1e-6, p, p, p, 4 * 64 * 16, None,
                                None) == 1
    assert b"workspace" in lib.ple_last_error()
    assert lib.ple_kv_proj_gate(p, p, 64, 64, 512, p, p, p, 1e-6, p, p, ctypes.c_void_p(272),
                                ws, None, None) == 1
    # gate_out missing
    assert lib.ple_kv_proj_gate(p, p, 64, 64, 512, p, p, p, 1e-6, p, None, p, ws, None,
                                None) == 1
    # no tokens: nothing to do
    assert lib.ple_kv_proj_gate(None, None, 0, 64, 512, None, None, None, 1e-6, None, None,
                                None, 0, None, None) == 0


def _ngram_lookup(lib, **kw):
    p = ctypes.c_void_p(256)  # never dereferenced: every case fails on the host first
    args = dict(input_ids=p, T=4, qsl=p, R=1, ctx=None, ctx_len=2, mult=[1, 2, 3], V=[7, 11],
                O=[0, 7], eos=2, hpn=1, table=p, rows=18, D=64, dtype=0, scale=None, loc=0,
                out=p, ids_out=None, ctx_out=None)
    args.update(kw)
    I64P = ctypes.POINTER(ctypes.c_int64)
    keep = [np.asarray(args[k], dtype=np.int64) for k in ("mult", "V", "O")]
    return lib.ple_ngram_lookup(args["input_ids"], args["T"], args["qsl"], args["R"], args["ctx"],
                                args["ctx_len"], *(a.ctypes.data_as(I64P) for a in keep),
                                args["eos"], args["hpn"], args["table"], args["rows"], args["D"],
                                args["dtype"], args["scale"], args["loc"], args["out"],
                                args["ids_out"], args["ctx_out"], 0, None, None)


def test_ngram_lookup_host_checks(lib):
    assert _ngram_lookup(lib, hpn=0) == 1                      # empty head shard
    assert b"empty head" in lib.ple_last_error()
    assert _ngram_lookup(lib, O=[0, 8]) == 1                   # head 1's partition past row 18
    assert b"outside" in lib.ple_last_error()
    assert _ngram_lookup(lib, O=[-1, 7]) == 1
    assert _ngram_lookup(lib, R=0) == 1                        # tokens but no request
    assert _ngram_lookup(lib, T=-1) == 1
    assert _ngram_lookup(lib, D=12) == 2                       # 24-byte rows
    assert _ngram_lookup(lib, dtype=7) == 1                    # no such table type
    assert _ngram_lookup(lib, dtype=1) == 1                    # fp8 without a scale
    buf = (ctypes.c_int32 * 8)()
    a = ctypes.addressof(buf)
    assert _ngram_lookup(lib, ctx=a, ctx_out=a + 4, R=2, T=0) == 1
    assert b"overlaps" in lib.ple_last_error()


def test_gated_conv_host_checks(lib):
    p = ctypes.c_void_p(256)
    # K = 9 is above the largest filter; dilation 30 with K = 4 exceeds the halo
    assert lib.ple_gated_conv(p, p, p, 1, 4, 64, p, 9, 1, None, None, p, None, None) == 1
    assert lib.ple_gated_conv(p, p, p, 1, 4, 64, p, 4, 30, None, None, p, None, None) == 1
    assert lib.ple_gated_conv(None, p, p, 1, 4, 64, p, 4, 3, None, None, p, None, None) == 1
    assert lib.ple_gated_conv(p, None, p, 1, 4, 64, p, 4, 3, None, None, p, None, None) == 1
    assert lib.ple_gated_conv(p, p, p, 1, 4, 12, p, 4, 3, None, None, p, None, None) == 1


def test_step_runtime_host_checks(lib):
    """The step runtime rejects missing or repeated streams, null events or
    graphs and malformed copy lists before any CUDA call; destroying NULL
    handles is a no-op."""
    from hashed_gram_embedding_gb300 import _lib
    s1, s2, s3, ev = (ctypes.c_void_p(v) for v in (16, 32, 48, 64))
    up = _lib.copies([(256, 512, 64)])
    bad = _lib.copies([(None, 512, 64)])
    assert lib.ple_step(None, s2, s3, up, 1, ev, up, 1, ev, ev, ev) == 1   # legacy stream
    assert lib.ple_step(s1, s1, s3, up, 1, ev, up, 1, ev, ev, ev) == 1    # repeated stream
    assert lib.ple_step(s1, s2, s3, up, 1, None, up, 1, ev, ev, ev) == 1  # no graph
    assert b"null graph" in lib.ple_last_error()
    assert lib.ple_step(s1, s2, s3, up, 1, ev, up, 1, ev, None, ev) == 1  # null event
    assert lib.ple_step(s1, s2, s3, bad, 1, ev, up, 1, ev, ev, ev) == 1   # null pointer
    assert b"copy 0" in lib.ple_last_error()
    assert lib.ple_step(s1, s2, s3, up, -1, ev, up, 1, ev, ev, ev) == 1   # negative count
    assert lib.ple_step(s1, s2, s3, None, 1, ev, up, 1, ev, ev, ev) == 1  # missing list
    assert lib.ple_step_begin(s1, s1, up, 1, ev, ev, ev) == 1
    assert lib.ple_step_begin(s1, s2, bad, 1, ev, ev, ev) == 1
    assert lib.ple_step_end(s2, s2, up, 1, ev, ev) == 1
    assert lib.ple_step_end(s2, s3, up, 1, None, ev) == 1
    assert lib.ple_step_end(s2, s3, bad, 1, ev, ev) == 1
    assert lib.ple_graph_launch(None, s1) == 1
    assert lib.ple_graph_begin(None) == 1
    assert lib.ple_graph_end(None, None) == 1
    assert lib.ple_event_create(None) == 1
    assert lib.ple_event_synchronize(None) == 1
    lib.ple_graph_destroy(None)
    lib.ple_event_destroy(None)


def test_lookup_shard_host_checks(lib):
    P = ctypes.c_void_p(16)
    # head range outside the ids' columns, empty head range, negative base
    assert lib.ple_lookup_shard(P, 4, 8, 6, 4, P, 10, 0, 64, 0, None, 0, 0, P, None, 0, None,
                                None) == 1
    assert lib.ple_lookup_shard(P, 4, 8, 0, 0, P, 10, 0, 64, 0, None, 0, 0, P, None, 0, None,
                                None) == 1
    assert lib.ple_lookup_shard(P, 4, 8, 0, 8, P, 10, -1, 64, 0, None, 0, 0, P, None, 0, None,
                                None) == 1
    # unknown shard kind; 24-byte rows
    assert lib.ple_lookup_shard(P, 4, 8, 0, 8, P, 10, 0, 64, 0, None, 0, 5, P, None, 0, None,
                                None) == 1
    assert lib.ple_lookup_shard(P, 4, 8, 0, 8, P, 10, 0, 12, 0, None, 0, 0, P, None, 0, None,
                                None) == 2
    # fp8 without a scale; an fp8 row shard without scale_out
    assert lib.ple_lookup_shard(P, 4, 8, 0, 8, P, 10, 0, 64, 1, None, 0, 0, P, None, 0, None,
                                None) == 1
    assert lib.ple_lookup_shard(P, 4, 8, 0, 8, P, 10, 0, 64, 1, P, 0, 1, P, None, 0, None,
                                None) == 1
    assert b"scale_out" in lib.ple_last_error()
    # no tokens: nothing to do
    assert lib.ple_lookup_shard(None, 0, 8, 0, 8, None, 10, 0, 64, 0, None, 0, 0, None, None, 0,
                                None, None) == 0


def test_select_rows_host_checks(lib):
    I32P = ctypes.POINTER(ctypes.c_int32)

    def call(T=4, H=2, part=(0, 1), col=(0, 1), r0=0, rows=10, parts=2, ph=2, D=64, dtype=0):
        p = np.asarray(part, dtype=np.int32)
        c = np.asarray(col, dtype=np.int32)
        return lib.ple_select_rows(ctypes.c_void_p(16), parts, rows, ph, None, r0, T, H,
                                   p.ctypes.data_as(I32P), c.ctypes.data_as(I32P), D, dtype,
                                   ctypes.c_void_p(16), None)

    assert call(r0=8) == 1                      # window past the rows
    assert call(part=(0, 2)) == 1               # part outside
    assert call(col=(0, 2)) == 1                # column outside
    assert call(H=65, part=[0] * 65, col=[0] * 65) == 2   # too many heads
    assert call(D=12) == 2                      # 24-byte bf16 rows
    assert call(dtype=1) == 1                   # fp8 without scales
    assert call(T=0) == 0                       # no tokens
