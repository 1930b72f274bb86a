"""ctypes binding of libple (the C ABI declared in include/ple.h).

Argument marshalling only: every step of the path runs in libple's CUDA
kernels. Functions take torch tensors for device buffers (their data
pointers are passed through) and raise PleError on a non-OK status. There is
no fallback: if libple.so is missing the first call raises.
"""

import ctypes
import os

import numpy as np

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libple.so")

PLE_OK = 0
PLE_ERR_INVALID_ARG = 1
PLE_ERR_UNSUPPORTED = 2
PLE_ERR_CUDA = 3
PLE_ERR_TIMEOUT = 4
PLE_ERR_BOUNDS = 5
STATUS_NAMES = {0: "PLE_OK", 1: "PLE_ERR_INVALID_ARG", 2: "PLE_ERR_UNSUPPORTED",
                3: "PLE_ERR_CUDA", 4: "PLE_ERR_TIMEOUT", 5: "PLE_ERR_BOUNDS"}

PLE_DEVERR_BOUNDS = 1
PLE_DEVERR_QSL = 2
PLE_DEVERR_TIMEOUT = 4

PLE_BF16 = 0
PLE_FP8_E4M3 = 1
PLE_FP8_E4M3_TENSOR = 2
PLE_HBM = 0
PLE_HOST_UVA = 1
PLE_SHARD_HEADS = 0
PLE_SHARD_ROWS = 1
PLE_HOST_TABLE_REGISTER = 1

# Every entry point of include/ple.h with its ctypes signature.
_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_F32 = ctypes.c_float
_I64P = ctypes.POINTER(ctypes.c_int64)
_I32P = ctypes.POINTER(ctypes.c_int32)
SIGNATURES = {
    "ple_ngram_ids": [_P, _I64, _P, _I32, _P, _I32, _I64P, _I64P, _I64P, _I32, _I32, _P, _P, _P, _P],
    "ple_lookup": [_P, _I64, _I32, _P, _I64, _I32, ctypes.c_int, _P, ctypes.c_int, _P, _I32, _P, _P],
    "ple_ngram_lookup": [_P, _I64, _P, _I32, _P, _I32, _I64P, _I64P, _I64P, _I32, _I32, _P, _I64,
                         _I32, ctypes.c_int, _P, ctypes.c_int, _P, _P, _P, _I32, _P, _P],
    "ple_lookup_prefetch": [_P, _I64, _I32, _P, _I64, _I32, ctypes.c_int, _P, ctypes.c_int, _P, _I32,
                            _P, _P, _P],
    "ple_lookup_ordered_workspace": [_I64, _I32, _I64, _I32, ctypes.c_int],
    "ple_lookup_ordered": [_P, _I64, _I32, _P, _I64, _I32, ctypes.c_int, _P, ctypes.c_int, _P, _I32,
                           _P, ctypes.c_size_t, _P, _P],
    "ple_lookup_ordered_static": [_P, _I64, _I32, _P, _I64, _I32, ctypes.c_int, _P, ctypes.c_int, _P,
                                  _I32, _P, _P],
    "ple_lookup_shard": [_P, _I64, _I32, _I32, _I32, _P, _I64, _I64, _I32, ctypes.c_int, _P,
                         ctypes.c_int, ctypes.c_int, _P, _P, _I32, _P, _P],
    "ple_select_rows": [_P, _I32, _I64, _I32, _P, _I64, _I64, _I32, _I32P, _I32P, _I32,
                        ctypes.c_int, _P, _P],
    "ple_wait": [_P, _P, _I32],
    "ple_kv_proj": [_P, _P, _I64, _I32, _I32, _P, _P, _P],
    "ple_kv_proj_gate_workspace": [_I64, _I32],
    "ple_kv_proj_gate": [_P, _P, _I64, _I32, _I32, _P, _P, _P, _F32, _P, _P, _P, ctypes.c_size_t,
                         _P, _P],
    "ple_gate": [_P, _P, _P, _P, _F32, _I64, _I32, _P, _P, _P],
    "ple_conv": [_P, _P, _I32, _I64, _I32, _P, _I32, _I32, _P, _P, _P, _P, _P],
    "ple_gate_conv": [_P, _P, _P, _P, _F32, _P, _I32, _I64, _I32, _P, _I32, _I32, _P, _P, _P, _P, _P, _P],
    "ple_gated_conv": [_P, _P, _P, _I32, _I64, _I32, _P, _I32, _I32, _P, _P, _P, _P, _P],
    "ple_host_table_alloc": [ctypes.c_size_t, ctypes.POINTER(ctypes.c_void_p)],
    "ple_host_table_free": [ctypes.c_void_p, ctypes.c_size_t],
    "ple_host_table_create_shared": [ctypes.c_char_p, ctypes.c_size_t, _I32,
                                     ctypes.POINTER(ctypes.c_void_p)],
    "ple_host_table_attach_shared": [ctypes.c_char_p, ctypes.c_size_t, _I32,
                                     ctypes.POINTER(ctypes.c_void_p)],
    "ple_host_table_unlink_shared": [ctypes.c_char_p],
    "ple_host_table_map_file": [ctypes.c_char_p, ctypes.c_size_t, _I32,
                                ctypes.POINTER(ctypes.c_void_p)],
    "ple_host_table_unmap": [ctypes.c_void_p, ctypes.c_size_t, _I32],
    "ple_graph_begin": [_P],
    "ple_graph_end": [_P, ctypes.POINTER(ctypes.c_void_p)],
    "ple_graph_launch": [_P, _P],
    "ple_graph_destroy": [_P],
    "ple_event_create": [ctypes.POINTER(ctypes.c_void_p)],
    "ple_event_destroy": [_P],
    "ple_event_synchronize": [_P],
    "ple_step_begin": [_P, _P, _P, _I32, _P, _P, _P],
    "ple_step_end": [_P, _P, _P, _I32, _P, _P],
    "ple_step": [_P, _P, _P, _P, _I32, _P, _P, _I32, _P, _P, _P],
    "ple_last_error": [],
    "ple_version": [],
}
_VOID = ("ple_graph_destroy", "ple_event_destroy")


class PleCopy(ctypes.Structure):
    """ple_copy: one host<->device copy of the step runtime."""
    _fields_ = [("dst", ctypes.c_void_p), ("src", ctypes.c_void_p), ("bytes", ctypes.c_size_t)]


class PleError(RuntimeError):
    def __init__(self, func, status, detail):
        self.status = status
        super().__init__(f"{func} -> {STATUS_NAMES.get(status, status)}: {detail}")


_lib = None


def lib():
    """The loaded libple (built in-tree); raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing: build it with "
                "`python -m hashed_gram_embedding_gb300.build` (there is no non-CUDA path)")
        handle = ctypes.CDLL(LIB_PATH)
        for name, args in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.argtypes = args
            fn.restype = (ctypes.c_char_p if name in ("ple_last_error", "ple_version") else
                          ctypes.c_size_t if name.endswith("_workspace") else
                          None if name in _VOID else ctypes.c_int)
        _lib = handle
    return _lib


def _check(name, status):
    if status != PLE_OK:
        detail = lib().ple_last_error().decode(errors="replace")
        raise PleError(name, status, detail)
    return status


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _i64_array(values):
    a = np.ascontiguousarray(np.asarray(values, dtype=np.int64))
    return a, a.ctypes.data_as(_I64P)


def ple_ngram_ids(input_ids, query_start_loc, ngram_context, layer_multipliers,
                  vocab_sizes, offsets, eos_token_id, heads_per_ngram, out,
                  ngram_context_out=None, dev_err=None, stream=None):
    """Device tensors: input_ids int32 [T], query_start_loc int32 [R+1],
    ngram_context int32 [R, L] or None, out int64 [T, H], ngram_context_out
    int32 [R, L] or None, dev_err int32 [1] or None. Host arrays:
    layer_multipliers [L+1], vocab_sizes [H], offsets [H] (int64)."""
    mult, mult_p = _i64_array(layer_multipliers)
    V, V_p = _i64_array(vocab_sizes)
    O, O_p = _i64_array(offsets)
    return _check("ple_ngram_ids", lib().ple_ngram_ids(
        _ptr(input_ids), input_ids.numel(), _ptr(query_start_loc), query_start_loc.numel() - 1,
        _ptr(ngram_context), len(mult) - 1, mult_p, V_p, O_p, int(eos_token_id),
        int(heads_per_ngram), _ptr(out), _ptr(ngram_context_out), _ptr(dev_err), _stream(stream)))


def _fp8_dtype(row_scale):
    """bf16 without a scale; one scale value -> the whole-table-scale fp8
    type (a one-row table means the same either way); else per-row fp8."""
    if row_scale is None:
        return PLE_BF16
    return PLE_FP8_E4M3_TENSOR if row_scale.numel() == 1 else PLE_FP8_E4M3


def _lookup_args(ids, table, row_scale, out, max_ctas, dev_err, loc):
    dtype = _fp8_dtype(row_scale)
    if loc is None:
        loc = PLE_HBM if table.is_cuda else PLE_HOST_UVA
    T, H = ids.shape
    return (_ptr(ids), T, H, _ptr(table), table.shape[0], table.shape[1], dtype, _ptr(row_scale),
            loc, _ptr(out), int(max_ctas), _ptr(dev_err))


def ple_lookup(ids, table, out, row_scale=None, max_ctas=0, dev_err=None, loc=None, stream=None):
    """ids int64 [T, H]; table [rows, D] bf16 (or uint8 e4m3 codes with
    row_scale float32 [rows], or [1] for one scale for the whole table), on
    the device or pinned on the host; out bf16 [T, H*D]."""
    return _check("ple_lookup", lib().ple_lookup(
        *_lookup_args(ids, table, row_scale, out, max_ctas, dev_err, loc), _stream(stream)))


def ple_ngram_lookup(input_ids, query_start_loc, ngram_context, layer_multipliers, vocab_sizes,
                     offsets, eos_token_id, heads_per_ngram, table, out, row_scale=None,
                     ids_out=None, ngram_context_out=None, max_ctas=0, dev_err=None, loc=None,
                     stream=None):
    """ple_ngram_ids + ple_lookup in one kernel: out bf16 [T, H*D] gets the
    rows of the hashed ids (ids_out int64 [T, H] also gets the ids when
    given). Other arguments as in ple_ngram_ids and ple_lookup."""
    mult, mult_p = _i64_array(layer_multipliers)
    V, V_p = _i64_array(vocab_sizes)
    O, O_p = _i64_array(offsets)
    if loc is None:
        loc = PLE_HBM if table.is_cuda else PLE_HOST_UVA
    return _check("ple_ngram_lookup", lib().ple_ngram_lookup(
        _ptr(input_ids), input_ids.numel(), _ptr(query_start_loc), query_start_loc.numel() - 1,
        _ptr(ngram_context), len(mult) - 1, mult_p, V_p, O_p, int(eos_token_id),
        int(heads_per_ngram), _ptr(table), table.shape[0], table.shape[1], _fp8_dtype(row_scale),
        _ptr(row_scale), loc, _ptr(out), _ptr(ids_out), _ptr(ngram_context_out), int(max_ctas),
        _ptr(dev_err), _stream(stream)))


def ple_lookup_ordered_workspace(num_tokens, num_heads, table, row_scale=None):
    """Bytes of device workspace ple_lookup_ordered needs."""
    dtype = _fp8_dtype(row_scale)
    return int(lib().ple_lookup_ordered_workspace(int(num_tokens), int(num_heads),
                                                  table.shape[0], table.shape[1], dtype))


def ple_lookup_ordered(ids, table, out, workspace, row_scale=None, max_ctas=0, dev_err=None,
                       loc=None, stream=None):
    """ple_lookup with the rows read in table order; workspace: a device
    uint8 tensor of at least ple_lookup_ordered_workspace(...) bytes."""
    a = _lookup_args(ids, table, row_scale, out, max_ctas, dev_err, loc)
    return _check("ple_lookup_ordered", lib().ple_lookup_ordered(
        *a[:-1], _ptr(workspace), workspace.numel() * workspace.element_size(), a[-1],
        _stream(stream)))


def ple_lookup_ordered_static(ids, table, out, row_scale=None, max_ctas=0, dev_err=None,
                              loc=None, stream=None):
    """ple_lookup_ordered with the library's fixed per-device scratch (no
    workspace, no allocation); calls in flight at once must not overlap."""
    return _check("ple_lookup_ordered_static", lib().ple_lookup_ordered_static(
        *_lookup_args(ids, table, row_scale, out, max_ctas, dev_err, loc), _stream(stream)))


def ple_lookup_shard(ids, table, out, kind, head_begin=0, num_heads=None, row_base=0,
                     row_scale=None, scale_out=None, max_ctas=0, dev_err=None, loc=None,
                     stream=None):
    """One rank's lookup in a table split over an exchange group.

    ids int64 [T, ids_heads] (global rows); the heads [head_begin,
    head_begin + num_heads) are looked up in ``table`` [rows, D], whose row 0
    is global row ``row_base``. kind PLE_SHARD_HEADS: out bf16 [T, heads*D]
    (fp8 dequantised). kind PLE_SHARD_ROWS: out holds the raw rows (bf16, or
    uint8 e4m3 codes with scale_out float32 [T, heads]); rows owned by other
    ranks are zero."""
    T, ids_heads = ids.shape
    if num_heads is None:
        num_heads = ids_heads - head_begin
    if loc is None:
        loc = PLE_HBM if table.is_cuda else PLE_HOST_UVA
    return _check("ple_lookup_shard", lib().ple_lookup_shard(
        _ptr(ids), T, ids_heads, int(head_begin), int(num_heads), _ptr(table), table.shape[0],
        int(row_base), table.shape[1], _fp8_dtype(row_scale), _ptr(row_scale), loc, int(kind),
        _ptr(out), _ptr(scale_out), int(max_ctas), _ptr(dev_err), _stream(stream)))


def ple_select_rows(src, row_begin, num_tokens, part_of_head, col_of_head, out, src_scale=None,
                    fp8_dtype=PLE_FP8_E4M3, stream=None):
    """out bf16 [num_tokens, H*D] <- rows [row_begin, row_begin + num_tokens)
    of src [parts, rows, part_heads*D] (bf16, or uint8 e4m3 codes with
    src_scale float32 [parts, rows, part_heads]), head h taken from part
    part_of_head[h], column col_of_head[h]."""
    parts, rows, width = src.shape
    H = len(part_of_head)
    D = out.shape[1] // H
    fp8 = src_scale is not None
    P = np.ascontiguousarray(np.asarray(part_of_head, dtype=np.int32))
    K = np.ascontiguousarray(np.asarray(col_of_head, dtype=np.int32))
    return _check("ple_select_rows", lib().ple_select_rows(
        _ptr(src), parts, rows, width // D, _ptr(src_scale), int(row_begin), int(num_tokens), H,
        P.ctypes.data_as(_I32P), K.ctypes.data_as(_I32P), D, fp8_dtype if fp8 else PLE_BF16,
        _ptr(out), _stream(stream)))


def _event_handle(event, stream):
    """Raw cudaEvent_t of a torch.cuda.Event (torch creates it lazily, on the
    first record: record it once on ``stream`` if it does not exist yet)."""
    if event.cuda_event == 0:
        event.record(stream)
    return ctypes.c_void_p(event.cuda_event)


def ple_lookup_prefetch(ids, table, out, side_stream, done_event, row_scale=None, max_ctas=0,
                        dev_err=None, loc=None):
    """ple_lookup on ``side_stream``, then ``done_event`` (torch.cuda.Event) recorded there."""
    done = _event_handle(done_event, side_stream)
    return _check("ple_lookup_prefetch", lib().ple_lookup_prefetch(
        *_lookup_args(ids, table, row_scale, out, max_ctas, dev_err, loc),
        ctypes.c_void_p(side_stream.cuda_stream), done))


def ple_wait(done_event, consumer_stream=None, timeout_ms=0):
    if done_event.cuda_event == 0:
        return PLE_OK  # never recorded: nothing to wait for
    return _check("ple_wait", lib().ple_wait(ctypes.c_void_p(done_event.cuda_event),
                                             _stream(consumer_stream), int(timeout_ms)))


def ple_kv_proj(emb, w, kv, dev_err=None, stream=None):
    """emb bf16 [T, E], w bf16 [2C, E], kv bf16 [T, 2C]."""
    T, E = emb.shape
    return _check("ple_kv_proj", lib().ple_kv_proj(
        _ptr(emb), _ptr(w), T, E, w.shape[0] // 2, _ptr(kv), _ptr(dev_err), _stream(stream)))


def ple_kv_proj_gate_workspace(num_tokens, hidden):
    """Bytes of device workspace ple_kv_proj_gate needs (0: sizes it rejects)."""
    return int(lib().ple_kv_proj_gate_workspace(int(num_tokens), int(hidden)))


def ple_kv_proj_gate(emb, w, hidden, gamma_h, gamma_k, kv, gate_out, workspace, eps=1e-6,
                     dev_err=None, stream=None):
    """Projection with the gate reductions fused: writes kv[:, C:] (v) and
    gate_out [T] float32; kv[:, :C] is left untouched. workspace: a device
    uint8 tensor of at least ple_kv_proj_gate_workspace(T, C) bytes,
    zero-filled before its first use (the call leaves it zeroed)."""
    T, E = emb.shape
    return _check("ple_kv_proj_gate", lib().ple_kv_proj_gate(
        _ptr(emb), _ptr(w), T, E, w.shape[0] // 2, _ptr(hidden), _ptr(gamma_h), _ptr(gamma_k),
        float(eps), _ptr(kv), _ptr(gate_out), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(dev_err), _stream(stream)))


def ple_gate(hidden, kv, gamma_h, gamma_k, out, eps=1e-6, gate_out=None, stream=None):
    T, C = hidden.shape
    return _check("ple_gate", lib().ple_gate(
        _ptr(hidden), _ptr(kv), _ptr(gamma_h), _ptr(gamma_k), float(eps), T, C, _ptr(out),
        _ptr(gate_out), _stream(stream)))


def ple_conv(x, query_start_loc, w, dilation, out, conv_state=None, conv_state_out=None,
             dev_err=None, stream=None):
    T, C = x.shape
    return _check("ple_conv", lib().ple_conv(
        _ptr(x), _ptr(query_start_loc), query_start_loc.numel() - 1, T, C, _ptr(w), w.shape[1],
        int(dilation), _ptr(conv_state), _ptr(conv_state_out), _ptr(out), _ptr(dev_err),
        _stream(stream)))


def ple_gate_conv(hidden, kv, gamma_h, gamma_k, query_start_loc, w, dilation, out, eps=1e-6,
                  conv_state=None, conv_state_out=None, gate_out=None, dev_err=None, stream=None):
    """gate_out [T] float32 receives the gate scalars (a fresh buffer is made
    when it is not given: pass one in to avoid the allocation)."""
    T, C = hidden.shape
    if gate_out is None:
        import torch
        gate_out = torch.empty((T,), dtype=torch.float32, device=hidden.device)
    return _check("ple_gate_conv", lib().ple_gate_conv(
        _ptr(hidden), _ptr(kv), _ptr(gamma_h), _ptr(gamma_k), float(eps), _ptr(query_start_loc),
        query_start_loc.numel() - 1, T, C, _ptr(w), w.shape[1], int(dilation), _ptr(conv_state),
        _ptr(conv_state_out), _ptr(out), _ptr(gate_out), _ptr(dev_err), _stream(stream)))


def ple_gated_conv(kv, gate, query_start_loc, w, dilation, out, conv_state=None,
                   conv_state_out=None, dev_err=None, stream=None):
    """Conv of u = bf16(gate * v), v = kv[:, C:]; kv [T, 2C] bf16, gate [T] float32."""
    T, C2 = kv.shape
    return _check("ple_gated_conv", lib().ple_gated_conv(
        _ptr(kv), _ptr(gate), _ptr(query_start_loc), query_start_loc.numel() - 1, T, C2 // 2,
        _ptr(w), w.shape[1], int(dilation), _ptr(conv_state), _ptr(conv_state_out), _ptr(out),
        _ptr(dev_err), _stream(stream)))


def ple_version():
    return lib().ple_version().decode()


class HostTable:
    """A table buffer from ple_host_table_alloc, viewed as a torch tensor.

    Keep this object alive as long as the tensor is used; the memory is
    unregistered and unmapped when it is garbage-collected (or on close()).
    """

    def __init__(self, rows, row_dim, dtype):
        import torch
        elem = torch.empty((), dtype=dtype).element_size()
        self.nbytes = int(rows) * int(row_dim) * elem
        ptr = ctypes.c_void_p()
        _check("ple_host_table_alloc", lib().ple_host_table_alloc(self.nbytes, ctypes.byref(ptr)))
        self.ptr = ptr.value
        buf = (ctypes.c_uint8 * self.nbytes).from_address(self.ptr)
        self.tensor = torch.frombuffer(buf, dtype=torch.uint8).view(dtype).view(int(rows), int(row_dim))

    def close(self):
        if getattr(self, "ptr", None):
            self.tensor = None
            lib().ple_host_table_free(ctypes.c_void_p(self.ptr), self.nbytes)
            self.ptr = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class MappedHostTable:
    """A table in a named shared-memory object or a file, mapped by
    ple_host_table_create_shared / _attach_shared / _map_file and viewed as a
    torch tensor [rows, row_dim]; ``register`` makes it readable by the GPU
    over UVA. Unmapped on close() (the shared object itself stays until
    unlink)."""

    def __init__(self, kind, target, rows, row_dim, dtype, register=True):
        import torch
        elem = torch.empty((), dtype=dtype).element_size()
        self.nbytes = int(rows) * int(row_dim) * elem
        self.flags = PLE_HOST_TABLE_REGISTER if register else 0
        fn = {"create": "ple_host_table_create_shared", "attach": "ple_host_table_attach_shared",
              "file": "ple_host_table_map_file"}[kind]
        ptr = ctypes.c_void_p()
        _check(fn, getattr(lib(), fn)(str(target).encode(), self.nbytes, self.flags,
                                      ctypes.byref(ptr)))
        self.ptr = ptr.value
        buf = (ctypes.c_uint8 * self.nbytes).from_address(self.ptr)
        view = torch.frombuffer(buf, dtype=torch.uint8)
        self.tensor = view.view(dtype).view(int(rows), int(row_dim))

    def close(self):
        if getattr(self, "ptr", None):
            self.tensor = None
            lib().ple_host_table_unmap(ctypes.c_void_p(self.ptr), self.nbytes, self.flags)
            self.ptr = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def ple_host_table_unlink_shared(name):
    return _check("ple_host_table_unlink_shared", lib().ple_host_table_unlink_shared(name.encode()))


# ---- step runtime (graph capture, events, one step over three streams) ----

def copies(items):
    """PleCopy array of (dst, src, bytes) triples (pointers as ints)."""
    arr = (PleCopy * max(len(items), 1))()
    for i, (dst, src, nbytes) in enumerate(items):
        arr[i].dst, arr[i].src, arr[i].bytes = dst, src, nbytes
    return arr


def ple_graph_begin(stream):
    _check("ple_graph_begin", lib().ple_graph_begin(_stream(stream)))


def ple_graph_end(stream):
    """End the capture begun on ``stream``; returns the graph handle (int)."""
    g = ctypes.c_void_p()
    _check("ple_graph_end", lib().ple_graph_end(_stream(stream), ctypes.byref(g)))
    return g.value


def ple_graph_launch(graph, stream):
    _check("ple_graph_launch", lib().ple_graph_launch(graph, _stream(stream)))


def ple_graph_destroy(graph):
    lib().ple_graph_destroy(graph)


def ple_event_create():
    ev = ctypes.c_void_p()
    _check("ple_event_create", lib().ple_event_create(ctypes.byref(ev)))
    return ev.value


def ple_event_destroy(event):
    lib().ple_event_destroy(event)


def ple_event_synchronize(event):
    _check("ple_event_synchronize", lib().ple_event_synchronize(event))


def ple_step_begin(copy_in, compute, uploads, num_uploads, loaded, computed, returned):
    _check("ple_step_begin", lib().ple_step_begin(_stream(copy_in), _stream(compute), uploads,
                                                  num_uploads, loaded, computed, returned))


def ple_step_end(compute, copy_out, downloads, num_downloads, computed, returned):
    _check("ple_step_end", lib().ple_step_end(_stream(compute), _stream(copy_out), downloads,
                                              num_downloads, computed, returned))


def ple_step(copy_in, compute, copy_out, uploads, num_uploads, graph, downloads, num_downloads,
             loaded, computed, returned):
    _check("ple_step", lib().ple_step(_stream(copy_in), _stream(compute), _stream(copy_out),
                                      uploads, num_uploads, graph, downloads, num_downloads,
                                      loaded, computed, returned))
