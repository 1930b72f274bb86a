"""GPU parity of ple_lookup / ple_lookup_prefetch / ple_wait against the
oracle: bit-exact bf16 rows (HBM and pinned-host UVA tables, several row
sizes, ragged token counts, capped grids), bit-exact fp8 e4m3 dequant with a
per-row scale over all 256 codes, out-of-range ids flagged and zeroed, the
side-stream prefetch, the bounded host wait, and the 8 GB 8k-prefill table at
full size."""

import numpy as np
import pytest
import torch

from oracle import lookup_bf16, lookup_fp8, ngram_ids as oracle_ids
from hashed_gram_embedding_gb300 import _lib
from hashed_gram_embedding_gb300 import workloads as wl

from _helpers import bits, dev_err_word

pytestmark = pytest.mark.gpu


def random_table_bits(rng, rows, D):
    return rng.integers(0, 1 << 16, size=(rows, D), dtype=np.uint16)


def to_dev_bf16(a, pinned=False):
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    if pinned:
        return t.pin_memory()
    return t.cuda()


@pytest.fixture(params=["tok", "vector", "bulk"])
def gather_mode(request, monkeypatch):
    """HBM gathers: the token-major kernel (default where the shape fits it),
    the vector-strided kernel, and the copy-engine one (bf16)."""
    if request.param != "tok":
        monkeypatch.setenv("PLE_GATHER_MODE", request.param)
    return request.param


@pytest.mark.parametrize("T,H,D,rows", [(1, 1, 64, 10), (37, 5, 64, 1000), (513, 16, 128, 4096),
                                        (29, 3, 8, 77), (31, 2, 24, 50), (1000, 8, 256, 333),
                                        (70, 40, 64, 900)])
def test_bf16_gather_bit_exact(T, H, D, rows, gather_mode):
    rng = np.random.default_rng(T * 7 + D)
    table = random_table_bits(rng, rows, D)
    ids = rng.integers(0, rows, size=(T, H))
    out = torch.empty((T, H * D), dtype=torch.bfloat16, device="cuda")
    err = dev_err_word()
    _lib.ple_lookup(torch.from_numpy(ids).cuda(), to_dev_bf16(table), out, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(bits(out), lookup_bf16(ids, table))


@pytest.mark.parametrize("max_ctas", [1, 3, 152])
def test_capped_grid_and_uva_table(max_ctas, gather_mode):
    rng = np.random.default_rng(max_ctas)
    rows, D, T, H = 5000, 128, 300, 16
    table = random_table_bits(rng, rows, D)
    ids = rng.integers(0, rows, size=(T, H))
    ref = lookup_bf16(ids, table)
    d_ids = torch.from_numpy(ids).cuda()
    for pinned in (False, True):
        out = torch.empty((T, H * D), dtype=torch.bfloat16, device="cuda")
        _lib.ple_lookup(d_ids, to_dev_bf16(table, pinned=pinned), out, max_ctas=max_ctas)
        torch.cuda.synchronize()
        assert np.array_equal(bits(out), ref), f"pinned={pinned}"


def test_uva_requires_pinned_host_memory():
    table = torch.zeros((10, 64), dtype=torch.bfloat16)  # pageable host memory
    ids = torch.zeros((1, 1), dtype=torch.int64, device="cuda")
    out = torch.empty((1, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(_lib.PleError, match="PLE_ERR_INVALID_ARG"):
        _lib.ple_lookup(ids, table, out, loc=_lib.PLE_HOST_UVA)
    with pytest.raises(_lib.PleError, match="PLE_ERR_INVALID_ARG"):
        _lib.ple_lookup(ids, table.pin_memory(), out, loc=_lib.PLE_HBM)


def test_fp8_all_codes_bit_exact():
    rng = np.random.default_rng(3)
    D = 128
    rows = 64
    codes = np.concatenate([np.arange(256, dtype=np.uint8).reshape(2, 128),
                            rng.integers(0, 256, size=(rows - 2, D), dtype=np.uint8)])
    scale = np.concatenate([[1.0, 0.5], np.abs(rng.standard_normal(rows - 2)) * 1e-3 + 1e-7]
                           ).astype(np.float32)
    ids = rng.integers(0, rows, size=(50, 4))
    ids[0] = [0, 1, 0, 1]
    out = torch.empty((50, 4 * D), dtype=torch.bfloat16, device="cuda")
    _lib.ple_lookup(torch.from_numpy(ids).cuda(), torch.from_numpy(codes).cuda(), out,
                    row_scale=torch.from_numpy(scale).cuda())
    torch.cuda.synchronize()
    got = bits(out)
    ref = lookup_fp8(ids, codes, scale)
    nan_g = (got & 0x7FFF) > 0x7F80
    nan_r = (ref & 0x7FFF) > 0x7F80
    assert np.array_equal(nan_g, nan_r)
    assert np.array_equal(got[~nan_r], ref[~nan_r])


def test_fp8_workload_rows_bit_exact():
    w = wl.scaled(wl.WORKLOADS["fp8x8"], vocab_start=1000, num_tokens=200, num_reqs=3)
    rows = wl.table_rows(w)
    codes = torch.empty((rows, w.head_dim), dtype=torch.uint8, device="cuda")
    scale = torch.empty((rows,), dtype=torch.float32, device="cuda")
    wl.fill_table_fp8(torch, codes, scale, w.seed, 10)
    rng = np.random.default_rng(4)
    ids = rng.integers(0, rows, size=(200, 16))
    out = torch.empty((200, 16 * w.head_dim), dtype=torch.bfloat16, device="cuda")
    _lib.ple_lookup(torch.from_numpy(ids).cuda(), codes, out, row_scale=scale)
    torch.cuda.synchronize()
    assert np.array_equal(bits(out), lookup_fp8(ids, codes.cpu().numpy(), scale.cpu().numpy()))


def test_out_of_range_ids_are_zeroed_and_flagged(gather_mode):
    rng = np.random.default_rng(5)
    rows, D = 100, 64
    table = random_table_bits(rng, rows, D)
    ids = rng.integers(0, rows, size=(20, 3))
    ids[4, 1] = rows
    ids[7, 0] = -1
    ids[9, 2] = 1 << 40
    out = torch.full((20, 3 * D), 1.0, dtype=torch.bfloat16, device="cuda")
    err = dev_err_word()
    _lib.ple_lookup(torch.from_numpy(ids).cuda(), to_dev_bf16(table), out, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & _lib.PLE_DEVERR_BOUNDS
    got = bits(out)
    bad = [(4, 1), (7, 0), (9, 2)]
    for t, h in bad:
        assert np.all(got[t, h * D:(h + 1) * D] == 0)
    ok_ids = ids.copy()
    for t, h in bad:
        ok_ids[t, h] = 0
    ref = lookup_bf16(ok_ids, table)
    for t, h in bad:
        ref[t, h * D:(h + 1) * D] = 0
    assert np.array_equal(got, ref)


def test_prefetch_on_side_stream_then_wait():
    rng = np.random.default_rng(6)
    rows, D, T, H = 20000, 128, 1024, 16
    table = random_table_bits(rng, rows, D)
    ids = rng.integers(0, rows, size=(T, H))
    d_ids = torch.from_numpy(ids).cuda()
    host_table = to_dev_bf16(table, pinned=True)
    side = torch.cuda.Stream()
    done = torch.cuda.Event()
    ready = torch.cuda.Event()
    ready.record(torch.cuda.current_stream())
    side.wait_event(ready)
    out = torch.empty((T, H * D), dtype=torch.bfloat16, device="cuda")
    _lib.ple_lookup_prefetch(d_ids, host_table, out, side, done, max_ctas=76)
    _lib.ple_wait(done, torch.cuda.current_stream(), timeout_ms=0)
    result = out.clone()  # ordered after the wait on the consumer stream
    torch.cuda.synchronize()
    assert np.array_equal(bits(result), lookup_bf16(ids, table))


def test_wait_times_out_then_completes():
    side = torch.cuda.Stream()
    done = torch.cuda.Event()
    ids = torch.zeros((1, 1), dtype=torch.int64, device="cuda")
    table = torch.zeros((4, 64), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((1, 64), dtype=torch.bfloat16, device="cuda")
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        a = torch.randn((8192, 8192), device="cuda", dtype=torch.bfloat16)
        for _ in range(40):
            a = (a @ a).clamp_(-1, 1)  # tens of milliseconds of work before the event
    _lib.ple_lookup_prefetch(ids, table, out, side, done)
    with pytest.raises(_lib.PleError, match="PLE_ERR_TIMEOUT"):
        _lib.ple_wait(done, torch.cuda.current_stream(), timeout_ms=1)
    _lib.ple_wait(done, torch.cuda.current_stream(), timeout_ms=60000)
    torch.cuda.synchronize()


def test_prefill_8k_full_size_table(gather_mode):
    w = wl.WORKLOADS["prefill8k"]
    h = wl.host_inputs(w)
    table, _ = wl.make_table(torch, w, "cuda")
    ids, _ = oracle_ids(h["input_ids"], h["query_start_loc"], None, h["multipliers"][0], h["V"],
                        h["O"], w.eos_token_id, w.heads_per_ngram)
    ids = np.asarray(ids, dtype=np.int64)
    d_ids = torch.from_numpy(ids).cuda()
    out = torch.empty((w.num_tokens, w.emb_dim), dtype=torch.bfloat16, device="cuda")
    err = dev_err_word()
    _lib.ple_lookup(d_ids, table, out, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    # every row: a plain index_select of the input table (library routine)
    assert torch.equal(out, table.index_select(0, d_ids.reshape(-1)).reshape(out.shape))
    # a sample through the oracle on the host
    rng = np.random.default_rng(8)
    sample = np.unique(np.concatenate([rng.integers(0, w.num_tokens, 256),
                                       h["query_start_loc"][:-1]]))
    sub_ids = ids[sample]
    uniq, inv = np.unique(sub_ids, return_inverse=True)
    compact = bits(table[torch.from_numpy(uniq).cuda()])
    ref = lookup_bf16(inv.reshape(sub_ids.shape), compact)
    assert np.array_equal(bits(out)[sample], ref)
    del table
    torch.cuda.empty_cache()


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_uva_gather_from_huge_page_host_table(dtype):
    """A table from ple_host_table_alloc (huge-page-backed registered host
    memory) is read in place over UVA, bit-exact, with bad ids flagged."""
    rng = np.random.default_rng(12)
    D, T, H = 128, 700, 16
    rows = 300000
    if dtype == "bf16":
        owner = _lib.HostTable(rows, D, torch.bfloat16)
        table = random_table_bits(rng, rows, D)
        owner.tensor.view(torch.int16).copy_(torch.from_numpy(table.view(np.int16)))
        scale = None
    else:
        owner = _lib.HostTable(rows, D, torch.uint8)
        codes = rng.integers(0, 0x7E, size=(rows, D), dtype=np.uint8)
        owner.tensor.copy_(torch.from_numpy(codes))
        sc = (np.abs(rng.standard_normal(rows)) * 1e-3 + 1e-6).astype(np.float32)
        scale = torch.from_numpy(sc).cuda()
    assert owner.ptr % (1 << 30) == 0
    ids = rng.integers(0, rows, size=(T, H))
    ids[3, 2] = rows + 5          # outside the table: zero row + flag
    ids[9, 0] = -7
    out = torch.full((T, H * D), 3.0, dtype=torch.bfloat16, device="cuda")
    err = dev_err_word()
    _lib.ple_lookup(torch.from_numpy(ids).cuda(), owner.tensor, out, row_scale=scale, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & _lib.PLE_DEVERR_BOUNDS
    ok = ids.copy()
    ok[3, 2] = 0
    ok[9, 0] = 0
    ref = lookup_bf16(ok, table) if dtype == "bf16" else lookup_fp8(ok, codes, sc)
    ref[3, 2 * D:3 * D] = 0
    ref[9, 0:D] = 0
    assert np.array_equal(bits(out), ref)
    owner.close()


def test_uva32g_full_size_ordered_gather():
    """The host-table workload at full size: 8192 tokens x 16 heads gathered
    in table order from the 32 GiB huge-page-backed registered host table
    (PLELayer.embed: ids, then the ordered gather), ids against the oracle
    and every row bit for bit against the table read on the host."""
    from hashed_gram_embedding_gb300 import PLELayer
    w = wl.WORKLOADS["uva32g"]
    host = wl.host_inputs(w)
    table, _ = wl.make_table(torch, w, "cuda")
    assert not table.is_cuda and wl.table_rows(w) == table.shape[0]
    C = w.hidden
    wkv = torch.zeros((2 * C, w.emb_dim), dtype=torch.bfloat16, device="cuda")
    g1 = torch.ones((C,), dtype=torch.bfloat16, device="cuda")
    cw = torch.zeros((C, w.conv_k), dtype=torch.bfloat16, device="cuda")
    layer = PLELayer(table, None, host["multipliers"][0], host["V"], host["O"], w.eos_token_id,
                     w.heads_per_ngram, wkv, g1, g1, cw, w.dilation)
    T = w.num_tokens
    b = layer.buffers(T, torch.device("cuda"))
    err = dev_err_word()
    layer.embed(torch.from_numpy(host["input_ids"]).cuda(),
                torch.from_numpy(host["query_start_loc"]).cuda(), b["ids"], b["emb"],
                b["order_ws"], dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ids, _ = oracle_ids(host["input_ids"], host["query_start_loc"], None, host["multipliers"][0],
                        host["V"], host["O"], w.eos_token_id, w.heads_per_ngram)
    ids = np.asarray(ids, dtype=np.int64).reshape(T, -1)
    assert np.array_equal(b["ids"].cpu().numpy(), ids)
    rows = table[torch.from_numpy(ids.reshape(-1))]  # read on the host
    assert torch.equal(b["emb"].cpu().view(torch.int16),
                       rows.reshape(T, -1).view(torch.int16))
    del layer, table
    torch.cuda.empty_cache()


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
@pytest.mark.parametrize("rows", [10, 5000, 300000])
def test_ordered_gather_equals_plain_gather(dtype, rows):
    """ple_lookup_ordered (items sorted by table span, then gathered) writes
    exactly what ple_lookup writes, for device and host tables, with ids
    outside the table zeroed and flagged."""
    rng = np.random.default_rng(rows)
    D, T, H = 128, 333, 16
    if dtype == "bf16":
        table = random_table_bits(rng, rows, D)
        dev_table = to_dev_bf16(table)
        host = _lib.HostTable(rows, D, torch.bfloat16)
        host.tensor.view(torch.int16).copy_(torch.from_numpy(table.view(np.int16)))
        scale = None
    else:
        codes = rng.integers(0, 0x7E, size=(rows, D), dtype=np.uint8)
        dev_table = torch.from_numpy(codes).cuda()
        host = _lib.HostTable(rows, D, torch.uint8)
        host.tensor.copy_(torch.from_numpy(codes))
        sc = (np.abs(rng.standard_normal(rows)) * 1e-3 + 1e-6).astype(np.float32)
        scale = torch.from_numpy(sc).cuda()
    ids = rng.integers(0, rows, size=(T, H))
    ids[5, 3] = rows
    ids[17, 0] = -2
    d_ids = torch.from_numpy(ids).cuda()
    ref = torch.empty((T, H * D), dtype=torch.bfloat16, device="cuda")
    err0 = dev_err_word()
    _lib.ple_lookup(d_ids, dev_table, ref, row_scale=scale, dev_err=err0)
    for tab in (dev_table, host.tensor):
        ws = torch.empty((_lib.ple_lookup_ordered_workspace(T, H, tab, scale),), dtype=torch.uint8,
                         device="cuda")
        ws.fill_(0xAB)  # contents on entry do not matter
        out = torch.full((T, H * D), 5.0, dtype=torch.bfloat16, device="cuda")
        err = dev_err_word()
        _lib.ple_lookup_ordered(d_ids, tab, out, ws, row_scale=scale, dev_err=err)
        torch.cuda.synchronize()
        assert int(err.item()) & _lib.PLE_DEVERR_BOUNDS
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))  # bits (tables hold NaNs)
    ok = ids.copy()
    ok[5, 3] = 0
    ok[17, 0] = 0
    want = lookup_bf16(ok, table) if dtype == "bf16" else lookup_fp8(ok, codes, sc)
    want[5, 3 * D:4 * D] = 0
    want[17, 0:D] = 0
    assert np.array_equal(bits(ref), want)
    host.close()


def test_ordered_gather_rejects_small_workspace():
    rows, D, T, H = 1000, 64, 8, 2
    table = torch.zeros((rows, D), dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros((T, H), dtype=torch.int64, device="cuda")
    out = torch.empty((T, H * D), dtype=torch.bfloat16, device="cuda")
    need = _lib.ple_lookup_ordered_workspace(T, H, table)
    ws = torch.empty((need - 256,), dtype=torch.uint8, device="cuda")
    with pytest.raises(_lib.PleError, match="workspace"):
        _lib.ple_lookup_ordered(ids, table, out, ws)


@pytest.mark.parametrize("ordered", [False, True])
def test_fp8_global_scale(ordered):
    """The pages' fp8 table carries one weight_scale for the whole table
    (PLE_FP8_E4M3_TENSOR: a one-value row_scale): e4m3 code times that scale,
    rounded to bf16 -- the oracle's per-row formula with every row's scale
    equal, bit for bit, and the same bits as a per-row scale array holding
    the value everywhere. Plain gather and table-order gather (host table)."""
    rng = np.random.default_rng(21)
    rows, D, T, H = 3000, 128, 64, 16
    codes = rng.integers(0, 0x7E, size=(rows, D), dtype=np.uint8)  # finite codes
    weight_scale = np.float32(0.0123)
    scale = np.full((rows,), weight_scale, dtype=np.float32)
    ids = rng.integers(0, rows, size=(T, H))
    d_ids = torch.from_numpy(ids).cuda()
    if ordered:
        table = torch.from_numpy(codes).pin_memory()
    else:
        table = torch.from_numpy(codes).cuda()
    one = torch.tensor([weight_scale], dtype=torch.float32, device="cuda")
    full = torch.from_numpy(scale).cuda()
    outs = []
    for row_scale in (one, full):
        out = torch.empty((T, H * D), dtype=torch.bfloat16, device="cuda")
        if ordered:
            ws = torch.empty((_lib.ple_lookup_ordered_workspace(T, H, table, row_scale),),
                             dtype=torch.uint8, device="cuda")
            _lib.ple_lookup_ordered(d_ids, table, out, ws, row_scale=row_scale)
        else:
            _lib.ple_lookup(d_ids, table, out, row_scale=row_scale)
        outs.append(out)
    torch.cuda.synchronize()
    assert np.array_equal(bits(outs[0]), lookup_fp8(ids, codes, scale))
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    # the same numbers from torch's own e4m3 decode times the one scale
    dec = torch.from_numpy(codes).view(torch.float8_e4m3fn).float() * float(weight_scale)
    want = dec[torch.from_numpy(ids.reshape(-1))].reshape(T, H * D).to(torch.bfloat16)
    assert torch.equal(outs[0].cpu().view(torch.int16), want.view(torch.int16))


@pytest.mark.parametrize("kind", ["shared", "file"])
def test_gather_from_shared_and_file_backed_tables(kind, tmp_path):
    """Tables in a named shared-memory object and in a file, registered for
    GPU reads (the file read-only), give bit-exact rows through the plain and
    the ordered gather."""
    import uuid
    rng = np.random.default_rng(31)
    rows, D, T, H = 20000, 128, 257, 16
    table = random_table_bits(rng, rows, D)
    name = "/ple_gpu_" + uuid.uuid4().hex[:12]
    if kind == "shared":
        t = _lib.MappedHostTable("create", name, rows, D, torch.bfloat16, register=True)
        t.tensor.view(torch.int16).copy_(torch.from_numpy(table.view(np.int16)))
    else:
        path = tmp_path / "rows.bin"
        table.tofile(path)
        t = _lib.MappedHostTable("file", path, rows, D, torch.bfloat16, register=True)
    try:
        ids = rng.integers(0, rows, size=(T, H))
        d_ids = torch.from_numpy(ids).cuda()
        want = lookup_bf16(ids, table)
        out = torch.empty((T, H * D), dtype=torch.bfloat16, device="cuda")
        _lib.ple_lookup(d_ids, t.tensor, out)
        torch.cuda.synchronize()
        assert np.array_equal(bits(out), want)
        ws = torch.empty((_lib.ple_lookup_ordered_workspace(T, H, t.tensor),), dtype=torch.uint8,
                         device="cuda")
        out.zero_()
        _lib.ple_lookup_ordered(d_ids, t.tensor, out, ws)
        torch.cuda.synchronize()
        assert np.array_equal(bits(out), want)
    finally:
        t.close()
        if kind == "shared":
            _lib.ple_host_table_unlink_shared(name)


@pytest.mark.parametrize("dtype", ["bf16", "fp8", "fp8_tensor"])
@pytest.mark.parametrize("T,H,D", [(1, 1, 64), (3, 3, 128), (201, 16, 128), (1025, 5, 64),
                                   (77, 12, 64), (64, 32, 64), (40, 2, 128), (9, 16, 64)])
def test_token_major_gather_equals_vector_gather_and_oracle(T, H, D, dtype, monkeypatch):
    """The token-major kernel (ragged last group, heads not dividing 32, ids
    outside the table) writes exactly what the vector-strided kernel writes,
    and the oracle's rows."""
    rng = np.random.default_rng(T * 13 + H * 7 + D)
    rows = 3001
    ids = rng.integers(0, rows, size=(T, H))
    ids[T // 2, H - 1] = rows + 5
    ids[0, 0] = -3
    if dtype == "bf16":
        table_np = random_table_bits(rng, rows, D)
        table = to_dev_bf16(table_np)
        scale = None
    else:
        codes = rng.integers(0, 256, size=(rows, D)).astype(np.uint8)
        codes[(codes & 0x7F) == 0x7F] = 0
        table = torch.from_numpy(codes).cuda()
        sc = (rng.random(rows if dtype == "fp8" else 1) * 1e-2 + 1e-4).astype(np.float32)
        scale = torch.from_numpy(sc).cuda()
    outs, errs = [], []
    for mode in ("tok", "vector"):
        if mode == "vector":
            monkeypatch.setenv("PLE_GATHER_MODE", "vector")
        out = torch.full((T, H * D), 3.0, dtype=torch.bfloat16, device="cuda")
        err = dev_err_word()
        _lib.ple_lookup(torch.from_numpy(ids).cuda(), table, out, row_scale=scale, dev_err=err)
        torch.cuda.synchronize()
        outs.append(bits(out))
        errs.append(int(err.item()))
    assert errs == [_lib.PLE_DEVERR_BOUNDS] * 2
    assert np.array_equal(outs[0], outs[1])
    ok = ids.copy()
    ok[T // 2, H - 1] = 0
    ok[0, 0] = 0
    if dtype == "bf16":
        ref = lookup_bf16(ok, table_np)
    else:
        full = np.full(rows, sc[0], dtype=np.float32) if sc.size == 1 else sc
        ref = lookup_fp8(ok, codes, full)
    ref[T // 2, (H - 1) * D:] = 0
    ref[0, :D] = 0
    assert np.array_equal(outs[0], ref)
