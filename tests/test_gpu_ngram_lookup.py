"""GPU parity of ple_ngram_lookup (n-gram ids hashed inside the row gather)
against the oracle (ids, carry-over and rows bit for bit) and against
ple_ngram_ids followed by ple_lookup (the same bits): bf16 tables, fp8 tables
with per-row and whole-table scales, the tiny / decode / 8k-prefill
workloads (the last at full size in the launch configuration the benchmark
times), many requests (boundaries searched outside shared memory), the
largest head count (64), zero tokens, a missing ids output, invalid
query_start_loc and a head partition outside the table."""

import numpy as np
import pytest
import torch

from oracle import lookup_bf16, lookup_fp8
from oracle import ngram_ids as oracle_ids
from hashed_gram_embedding_gb300 import _lib
from hashed_gram_embedding_gb300 import workloads as wl

from _helpers import bits, dev_err_word

pytestmark = pytest.mark.gpu


def table_for(rows, D, dtype, seed):
    rng = np.random.default_rng(seed)
    if dtype == "bf16":
        t = (torch.from_numpy(rng.standard_normal((rows, D), dtype=np.float32)) * 0.02)
        return t.to(torch.bfloat16), None
    codes = torch.from_numpy(rng.integers(0, 0x7E, size=(rows, D), dtype=np.uint8))
    if dtype == "fp8-row":
        return codes, torch.from_numpy(rng.uniform(1e-3, 1e-2, size=rows).astype(np.float32))
    return codes, torch.tensor([0.0071], dtype=torch.float32)  # one scale for the table


def run_both(h, w, layer, table, row_scale, with_ctx=True):
    """(fused out, fused ids, fused ctx_out, separate out, separate ids, separate ctx_out, err)"""
    T, H, D = len(h["input_ids"]), w.num_heads, table.shape[1]
    ids_d = torch.from_numpy(np.asarray(h["input_ids"], dtype=np.int32)).cuda()
    qsl = torch.from_numpy(np.asarray(h["query_start_loc"], dtype=np.int32)).cuda()
    R = qsl.numel() - 1
    ctx = (torch.from_numpy(np.asarray(h["ngram_context"], dtype=np.int32)).cuda()
           if with_ctx and h["ngram_context"] is not None else None)
    mult = h["multipliers"][layer]
    tab = table.cuda()
    rs = None if row_scale is None else row_scale.cuda()
    res = []
    err = dev_err_word()
    out = torch.full((T, H * D), float("nan"), dtype=torch.bfloat16, device="cuda")
    ids = torch.full((T, H), -1, dtype=torch.int64, device="cuda")
    cto = torch.full((R, w.ctx_len), -5, dtype=torch.int32, device="cuda")
    _lib.ple_ngram_lookup(ids_d, qsl, ctx, mult, h["V"], h["O"], w.eos_token_id,
                          w.heads_per_ngram, tab, out, row_scale=rs, ids_out=ids,
                          ngram_context_out=cto, dev_err=err)
    res += [out, ids, cto]
    out2 = torch.full_like(out, float("nan"))
    ids2 = torch.full_like(ids, -1)
    cto2 = torch.full_like(cto, -5)
    _lib.ple_ngram_ids(ids_d, qsl, ctx, mult, h["V"], h["O"], w.eos_token_id, w.heads_per_ngram,
                       ids2, cto2, err)
    _lib.ple_lookup(ids2, tab, out2, row_scale=rs, dev_err=err)
    torch.cuda.synchronize()
    res += [out2, ids2, cto2, int(err.item())]
    return res


def assert_same(res):
    out, ids, cto, out2, ids2, cto2, err = res
    assert err == 0
    assert torch.equal(ids, ids2)
    assert torch.equal(cto, cto2)
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))


@pytest.fixture(params=["tok", "vector"])
def gather_mode(request, monkeypatch):
    """The token-major kernels (default where the shape fits) and the
    vector-strided ones."""
    if request.param == "vector":
        monkeypatch.setenv("PLE_GATHER_MODE", "vector")
    return request.param


@pytest.mark.parametrize("dtype", ["bf16", "fp8-row", "fp8-tensor"])
@pytest.mark.parametrize("workload", ["tiny", "decode256x4", "fp8x8-small"])
def test_matches_oracle_and_separate_kernels(workload, dtype, gather_mode):
    if workload == "fp8x8-small":  # 2000 Zipf tokens over 64 ragged requests
        w = wl.scaled(wl.WORKLOADS["fp8x8"], vocab_start=5003, num_tokens=2000)
    else:
        w = wl.WORKLOADS[workload]
    if workload == "decode256x4":  # a small table with the workload's ids and context
        w = wl.scaled(w, vocab_start=5003)
    h = wl.host_inputs(w)
    rows = wl.table_rows(w)
    table, row_scale = table_for(rows, 128, dtype, 3)
    res = run_both(h, w, 0, table, row_scale)
    assert_same(res)
    T = len(h["input_ids"])
    ref_ids, ref_ctx = oracle_ids(h["input_ids"], h["query_start_loc"], h["ngram_context"],
                                  h["multipliers"][0], h["V"], h["O"], w.eos_token_id,
                                  w.heads_per_ngram, num_tokens=T)
    ref_ids = np.asarray(ref_ids, dtype=np.int64).reshape(T, -1)
    assert np.array_equal(res[1].cpu().numpy(), ref_ids)
    assert np.array_equal(res[2].cpu().numpy(),
                          np.asarray(ref_ctx, dtype=np.int64).reshape(len(h["query_start_loc"]) - 1, -1))
    if dtype == "bf16":
        ref = lookup_bf16(ref_ids, bits(table))
    else:
        scale = row_scale.numpy() if row_scale.numel() == rows else np.full(rows, float(row_scale[0]), np.float32)
        ref = lookup_fp8(ref_ids, table.numpy(), scale)
    assert np.array_equal(bits(res[0]), ref)


def test_prefill_8k_full_size_against_separate_kernels():
    """The 8k prefill with its 8.2 GB table, in the launch configuration
    the benchmark times: the same ids and rows as the two-kernel path."""
    w = wl.WORKLOADS["prefill8k"]
    h = wl.host_inputs(w)
    table, _ = wl.make_table(torch, w, "cuda")
    res = run_both(h, w, 0, table, None)
    assert_same(res)
    ids = res[1].cpu().numpy()
    assert np.all((ids >= h["O"]) & (ids < h["O"] + h["V"]))


def test_fp8_32k_full_size_against_separate_kernels():
    """One layer of the 32k-token fp8 workload with its 8 GiB table, in the
    benchmark's launch configuration: the same ids and rows as the two-kernel
    path."""
    w = wl.WORKLOADS["fp8x8"]
    h = wl.host_inputs(w)
    table, scale = wl.make_table(torch, w, "cuda", layer=2)
    res = run_both(h, w, 2, table, scale)
    assert_same(res)
    del table, scale, res
    torch.cuda.empty_cache()


def test_many_requests_and_no_ids_output(gather_mode):
    # more request boundaries than the kernel stages in shared memory; no ids output
    rng = np.random.default_rng(12)
    lengths = rng.integers(0, 4, size=5000)
    qsl = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    T = int(qsl[-1])
    tokens = rng.integers(0, 50, size=T).astype(np.int32)
    ctx = rng.integers(0, 50, size=(5000, 2)).astype(np.int32)
    mult, V, O = [7, -11, 13], [101, 103], [0, 101]
    table = (torch.randn((204, 64)) * 0.02).to(torch.bfloat16).cuda()
    d = dict(input_ids=torch.from_numpy(tokens).cuda(), qsl=torch.from_numpy(qsl).cuda(),
             ctx=torch.from_numpy(ctx).cuda())
    out = torch.empty((T, 2 * 64), dtype=torch.bfloat16, device="cuda")
    err = dev_err_word()
    _lib.ple_ngram_lookup(d["input_ids"], d["qsl"], d["ctx"], mult, V, O, 2, 1, table, out,
                          dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref_ids, _ = oracle_ids(tokens, qsl, ctx, mult, V, O, 2, 1, num_tokens=T)
    ref_ids = np.asarray(ref_ids, dtype=np.int64).reshape(T, 2)
    assert np.array_equal(bits(out), lookup_bf16(ref_ids, bits(table)))


def test_zero_tokens_carry_over_and_argument_errors():
    table = torch.zeros((18, 64), dtype=torch.bfloat16, device="cuda")
    mult, V, O = [3, 5, 7], [7, 11], [0, 7]
    qsl = torch.tensor([0, 0, 0], dtype=torch.int32, device="cuda")
    none = torch.empty((0,), dtype=torch.int32, device="cuda")
    out = torch.empty((0, 128), dtype=torch.bfloat16, device="cuda")
    cto = torch.full((2, 2), -1, dtype=torch.int32, device="cuda")
    _lib.ple_ngram_lookup(none, qsl, None, mult, V, O, 9, 1, table, out, ngram_context_out=cto)
    torch.cuda.synchronize()
    assert torch.all(cto == 9)  # no history: EOS
    ctx = torch.tensor([[1, 2], [3, 4]], dtype=torch.int32, device="cuda")
    _lib.ple_ngram_lookup(none, qsl, ctx, mult, V, O, 9, 1, table, out, ngram_context_out=cto)
    torch.cuda.synchronize()
    assert torch.equal(cto, ctx)
    # a head partition past the table's rows is refused on the host
    toks = torch.arange(4, dtype=torch.int32, device="cuda")
    q = torch.tensor([0, 4], dtype=torch.int32, device="cuda")
    out = torch.empty((4, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(_lib.PleError, match="outside"):
        _lib.ple_ngram_lookup(toks, q, None, mult, V, [0, 8], 9, 1, table, out)


def test_invalid_query_start_loc_is_flagged_not_faulted():
    table = (torch.randn((18, 64)) * 0.02).to(torch.bfloat16).cuda()
    mult, V, O = [3, 5, 7], [7, 11], [0, 7]
    toks = torch.arange(8, dtype=torch.int32, device="cuda")
    for q in ([0, 5, 3, 8], [2, 4, 6, 8], [0, 4, 6, 12], [0, -3, 6, 8]):
        out = torch.empty((8, 128), dtype=torch.bfloat16, device="cuda")
        ids = torch.empty((8, 2), dtype=torch.int64, device="cuda")
        err = dev_err_word()
        _lib.ple_ngram_lookup(toks, torch.tensor(q, dtype=torch.int32, device="cuda"), None, mult,
                              V, O, 9, 1, table, out, ids_out=ids, dev_err=err)
        torch.cuda.synchronize()
        assert int(err.item()) & _lib.PLE_DEVERR_QSL
        got = ids.cpu().numpy()
        assert np.all((got >= O) & (got < np.add(O, V)))


def test_largest_head_count():
    """64 heads (2 n-gram orders x 32 heads each, the library's maximum) with
    64-dim rows: the fused lookup equals ple_ngram_ids + ple_lookup and the
    oracle."""
    rng = np.random.default_rng(41)
    L, hpn, D = 2, 32, 64
    H = L * hpn
    V = [int(v) for v in rng.integers(50, 120, size=H)]
    O = [int(o) for o in np.concatenate([[0], np.cumsum(V)[:-1]])]
    rows = int(sum(V))
    table = (torch.randn((rows, D)) * 0.02).to(torch.bfloat16)
    qsl = np.array([0, 40, 41, 100, 333], dtype=np.int32)
    T = int(qsl[-1])
    tokens = rng.integers(0, 60, size=T).astype(np.int32)
    mult = [int(x) for x in (rng.integers(1 << 32, 1 << 62, size=L + 1) | 1)]
    d_tok, d_qsl = torch.from_numpy(tokens).cuda(), torch.from_numpy(qsl).cuda()
    tab = table.cuda()
    out = torch.empty((T, H * D), dtype=torch.bfloat16, device="cuda")
    ids = torch.empty((T, H), dtype=torch.int64, device="cuda")
    _lib.ple_ngram_lookup(d_tok, d_qsl, None, mult, V, O, 2, hpn, tab, out, ids_out=ids)
    ids2 = torch.empty_like(ids)
    out2 = torch.empty_like(out)
    _lib.ple_ngram_ids(d_tok, d_qsl, None, mult, V, O, 2, hpn, ids2)
    _lib.ple_lookup(ids2, tab, out2)
    torch.cuda.synchronize()
    assert torch.equal(ids, ids2) and torch.equal(out.view(torch.int16), out2.view(torch.int16))
    ref_ids, _ = oracle_ids(tokens, qsl, None, mult, V, O, 2, hpn, num_tokens=T)
    ref_ids = np.asarray(ref_ids, dtype=np.int64).reshape(T, H)
    assert np.array_equal(ids.cpu().numpy(), ref_ids)
    assert np.array_equal(bits(out), lookup_bf16(ref_ids, bits(table)))
