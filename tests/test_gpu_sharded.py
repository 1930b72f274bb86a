"""GPU parity of the sharded-lookup kernels (ple_lookup_shard,
ple_select_rows) through the C ABI, and of whole head- and row-sharded groups
emulated in one process on one GPU: every rank's kernels run in turn on its
own shard, the collectives are replaced by concatenation (all-gather) and an
8-bit integer sum (reduce), and every replica's rows must equal the oracle's
full-table lookup bit for bit. No kernel waits on another."""

import numpy as np
import pytest
import torch

import oracle
from hashed_gram_embedding_gb300 import _lib, sharded
from hashed_gram_embedding_gb300 import workloads as wl

from _helpers import bits, dev_err_word

pytestmark = pytest.mark.gpu


def make_table(dtype, rows, D, seed):
    g = torch.Generator().manual_seed(seed)
    if dtype == "bf16":
        return (torch.randn((rows, D), generator=g) * 0.02).to(torch.bfloat16), None
    codes = torch.randint(0, 256, (rows, D), generator=g, dtype=torch.int32)
    codes[(codes & 0x7F) == 0x7F] = 0x01  # no NaN codes
    scale = (torch.rand((rows,), generator=g) * 1e-3 + 1e-5).to(torch.float32)
    if dtype == "fp8_tensor":
        scale = scale[:1].clone()
    return codes.to(torch.uint8), scale


def oracle_rows(ids, table, scale):
    ids = np.asarray(ids, dtype=np.int64)
    if scale is None:
        return oracle.lookup_bf16(ids, bits(table))
    sc = scale.numpy()
    sc = np.full(table.shape[0], sc[0], dtype=np.float32) if sc.size == 1 else sc
    return oracle.lookup_fp8(ids, table.numpy(), sc)


def dev(t):
    return None if t is None else t.cuda()


@pytest.mark.parametrize("dtype", ["bf16", "fp8", "fp8_tensor"])
@pytest.mark.parametrize("T,H,D", [(1, 4, 64), (333, 16, 128), (1000, 6, 32)])
def test_head_shard_gather(dtype, T, H, D):
    """Heads [hb, hb+n) of full-width ids, looked up in a table that holds
    global rows [base, base+rows): the oracle's rows of the local ids; an id
    outside the shard gives a zero row and the bounds flag."""
    rows, base = 5000, 12345
    table, scale = make_table(dtype, rows, D, T + H)
    rng = np.random.default_rng(T)
    ids = rng.integers(base, base + rows, size=(T, H)).astype(np.int64)
    hb, n = (1, H - 2) if H > 2 else (0, H)
    out = torch.empty((T, n * D), dtype=torch.bfloat16, device="cuda")
    err = dev_err_word()
    _lib.ple_lookup_shard(torch.from_numpy(ids).cuda(), dev(table), out, _lib.PLE_SHARD_HEADS,
                          head_begin=hb, num_heads=n, row_base=base, row_scale=dev(scale),
                          dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(bits(out), oracle_rows(ids[:, hb:hb + n] - base, table, scale))
    # one id below the shard, one above
    bad = ids.copy()
    bad[0, hb] = base - 1
    bad[T - 1, hb + n - 1] = base + rows
    _lib.ple_lookup_shard(torch.from_numpy(bad).cuda(), dev(table), out, _lib.PLE_SHARD_HEADS,
                          head_begin=hb, num_heads=n, row_base=base, row_scale=dev(scale),
                          dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == _lib.PLE_DEVERR_BOUNDS
    ok = bad[:, hb:hb + n] - base
    ok[0, 0] = 0
    ok[T - 1, n - 1] = 0
    want = oracle_rows(ok, table, scale)
    want[0, :D] = 0
    want[T - 1, (n - 1) * D:] = 0
    assert np.array_equal(bits(out), want)


@pytest.mark.parametrize("dtype", ["bf16", "fp8", "fp8_tensor"])
def test_row_shard_gather_keeps_raw_bytes(dtype):
    """A row shard writes the raw row bytes (and scales) of the rows it owns
    and zeros for every other id, without raising the bounds flag."""
    T, H, D, rows, base = 257, 16, 128, 3000, 7000
    table, scale = make_table(dtype, rows, D, 3)
    rng = np.random.default_rng(5)
    ids = rng.integers(0, 20000, size=(T, H)).astype(np.int64)
    ids[::7, 3] = base + rng.integers(0, rows, size=ids[::7, 3].shape)
    local = ids - base
    inside = (local >= 0) & (local < rows)
    assert inside.any() and not inside.all()
    raw = torch.empty((T, H * D), dtype=table.dtype, device="cuda")
    sc = torch.empty((T, H), dtype=torch.float32, device="cuda") if scale is not None else None
    err = dev_err_word()
    _lib.ple_lookup_shard(torch.from_numpy(ids).cuda(), dev(table), raw, _lib.PLE_SHARD_ROWS,
                          row_base=base, row_scale=dev(scale), scale_out=sc, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    safe = np.where(inside, local, 0)
    tab = bits(table) if scale is None else table.numpy()
    want = (tab[safe] * inside[..., None]).reshape(T, H * D)
    got = bits(raw) if scale is None else raw.cpu().numpy()
    assert np.array_equal(got, want)
    if scale is not None:
        s = scale.numpy()
        ws = (s[0] if s.size == 1 else s[safe]) * inside
        assert np.array_equal(sc.cpu().numpy(), ws.astype(np.float32))


@pytest.mark.parametrize("fp8", [False, True])
def test_select_rows(fp8):
    """out[t][h] = src[part(h)][row_begin + t][col(h)], fp8 codes dequantised."""
    parts, prow, ph, D, H = 3, 50, 4, 64, 12
    rng = np.random.default_rng(9)
    if fp8:
        codes = rng.integers(0, 256, size=(parts, prow, ph * D)).astype(np.uint8)
        codes[(codes & 0x7F) == 0x7F] = 1
        src = torch.from_numpy(codes)
        scl = torch.from_numpy((rng.random((parts, prow, ph)) * 1e-2).astype(np.float32))
    else:
        src = torch.randn((parts, prow, ph * D)).to(torch.bfloat16)
        scl = None
    part = [int(x) for x in rng.integers(0, parts, H)]
    col = [int(x) for x in rng.integers(0, ph, H)]
    r0, T = 7, 40
    out = torch.empty((T, H * D), dtype=torch.bfloat16, device="cuda")
    _lib.ple_select_rows(src.cuda(), r0, T, part, col, out, src_scale=dev(scl))
    torch.cuda.synchronize()
    want = np.empty((T, H * D), dtype=np.uint16)
    for h in range(H):
        if fp8:
            c = codes[part[h], r0:r0 + T, col[h] * D:(col[h] + 1) * D]
            s = scl.numpy()[part[h], r0:r0 + T, col[h]]
            # row-by-row through the oracle's fp8 lookup (one row per "token")
            want[:, h * D:(h + 1) * D] = oracle.lookup_fp8(
                np.arange(T)[:, None], c, s)
        else:
            want[:, h * D:(h + 1) * D] = bits(src[part[h], r0:r0 + T, col[h] * D:(col[h] + 1) * D])
    assert np.array_equal(bits(out), want)


def test_select_rows_rejects_bad_maps():
    src = torch.zeros((2, 10, 2 * 64), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((4, 2 * 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(_lib.PleError, match="maps to part"):
        _lib.ple_select_rows(src, 0, 4, [0, 2], [0, 1], out)
    with pytest.raises(_lib.PleError, match="bad sizes"):
        _lib.ple_select_rows(src, 8, 4, [0, 1], [0, 1], out)


W = wl.scaled(wl.WORKLOADS["prefill8k"], vocab_start=3001)


def replica_ids(d, n, V, O):
    if n == 0:
        return np.empty((0, len(V)), dtype=np.int64)
    rng = np.random.default_rng(40 + d)
    toks = rng.integers(0, W.token_vocab, n).astype(np.int32)
    cuts = sorted(rng.choice(np.arange(1, n), size=min(3, n - 1), replace=False)) if n > 1 else []
    qsl = [0, *[int(c) for c in cuts], n]
    ids, _ = oracle.ngram_ids(toks, qsl, None, wl.layer_multipliers(W, 0), V, O,
                              W.eos_token_id, W.heads_per_ngram)
    return np.asarray(ids, dtype=np.int64).reshape(n, -1)


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
@pytest.mark.parametrize("tp,dp,counts", [(1, 2, (300, 170)), (2, 2, (0, 257)),
                                          (1, 4, (64, 1, 200, 129)), (2, 4, (5, 6, 7, 8))])
def test_emulated_head_sharded_group(tp, dp, counts, dtype):
    """Every rank of a tp x dp engram-DP group (16 heads of 128 over primes
    near 3001) on one GPU: pad + id all-gather (concatenation), its own heads'
    gather, the rank-major all-gather of shard rows (stacking by group rank),
    and its replica's select; each replica gets the oracle's full-table rows."""
    V, O = wl.head_vocab(W)
    table, scale = make_table(dtype, int(V.sum()), W.head_dim, 21)
    ids = [replica_ids(d, counts[d], V, O) for d in range(dp)]
    G = tp * dp
    ranks = {}
    for r in range(G):
        d, t = divmod(r, tp)
        _, hb, n = sharded.head_shard(W.num_heads, tp, t, dp, d)
        r0, r1 = sharded.head_rows(V, O, hb, n)
        sc = None if scale is None else (scale[r0:r1] if scale.numel() > 1 else scale)
        ranks[r] = sharded.HeadShardedLookup(table[r0:r1].cuda(), dev(sc), V, O, tp, t, dp, d)
    slot, _ = sharded.gather_slot(counts, 0)
    padded = [ranks[d * tp].pad(torch.from_numpy(ids[d]).cuda(), slot) for d in range(dp)]
    all_ids = torch.cat(padded)
    err = dev_err_word()
    shard_rows = torch.stack([ranks[r].gather(all_ids, dev_err=err) for r in range(G)])
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for r in range(G):
        d = r // tp
        out = ranks[r].select(shard_rows, counts[d], slot)
        torch.cuda.synchronize()
        assert np.array_equal(bits(out), oracle_rows(ids[d], table, scale)), f"rank {r}"


@pytest.mark.parametrize("dtype", ["bf16", "fp8", "fp8_tensor"])
@pytest.mark.parametrize("tp,dp,counts", [(1, 2, (300, 170)), (2, 2, (0, 257)),
                                          (1, 4, (64, 1, 200, 129))])
def test_emulated_row_sharded_group(tp, dp, counts, dtype):
    """Every rank of a tp x dp ETP group on one GPU: the table split into
    row ranges, each rank's raw rows for every gathered id (zeros where it
    does not own the row), the ranks' outputs summed as 8-bit integers, and
    each replica's select (fp8 dequantised there): the oracle's rows."""
    V, O = wl.head_vocab(W)
    table, scale = make_table(dtype, int(V.sum()), W.head_dim, 22)
    ids = [replica_ids(d, counts[d], V, O) for d in range(dp)]
    G = tp * dp
    look = {}
    for r in range(G):
        r0, r1 = sharded.row_shard(table.shape[0], G, r)
        sc = None if scale is None else (scale[r0:r1] if scale.numel() > 1 else scale)
        look[r] = sharded.RowShardedLookup(table[r0:r1].cuda(), dev(sc), r0, W.num_heads, dp,
                                           r // tp)
    slot, _ = sharded.gather_slot(counts, 0)
    all_ids = torch.cat([look[d * tp].pad(torch.from_numpy(ids[d]).cuda(), slot, O)
                         for d in range(dp)])
    err = dev_err_word()
    outs = [look[r].gather(all_ids, dev_err=err) for r in range(G)]
    torch.cuda.synchronize()
    assert int(err.item()) == 0

    def int8_sum(ts):  # one nonzero contributor per byte: the sum is that byte
        s = torch.stack([t.view(torch.int8) for t in ts]).sum(dim=0, dtype=torch.int32)
        return s.to(torch.int8).view(ts[0].dtype)

    raw = int8_sum([o[0] for o in outs])
    sc = None if scale is None else int8_sum([o[1] for o in outs])
    for r in range(G):
        d = r // tp
        out = look[r].select(raw, sc, counts[d], slot)
        torch.cuda.synchronize()
        assert np.array_equal(bits(out), oracle_rows(ids[d], table, scale)), f"rank {r}"
