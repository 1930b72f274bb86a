"""Sharded lookups on CPU ranks (gloo), against the oracle's full-table lookup.

The host logic of hashed_gram_embedding_gb300.sharded -- TP-major head
shards, slot padding, the id all-gather, the shard gathers, the exchange of
rows (all-gather of head shards; 8-bit integer reduce of row shards) and the
selection of each replica's window -- runs in 2 and 4 gloo processes. The two
libple kernels it calls (ple_lookup_shard, ple_select_rows) need a GPU, so
here they are replaced by plain CPU stand-ins that follow the header's
definition (the GPU tests check the kernels themselves against the same
definition); every replica's result must equal the oracle's lookup over the
whole table bit for bit.
"""

import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
from oracle.numerics import E4M3_VALUES, f64_to_bf16_bits

from hashed_gram_embedding_gb300 import sharded
from hashed_gram_embedding_gb300 import workloads as wl
from hashed_gram_embedding_gb300._lib import PLE_SHARD_HEADS, PLE_SHARD_ROWS


# ---------------------------------------------------------------------------
# host logic alone
# ---------------------------------------------------------------------------

def test_head_shards_are_tp_major_and_cover_every_head():
    H, tp, dp = 16, 2, 4
    seen = []
    for t in range(tp):
        for d in range(dp):
            s, b, n = sharded.head_shard(H, tp, t, dp, d)
            assert s == t * dp + d and n == 2 and b == 2 * s
            seen.extend(range(b, b + n))
    assert sorted(seen) == list(range(H))
    # rank (tp=1, dp=0) owns shard 4: heads 8, 9
    assert sharded.head_shard(H, tp, 1, dp, 0) == (4, 8, 2)


def test_empty_and_uneven_head_shards_are_rejected():
    with pytest.raises(ValueError, match="empty head shard"):
        sharded.head_shard(4, 2, 0, 4, 0)
    with pytest.raises(ValueError, match="evenly"):
        sharded.head_shard(12, 1, 0, 8, 0)
    with pytest.raises(ValueError):
        sharded.head_shard(16, 2, 2, 2, 0)


def test_slots_rows_and_padding():
    assert sharded.gather_slot([5, 9, 0, 3], 2) == (9, 18)
    spans = [sharded.row_shard(10, 4, r) for r in range(4)]
    assert spans == [(0, 3), (3, 6), (6, 9), (9, 10)]
    assert sharded.row_shard(2, 4, 3) == (2, 2)  # a rank may own no row
    V, O = np.array([3, 5, 7, 11]), np.array([0, 3, 8, 15])
    assert sharded.head_rows(V, O, 1, 2) == (3, 15)
    ids = torch.tensor([[1, 4, 9, 20]], dtype=torch.int64)
    p = sharded.pad_ids(ids, 3, O)
    assert p.tolist() == [[1, 4, 9, 20], [0, 3, 8, 15], [0, 3, 8, 15]]
    with pytest.raises(ValueError):
        sharded.pad_ids(ids, 0, O)


# ---------------------------------------------------------------------------
# CPU stand-ins of the two kernels (definitions of include/ple.h)
# ---------------------------------------------------------------------------

def _np_bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


class CpuOps:
    @staticmethod
    def ple_lookup_shard(ids, table, out, kind, head_begin=0, num_heads=None, row_base=0,
                         row_scale=None, scale_out=None, dev_err=None, stream=None, max_ctas=0):
        H = ids.shape[1] - head_begin if num_heads is None else num_heads
        local = ids.numpy()[:, head_begin:head_begin + H] - row_base
        rows, D = table.shape
        inside = (local >= 0) & (local < rows)
        if kind == PLE_SHARD_HEADS:
            assert inside.all()
            if row_scale is None:
                res = oracle.lookup_bf16(local, _np_bits(table))
            else:
                sc = row_scale.numpy()
                sc = np.full(rows, sc[0], dtype=np.float32) if sc.size == 1 else sc
                res = oracle.lookup_fp8(local, table.numpy(), sc)
            out.view(torch.int16).copy_(torch.from_numpy(res.view(np.int16)))
            return
        safe = np.where(inside, local, 0)
        if row_scale is None:
            raw = _np_bits(table)[safe] * inside[..., None]
            out.view(torch.int16).copy_(torch.from_numpy(raw.reshape(out.shape).view(np.int16)))
        else:
            raw = table.numpy()[safe] * inside[..., None]
            out.copy_(torch.from_numpy(raw.reshape(out.shape).astype(np.uint8)))
            sc = row_scale.numpy()
            s = (sc[0] if sc.size == 1 else sc[safe]) * inside
            scale_out.copy_(torch.from_numpy(s.astype(np.float32)))

    @staticmethod
    def ple_select_rows(src, row_begin, num_tokens, part_of_head, col_of_head, out,
                        src_scale=None, stream=None, **_):
        H = len(part_of_head)
        D = out.shape[1] // H
        res = np.empty((num_tokens, H * D), dtype=np.uint16)
        rows = slice(row_begin, row_begin + num_tokens)
        for h in range(H):
            p, k = part_of_head[h], col_of_head[h]
            if src_scale is None:
                res[:, h * D:(h + 1) * D] = _np_bits(src[p])[rows, k * D:(k + 1) * D]
            else:
                codes = src[p].numpy()[rows, k * D:(k + 1) * D]
                sc = src_scale[p].numpy()[rows, k].astype(np.float32)
                prod = E4M3_VALUES[codes] * sc[:, None]
                res[:, h * D:(h + 1) * D] = f64_to_bf16_bits(prod.astype(np.float64))
        out.view(torch.int16).copy_(torch.from_numpy(res.view(np.int16)))


# ---------------------------------------------------------------------------
# gloo groups
# ---------------------------------------------------------------------------

W = wl.scaled(wl.WORKLOADS["tiny"], vocab_start=101, heads_per_ngram=4, head_dim=32)


def full_table(dtype):
    rows = wl.table_rows(W)
    g = torch.Generator().manual_seed(11)
    if dtype == "bf16":
        return (torch.randn((rows, W.head_dim), generator=g) * 0.02).to(torch.bfloat16), None
    codes = torch.randint(0, 256, (rows, W.head_dim), generator=g, dtype=torch.int32)
    codes[(codes & 0x7F) == 0x7F] = 0  # no NaN codes
    scale = (torch.rand((rows,), generator=g) * 1e-3 + 1e-5).to(torch.float32)
    if dtype == "fp8_tensor":
        scale = scale[:1].clone()
    return codes.to(torch.uint8), scale


def replica_ids(dp_rank, num_tokens):
    """Oracle n-gram ids of replica dp_rank's own tokens (seeded per replica)."""
    V, O = wl.head_vocab(W)
    if num_tokens == 0:
        return np.empty((0, W.num_heads), dtype=np.int64)
    rng = np.random.default_rng(100 + dp_rank)
    toks = rng.integers(0, 300, size=num_tokens).astype(np.int32)
    qsl = [0, num_tokens // 2, num_tokens]
    ids, _ = oracle.ngram_ids(toks, qsl, None, wl.layer_multipliers(W, 0), V, O,
                              W.eos_token_id, W.heads_per_ngram)
    return np.asarray(ids, dtype=np.int64).reshape(num_tokens, -1)


def expected_rows(ids, table, scale):
    if scale is None:
        return oracle.lookup_bf16(ids, _np_bits(table))
    sc = scale.numpy()
    sc = np.full(table.shape[0], sc[0], dtype=np.float32) if sc.size == 1 else sc
    return oracle.lookup_fp8(ids, table.numpy(), sc)


def _worker(rank, world, port, tp, kind, dtype, counts, results):
    import torch.distributed as dist
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    dist.init_process_group("gloo", rank=rank, world_size=world)
    dp = world // tp
    dp_rank, tp_rank = divmod(rank, tp)  # replicas contiguous: rank = dp * tp + tp_rank
    assert sharded.group_rank(tp_rank, dp_rank, tp) == rank
    dp_groups = [dist.new_group([d * tp + t for d in range(dp)]) for t in range(tp)]
    dp_group = dp_groups[tp_rank]
    table, scale = full_table(dtype)
    V, O = wl.head_vocab(W)
    n_tok = counts[dp_rank]
    ids = torch.from_numpy(replica_ids(dp_rank, n_tok))
    assert sharded.gather_token_counts(n_tok, dp_group) == list(counts)
    if kind == "heads":
        _, hb, n = sharded.head_shard(W.num_heads, tp, tp_rank, dp, dp_rank)
        r0, r1 = sharded.head_rows(V, O, hb, n)
        look = sharded.HeadShardedLookup(table[r0:r1], scale if scale is None or scale.numel() == 1
                                         else scale[r0:r1], V, O, tp, tp_rank, dp, dp_rank,
                                         ops=CpuOps)
        out = look.lookup(ids, counts, None, dp_group)
    else:
        r0, r1 = sharded.row_shard(table.shape[0], world, rank)
        look = sharded.RowShardedLookup(table[r0:r1], scale if scale is None or scale.numel() == 1
                                        else scale[r0:r1], r0, W.num_heads, dp, dp_rank,
                                        ops=CpuOps)
        out = look.lookup(ids, counts, O, None, dp_group)
    want = expected_rows(ids.numpy(), table, scale)
    results[rank] = bool(np.array_equal(_np_bits(out), want))
    dist.destroy_process_group()


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


@pytest.mark.parametrize("dtype", ["bf16", "fp8", "fp8_tensor"])
@pytest.mark.parametrize("kind", ["heads", "rows"])
@pytest.mark.parametrize("world,tp,counts", [(2, 1, (37, 20)), (4, 2, (0, 33)),
                                             (4, 1, (12, 40, 7, 1))])
def test_sharded_lookup_equals_full_table(world, tp, counts, kind, dtype):
    """Every replica of a world-size 2 or 4 group (TP x DP = 1x2, 2x2, 1x4;
    replicas with different token counts, one with none) gets exactly the
    oracle's full-table rows of its own ids."""
    port = _free_port()
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    results = manager.dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, tp, kind, dtype, counts, results))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    assert dict(results) == {r: True for r in range(world)}
