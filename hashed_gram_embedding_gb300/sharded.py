"""Lookups whose PLE table is split over the ranks of an exchange group.

Two ways the pages split a table, both built from the same two libple
kernels (ple_lookup_shard, ple_select_rows) around torch.distributed
collectives:

* HeadShardedLookup -- the engram-DP split of PR#56512 report ("[DS
  V4.1][Engram] Support async prefetch for offloaded engram lookups and
  engram DP sharding"), 执行摘要 and 实现拆解 items 3-4: a group of
  tp_size x dp_size ranks; the heads are split into tp_size * dp_size equal
  shards assigned in TP-major order (rank (tp, dp) owns shard
  tp * dp_size + dp, engram_head_shard_rank), so that the shards read in
  shard order give the heads in head order; every replica's hashed ids are
  padded to the group's slot size and all-gathered over the DP ranks
  (gather_engram_hashes); each rank gathers its own heads' rows for every
  gathered token; the shard outputs are all-gathered over the whole group;
  each rank then selects its replica's token window from the rank-major
  buffer (_engram_select_rows). Empty head shards are rejected (the test
  test_engram_rejects_empty_head_shards).

* RowShardedLookup -- the ETP split of PR#54371 report ("[Qwen4Exp] Support
  UVA PLE-offload and Engram tensor parallelism"), 实现拆解 item 3 and
  关键源码片段: the concatenated table split into contiguous row ranges over
  the ETP group; ids padded to the slot of the group's largest token count
  (_get_dp_gather_slot) and all-gathered (_gather_dp_ids); each rank fills
  the rows it owns (zeros elsewhere); a parallel reduce combines them --
  through an 8-bit integer view, so that fp8 codes (and bf16 bits) travel
  unchanged (test_ple_fp8_embedding_uses_int8_for_parallel_reduce): every
  byte has exactly one nonzero contributor, so the integer sum is exact --
  and each replica selects its slot (_select_embeddings), dequantising fp8
  codes there.

Readings where the pages are silent (the plainest that the rest supports):
the group's ranks are numbered replica-major (rank = dp * tp_size + tp); the
padding rows of a slot hold each head's first row (offsets[h], a valid row,
so padding never raises the bounds flag); a row-sharded table splits its
rows into group_size ranges of ceil(rows / group_size).

Kernels run through ``ops`` (default: the libple binding); collectives
through torch.distributed (NCCL on GPUs, gloo on CPU ranks). The split into
pad / gather / exchange / select steps lets one process emulate a group (the
kernels of every rank, the collectives by concatenation or sum).
"""

import numpy as np
import torch

from . import _lib


def head_shard(num_heads, tp_size, tp_rank, dp_size, dp_rank):
    """(shard, head_begin, shard_heads) of rank (tp_rank, dp_rank): the
    heads are split into tp_size * dp_size equal shards in TP-major order
    (shard = tp_rank * dp_size + dp_rank)."""
    G = int(tp_size) * int(dp_size)
    if G < 1 or not (0 <= tp_rank < tp_size and 0 <= dp_rank < dp_size):
        raise ValueError(f"rank ({tp_rank}, {dp_rank}) outside a {tp_size} x {dp_size} group")
    n = int(num_heads) // G
    if n == 0:
        raise ValueError(f"empty head shard: {num_heads} heads over {G} ranks")
    if n * G != num_heads:
        raise ValueError(f"{num_heads} heads do not split evenly over {G} ranks")
    s = int(tp_rank) * int(dp_size) + int(dp_rank)
    return s, s * n, n


def group_rank(tp_rank, dp_rank, tp_size):
    """Rank of (tp_rank, dp_rank) in the group: replicas are contiguous."""
    return int(dp_rank) * int(tp_size) + int(tp_rank)


def gather_slot(token_counts, dp_rank):
    """(slot, offset): every replica's tokens padded to the group's largest
    count; this replica's rows start at dp_rank * slot."""
    slot = max(int(c) for c in token_counts)
    return slot, int(dp_rank) * slot


def row_shard(total_rows, group_size, rank):
    """[begin, end) of the concatenated table's rows that rank holds."""
    per = -(-int(total_rows) // int(group_size))
    begin = min(int(rank) * per, int(total_rows))
    return begin, min(begin + per, int(total_rows))


def head_rows(vocab_sizes, offsets, head_begin, num_heads):
    """[begin, end) of the concatenated table's rows holding heads
    [head_begin, head_begin + num_heads)."""
    last = head_begin + num_heads - 1
    return int(offsets[head_begin]), int(offsets[last]) + int(vocab_sizes[last])


def pad_ids(ids, slot, offsets):
    """ids [T, H] int64 -> [slot, H]: rows past T hold offsets[h] (each
    head's first row: valid, so padding never reads outside a shard)."""
    T, H = ids.shape
    if T > slot:
        raise ValueError(f"{T} tokens exceed the slot of {slot}")
    out = torch.empty((slot, H), dtype=ids.dtype, device=ids.device)
    out[:T].copy_(ids)
    if slot > T:
        out[T:].copy_(torch.as_tensor(np.asarray(offsets, dtype=np.int64), device=ids.device)
                      .expand(slot - T, H))
    return out


def _all_gather_cat(t, group):
    import torch.distributed as dist
    n = dist.get_world_size(group)
    parts = [torch.empty_like(t) for _ in range(n)]
    dist.all_gather(parts, t.contiguous(), group=group)
    return torch.stack(parts)


def gather_token_counts(num_tokens, dp_group, device="cpu"):
    """Every replica's token count (what the DP metadata of the pages holds)."""
    t = torch.tensor([int(num_tokens)], dtype=torch.int64, device=device)
    return [int(x) for x in _all_gather_cat(t, dp_group).reshape(-1).tolist()]


class HeadShardedLookup:
    """One rank of a head-sharded (engram-DP) lookup.

    table [rows, D]: this rank's heads' rows of the concatenated table (bf16,
    or uint8 e4m3 codes with row_scale float32 [rows] or [1]); vocab_sizes /
    offsets: the whole table's per-head sizes and offsets (host arrays)."""

    def __init__(self, table, row_scale, vocab_sizes, offsets, tp_size, tp_rank, dp_size,
                 dp_rank, ops=None):
        self.V = np.asarray(vocab_sizes, dtype=np.int64)
        self.O = np.asarray(offsets, dtype=np.int64)
        self.num_heads = len(self.V)
        self.tp_size, self.tp_rank = int(tp_size), int(tp_rank)
        self.dp_size, self.dp_rank = int(dp_size), int(dp_rank)
        self.shard, self.head_begin, self.shard_heads = head_shard(
            self.num_heads, tp_size, tp_rank, dp_size, dp_rank)
        self.row_base, row_end = head_rows(self.V, self.O, self.head_begin, self.shard_heads)
        if table.shape[0] != row_end - self.row_base:
            raise ValueError(f"table of {table.shape[0]} rows; heads {self.head_begin}.."
                             f"{self.head_begin + self.shard_heads - 1} hold {row_end - self.row_base}")
        self.table, self.row_scale = table, row_scale
        self.head_dim = table.shape[1]
        self.ops = ops if ops is not None else _lib
        G = self.tp_size * self.dp_size
        n = self.shard_heads
        # head h lives in shard h // n, owned by rank (tp, dp) = divmod(shard, dp_size)
        self.part_of_head = [group_rank((h // n) // self.dp_size, (h // n) % self.dp_size,
                                        self.tp_size) for h in range(self.num_heads)]
        self.col_of_head = [h % n for h in range(self.num_heads)]
        assert sorted(set(self.part_of_head)) == list(range(G))

    def pad(self, ids, slot):
        return pad_ids(ids, slot, self.O)

    def gather(self, all_ids, dev_err=None, stream=None):
        """all_ids [dp_size * slot, H] -> this shard's rows [dp_size * slot, n*D] bf16."""
        out = torch.empty((all_ids.shape[0], self.shard_heads * self.head_dim),
                          dtype=torch.bfloat16, device=all_ids.device)
        self.ops.ple_lookup_shard(all_ids, self.table, out, _lib.PLE_SHARD_HEADS,
                                  head_begin=self.head_begin, num_heads=self.shard_heads,
                                  row_base=self.row_base, row_scale=self.row_scale,
                                  dev_err=dev_err, stream=stream)
        return out

    def select(self, exchanged, num_tokens, slot, out=None, stream=None):
        """exchanged [G, dp_size * slot, n*D] (group-rank order) -> this
        replica's rows [num_tokens, H*D] bf16 in head order."""
        if out is None:
            out = torch.empty((num_tokens, self.num_heads * self.head_dim), dtype=torch.bfloat16,
                              device=exchanged.device)
        self.ops.ple_select_rows(exchanged, self.dp_rank * slot, num_tokens, self.part_of_head,
                                 self.col_of_head, out, stream=stream)
        return out

    def lookup(self, ids, token_counts, group, dp_group, out=None, dev_err=None):
        """ids [T, H] int64 of this replica -> its rows [T, H*D] bf16, with
        the two all-gathers run on ``dp_group`` (this rank's DP peers, same
        tp_rank) and ``group`` (every rank)."""
        slot, _ = gather_slot(token_counts, self.dp_rank)
        all_ids = _all_gather_cat(self.pad(ids, slot), dp_group).reshape(-1, self.num_heads)
        rows = self.gather(all_ids, dev_err=dev_err)
        exchanged = _all_gather_cat(rows, group)
        return self.select(exchanged, ids.shape[0], slot, out=out)


class RowShardedLookup:
    """One rank of a row-sharded (ETP) lookup.

    table [rows, D]: rows [row_begin, row_begin + rows) of the concatenated
    table (bf16, or uint8 e4m3 codes with row_scale float32 [rows] or [1]);
    num_heads: heads per token; dp_size / dp_rank: this rank's replica in
    the group."""

    def __init__(self, table, row_scale, row_begin, num_heads, dp_size, dp_rank, ops=None):
        self.table, self.row_scale = table, row_scale
        self.row_begin = int(row_begin)
        self.num_heads = int(num_heads)
        self.dp_size, self.dp_rank = int(dp_size), int(dp_rank)
        self.head_dim = table.shape[1]
        self.fp8 = row_scale is not None
        self.ops = ops if ops is not None else _lib

    def pad(self, ids, slot, offsets):
        return pad_ids(ids, slot, offsets)

    def gather(self, all_ids, dev_err=None, stream=None):
        """all_ids [rows, H] -> (raw [rows, H*D] in the table's element type,
        scale [rows, H] float32 or None): this rank's rows, zero elsewhere."""
        R, H = all_ids.shape
        raw = torch.empty((R, H * self.head_dim), dtype=self.table.dtype, device=all_ids.device)
        scale = (torch.empty((R, H), dtype=torch.float32, device=all_ids.device)
                 if self.fp8 else None)
        self.ops.ple_lookup_shard(all_ids, self.table, raw, _lib.PLE_SHARD_ROWS,
                                  row_base=self.row_begin, row_scale=self.row_scale,
                                  scale_out=scale, dev_err=dev_err, stream=stream)
        return raw, scale

    @staticmethod
    def reduce(raw, scale, group):
        """Sum the ranks' outputs as 8-bit integers, in place: every byte has
        one nonzero contributor, so the sum is that byte (bf16 bits, e4m3
        codes and float32 scales all arrive unchanged)."""
        import torch.distributed as dist
        dist.all_reduce(raw.view(torch.int8), group=group)
        if scale is not None:
            dist.all_reduce(scale.view(torch.int8), group=group)
        return raw, scale

    def select(self, raw, scale, num_tokens, slot, out=None, stream=None):
        """Reduced rows -> this replica's rows [num_tokens, H*D] bf16."""
        if out is None:
            out = torch.empty((num_tokens, self.num_heads * self.head_dim), dtype=torch.bfloat16,
                              device=raw.device)
        H = self.num_heads
        self.ops.ple_select_rows(raw.unsqueeze(0), self.dp_rank * slot, num_tokens, [0] * H,
                                 list(range(H)), out,
                                 src_scale=None if scale is None else scale.unsqueeze(0),
                                 stream=stream)
        return out

    def lookup(self, ids, token_counts, offsets, group, dp_group, out=None, dev_err=None):
        """ids [T, H] int64 of this replica -> its rows [T, H*D] bf16."""
        slot, _ = gather_slot(token_counts, self.dp_rank)
        all_ids = _all_gather_cat(self.pad(ids, slot, offsets), dp_group).reshape(-1, self.num_heads)
        raw, scale = self.gather(all_ids, dev_err=dev_err)
        self.reduce(raw, scale, group)
        return self.select(raw, scale, ids.shape[0], slot, out=out)
