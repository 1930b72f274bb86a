"""Seeded synthetic workloads shaped like the pages' PLE / Engram serving loads.

This module makes inputs only: token streams, ragged request boundaries,
per-layer hash constants (multipliers, per-head vocab sizes and offsets) and
random tables / weights / activations. It holds none of the method's
arithmetic, so the CUDA path and the CPU oracle can both be fed from it.

The pages give no dataset, only workload descriptions (8k-token prefills,
decode with n-gram context carry-over, tables of up to ~100 GB per layer, fp8
tables with a scale, a pinned-host table read over UVA). Every workload here is
synthetic; the recipe of each one is in ``WORKLOADS`` and in the docstrings.

Recipe common to all workloads:
  * eos_token_id = 2; n-gram orders 2 and 3 (NGRAM_CONTEXT_LEN = 2).
  * per-layer multipliers: 3 odd int64 drawn uniformly from [2^32, 2^62) by
    ``numpy.random.default_rng(seed * 1000 + layer)``, large enough that the
    products wrap around int64.
  * per-head vocab sizes V_h: consecutive primes >= N0; offsets O_h: exclusive
    prefix sum of V (one concatenated table of sum(V) rows).
  * ragged lengths: R - 1 distinct cut points uniform in [1, T - 1], sorted.
  * Zipf(s) tokens: rank k in [1, 131072] with P(k) proportional to k^-s,
    mapped to token ids through a seeded permutation of the vocabulary.
  * table rows ~ N(0, 0.02) in bf16; fp8 tables quantise N(0, 0.02) rows to
    e4m3 with a per-row float32 scale amax/448; kv_proj weight ~ N(0, 0.02);
    hidden ~ N(0, 1); gammas = 1 (tests also use 1 + N(0, 0.1)); conv taps
    ~ N(0, 1/K) (standard deviation 1/sqrt(K)); conv state ~ N(0, 0.01).
"""

from dataclasses import dataclass, replace

import numpy as np

EOS_TOKEN_ID = 2
TOKEN_VOCAB = 131072  # "128k vocab"
NGRAM_CONTEXT_LEN = 2  # n-gram orders 2 and 3


@dataclass(frozen=True)
class Workload:
    name: str
    num_tokens: int
    num_reqs: int
    fixed_lengths: tuple        # explicit request lengths, or () for random cuts
    token_vocab: int
    token_dist: str             # "uniform" or "zipf"
    zipf_s: float
    heads_per_ngram: int
    vocab_start: int            # N0: V_h are the consecutive primes >= N0
    head_dim: int
    table_dtype: str            # "bf16" or "fp8"
    table_loc: str              # "hbm" or "host" (pinned host memory read over UVA)
    hidden: int
    conv_k: int
    dilation: int
    num_layers: int
    decode: bool                # requests carry ngram_context and conv_state
    seed: int

    @property
    def num_heads(self):
        return NGRAM_CONTEXT_LEN * self.heads_per_ngram

    @property
    def emb_dim(self):
        return self.num_heads * self.head_dim

    @property
    def eos_token_id(self):
        return EOS_TOKEN_ID

    @property
    def ctx_len(self):
        return NGRAM_CONTEXT_LEN


WORKLOADS = {
    # 4 requests of 64/100/150/198 tokens, 8 heads over primes near 10007,
    # dim-64 rows, hidden 1024, kv_proj 512 -> 2 x 1024.
    "tiny": Workload("tiny", 512, 4, (64, 100, 150, 198), 32000, "uniform", 0.0,
                     4, 10007, 64, "bf16", "hbm", 1024, 4, 3, 1, False, 0),
    # 8192-token prefill over 16 ragged requests, 16 heads over primes near
    # 2M (32,002,074 rows x 128 bf16 = 8.2 GB in HBM), hidden 4096,
    # kv_proj 2048 -> 2 x 4096.
    "prefill8k": Workload("prefill8k", 8192, 16, (), TOKEN_VOCAB, "uniform", 0.0,
                          8, 2_000_000, 128, "bf16", "hbm", 4096, 4, 3, 1, False, 1),
    # 256 decode requests x 4 tokens, Zipf(1.1) tokens, per-request n-gram
    # context of the last 2 tokens and a conv state; table as prefill8k.
    "decode256x4": Workload("decode256x4", 1024, 256, (4,) * 256, TOKEN_VOCAB, "zipf", 1.1,
                            8, 2_000_000, 128, "bf16", "hbm", 4096, 4, 3, 1, True, 2),
    # prefill8k shapes with a 32 GiB bf16 table (primes near 2^23,
    # 134,219,512 rows) in pinned host memory, read over UVA.
    "uva32g": Workload("uva32g", 8192, 16, (), TOKEN_VOCAB, "uniform", 0.0,
                       8, 1 << 23, 128, "bf16", "host", 4096, 4, 3, 1, False, 3),
    # 8 layers, each with an 8 GiB fp8 e4m3 table slice (primes near 2^22,
    # 67,110,742 rows) plus a per-row float32 scale, 32768-token prefill over
    # 64 ragged requests, Zipf(1.1) tokens.
    "fp8x8": Workload("fp8x8", 32768, 64, (), TOKEN_VOCAB, "zipf", 1.1,
                      8, 1 << 22, 128, "fp8", "hbm", 4096, 4, 3, 8, False, 4),
}


def scaled(w, **changes):
    """A copy of workload ``w`` with some fields changed (for small test cases)."""
    return replace(w, **changes)


# ---------------------------------------------------------------------------
# integer inputs (host, numpy)
# ---------------------------------------------------------------------------

def _is_prime(n):
    if n < 2:
        return False
    if n % 2 == 0:
        return n == 2
    f = 3
    while f * f <= n:
        if n % f == 0:
            return False
        f += 2
    return True


def consecutive_primes(start, count):
    """The ``count`` smallest primes >= ``start``."""
    out = []
    n = start
    while len(out) < count:
        if _is_prime(n):
            out.append(n)
        n += 1
    return out


def head_vocab(w):
    """(V, O) int64 arrays: per-head vocab sizes and table-row offsets."""
    V = np.array(consecutive_primes(w.vocab_start, w.num_heads), dtype=np.int64)
    O = np.concatenate([[0], np.cumsum(V)[:-1]]).astype(np.int64)
    return V, O


def table_rows(w):
    V, _ = head_vocab(w)
    return int(V.sum())


def layer_multipliers(w, layer):
    rng = np.random.default_rng(w.seed * 1000 + layer)
    m = rng.integers(1 << 32, 1 << 62, size=NGRAM_CONTEXT_LEN + 1, dtype=np.int64)
    return m | np.int64(1)


def ragged_lengths(num_tokens, num_reqs, rng):
    if num_reqs == 1:
        return [num_tokens]
    cuts = np.sort(rng.choice(np.arange(1, num_tokens), size=num_reqs - 1, replace=False))
    bounds = np.concatenate([[0], cuts, [num_tokens]])
    return [int(x) for x in np.diff(bounds)]


def _zipf_tokens(n, vocab, s, rng):
    ranks = np.arange(1, vocab + 1, dtype=np.float64)
    cdf = np.cumsum(ranks ** (-s))
    cdf /= cdf[-1]
    perm = rng.permutation(vocab)
    k = np.searchsorted(cdf, rng.random(n), side="left")
    k = np.minimum(k, vocab - 1)
    return perm[k]


def draw_tokens(n, w, rng):
    if w.token_dist == "zipf":
        return _zipf_tokens(n, w.token_vocab, w.zipf_s, rng).astype(np.int32)
    return rng.integers(0, w.token_vocab, size=n, dtype=np.int64).astype(np.int32)


def host_inputs(w, step=0):
    """Integer inputs of one step of workload ``w``.

    Returns a dict: input_ids int32 [T], query_start_loc int32 [R+1],
    ngram_context int32 [R, 2] or None, lengths (list), V / O int64 [H],
    multipliers int64 [num_layers, 3].
    """
    rng = np.random.default_rng([w.seed, step, 17])
    if w.fixed_lengths:
        lengths = list(w.fixed_lengths)
        assert len(lengths) == w.num_reqs and sum(lengths) == w.num_tokens
    else:
        lengths = ragged_lengths(w.num_tokens, w.num_reqs, rng)
    qsl = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    input_ids = draw_tokens(w.num_tokens, w, rng)
    ctx = None
    if w.decode:
        ctx = draw_tokens(w.num_reqs * NGRAM_CONTEXT_LEN, w, rng).reshape(
            w.num_reqs, NGRAM_CONTEXT_LEN)
    V, O = head_vocab(w)
    mult = np.stack([layer_multipliers(w, layer) for layer in range(w.num_layers)])
    return {"input_ids": input_ids, "query_start_loc": qsl, "ngram_context": ctx,
            "lengths": lengths, "V": V, "O": O, "multipliers": mult}


# ---------------------------------------------------------------------------
# float inputs (torch, generated on the device that will hold them)
# ---------------------------------------------------------------------------

def _gen(torch, device, seed, tag):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1009 + int(tag))
    return g


def normal_bf16(torch, shape, std, device, seed, tag, mean=0.0):
    g = _gen(torch, device, seed, tag)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    return (x.mul_(std).add_(mean)).to(torch.bfloat16)


def fill_table_bf16(torch, out, seed, tag, chunk_rows=1 << 22):
    """Fill ``out`` [rows, D] bf16 (device or pinned host) with N(0, 0.02).

    Generated chunk by chunk on the current CUDA device when ``out`` is on the
    host (then copied), or in place on ``out``'s device.
    """
    rows = out.shape[0]
    gen_device = out.device if out.device.type == "cuda" else torch.device("cuda")
    if not torch.cuda.is_available():
        gen_device = torch.device("cpu")
    g = _gen(torch, gen_device, seed, tag)
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        x = torch.randn((r1 - r0, out.shape[1]), generator=g, device=gen_device,
                        dtype=torch.float32).mul_(0.02).to(torch.bfloat16)
        out[r0:r1].copy_(x, non_blocking=False)


def fill_table_fp8(torch, codes, scale, seed, tag, chunk_rows=1 << 22):
    """Fill ``codes`` [rows, D] uint8 (e4m3 bits) and ``scale`` [rows] float32.

    Each row is N(0, 0.02) quantised with scale = amax(|row|) / 448.
    """
    rows = codes.shape[0]
    g = _gen(torch, codes.device, seed, tag)
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        x = torch.randn((r1 - r0, codes.shape[1]), generator=g, device=codes.device,
                        dtype=torch.float32).mul_(0.02)
        s = x.abs().amax(dim=1).clamp_min(1e-12) / 448.0
        q = (x / s[:, None]).clamp_(-448.0, 448.0).to(torch.float8_e4m3fn)
        codes[r0:r1].copy_(q.view(torch.uint8))
        scale[r0:r1].copy_(s)


def dense_inputs(torch, w, device, layer=0, step=0, random_gamma=False):
    """Per-layer weights and per-step activations of workload ``w`` on ``device``.

    Returns a dict of torch tensors: w_kv [2C, E] bf16, gamma_h / gamma_k [C]
    bf16, conv_w [C, K] bf16, hidden [T, C] bf16 and, for decode workloads,
    conv_state [R, (K-1)*d, C] bf16. Tables are made separately
    (``make_table``) because of their size.
    """
    C, E, K = w.hidden, w.emb_dim, w.conv_k
    base = w.seed * 100 + layer
    out = {
        "w_kv": normal_bf16(torch, (2 * C, E), 0.02, device, base, 1),
        "conv_w": normal_bf16(torch, (C, K), 1.0 / np.sqrt(K), device, base, 2),
        "hidden": normal_bf16(torch, (w.num_tokens, C), 1.0, device, base + 7 * step, 3),
    }
    if random_gamma:
        out["gamma_h"] = normal_bf16(torch, (C,), 0.1, device, base, 4, mean=1.0)
        out["gamma_k"] = normal_bf16(torch, (C,), 0.1, device, base, 5, mean=1.0)
    else:
        out["gamma_h"] = torch.ones(C, dtype=torch.bfloat16, device=device)
        out["gamma_k"] = torch.ones(C, dtype=torch.bfloat16, device=device)
    if w.decode:
        W = (K - 1) * w.dilation
        out["conv_state"] = normal_bf16(torch, (w.num_reqs, W, C), 0.01, device,
                                        base + 7 * step, 6)
    return out


def make_table(torch, w, device, layer=0, rows=None):
    """The PLE table of one layer: (table, row_scale or None).

    bf16 tables are [rows, D] bfloat16; fp8 tables are [rows, D] uint8 e4m3
    codes plus [rows] float32 scales. ``w.table_loc == "host"`` gives a pinned
    host tensor (the scale, if any, stays on ``device``).
    """
    if rows is None:
        rows = table_rows(w)
    D = w.head_dim
    tag = 10 + layer
    if w.table_dtype == "fp8":
        codes = torch.empty((rows, D), dtype=torch.uint8, device=device)
        scale = torch.empty((rows,), dtype=torch.float32, device=device)
        fill_table_fp8(torch, codes, scale, w.seed, tag)
        if w.table_loc == "host":
            host = torch.empty((rows, D), dtype=torch.uint8, pin_memory=True)
            host.copy_(codes)
            del codes
            codes = host
        return codes, scale
    if w.table_loc == "host":
        # huge-page-backed registered host memory (see ple_host_table_alloc);
        # the HostTable owner rides along on the tensor to keep it alive
        from ._lib import HostTable
        owner = HostTable(rows, D, torch.bfloat16)
        table = owner.tensor
        table.host_table_owner = owner
    else:
        table = torch.empty((rows, D), dtype=torch.bfloat16, device=device)
    fill_table_bf16(torch, table, w.seed, tag)
    return table, None
