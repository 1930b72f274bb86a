"""GPU parity of ple_ngram_ids against the oracle: bit-exact ids and
carry-over, on hand cases, random ragged batches with overflowing and
negative multipliers, the tiny / decode / 8k-prefill / 32k-prefill workloads,
and the edge cases (empty requests, padding tokens, zero tokens, V = 1,
huge V, the largest context length, invalid query_start_loc)."""

import numpy as np
import pytest
import torch

from oracle import ngram_ids as oracle_ids
from hashed_gram_embedding_gb300 import _lib
from hashed_gram_embedding_gb300 import workloads as wl

from _helpers import dev_err_word
from test_oracle_ngram_ids import load_golden_cases, random_batch

pytestmark = pytest.mark.gpu


def run_gpu(tokens, qsl, ctx, mult, V, O, eos, hpn, with_ctx_out=True):
    dev = "cuda"
    T = len(tokens)
    R = len(qsl) - 1
    L = len(mult) - 1
    H = L * hpn
    t_tok = torch.tensor(np.asarray(tokens, dtype=np.int32).reshape(-1), dtype=torch.int32, device=dev)
    t_qsl = torch.tensor(np.asarray(qsl, dtype=np.int32), dtype=torch.int32, device=dev)
    t_ctx = None if ctx is None else torch.tensor(
        np.asarray(ctx, dtype=np.int32).reshape(R, L), dtype=torch.int32, device=dev)
    out = torch.full((T, H), -1, dtype=torch.int64, device=dev)
    ctx_out = torch.full((R, L), -7, dtype=torch.int32, device=dev) if with_ctx_out else None
    err = dev_err_word()
    _lib.ple_ngram_ids(t_tok, t_qsl, t_ctx, mult, V, O, eos, hpn, out, ctx_out, err)
    torch.cuda.synchronize()
    return (out.cpu().numpy(), None if ctx_out is None else ctx_out.cpu().numpy(),
            int(err.item()))


def check(tokens, qsl, ctx, mult, V, O, eos, hpn):
    ids, ctx_out = oracle_ids(tokens, qsl, ctx, mult, V, O, eos, hpn, num_tokens=len(tokens))
    g_ids, g_ctx, err = run_gpu(tokens, qsl, ctx, mult, V, O, eos, hpn)
    L = len(mult) - 1
    assert err == 0
    assert np.array_equal(g_ids, np.asarray(ids, dtype=np.int64).reshape(len(tokens), L * hpn))
    assert np.array_equal(g_ctx, np.asarray(ctx_out, dtype=np.int64).reshape(len(qsl) - 1, L))
    return g_ids


@pytest.mark.parametrize("case", load_golden_cases(), ids=lambda c: c["name"])
def test_hand_worked_cases(case):
    check(case["input_ids"], case["query_start_loc"], case["context"], case["multipliers"],
          [7, 11], [0, 7], 9, 1)


@pytest.mark.parametrize("seed", range(24))
def test_random_ragged_batches(seed):
    rng = np.random.default_rng(100 + seed)
    eos = 3
    hpn = int(rng.integers(1, 5))
    L = int(rng.integers(1, 4))
    V = [int(v) for v in rng.integers(1, 1 << int(rng.integers(2, 40)), size=L * hpn)]
    O = [int(o) for o in np.concatenate([[0], np.cumsum(V)[:-1]])]
    mult = [int(m) for m in rng.integers(-(1 << 63), (1 << 63) - 1, size=L + 1, dtype=np.int64)]
    tokens, qsl, ctx = random_batch(rng, int(rng.integers(1, 40)), 70, 12, eos, seed % 2 == 0)
    if ctx is not None and L != 2:
        ctx = rng.integers(0, 12, size=(len(qsl) - 1, L))
    if not tokens:
        tokens, qsl = [5], [0] + [1] * (len(qsl) - 1)
    check(tokens, qsl, ctx, mult, V, O, eos, hpn)


def test_padding_tokens_continue_last_request():
    check([5, 6, 7, 8, 9, 2, 4], [0, 2, 3], None, [11, 13, 17], [101, 103], [0, 101], 2, 1)


def test_extreme_vocab_sizes_and_context_length():
    rng = np.random.default_rng(7)
    L = 7
    hpn = 2
    V = [1, 2, (1 << 62) + 135, (1 << 63) - 25, 3, 10007, (1 << 63) - 1, 7, 1, 1 << 40,
         2_000_003, 8_388_617, 5, 11]
    # offsets small enough that offset + remainder stays inside int64
    O = [0, 5, 0, 0, 7, 9, 0, 11, 13, 1 << 20, 17, 19, 23, 29]
    mult = [int(m) for m in rng.integers(-(1 << 63), (1 << 63) - 1, size=L + 1, dtype=np.int64)]
    tokens, qsl, _ = random_batch(rng, 6, 30, 9, 4, False)
    ctx = rng.integers(0, 9, size=(6, L))
    check(tokens, qsl, ctx, mult, V, O, 4, hpn)


def test_tiny_workload():
    w = wl.WORKLOADS["tiny"]
    h = wl.host_inputs(w)
    check(h["input_ids"], h["query_start_loc"], None, h["multipliers"][0], h["V"], h["O"],
          w.eos_token_id, w.heads_per_ngram)


def test_decode_workload_with_context():
    w = wl.WORKLOADS["decode256x4"]
    h = wl.host_inputs(w)
    check(h["input_ids"], h["query_start_loc"], h["ngram_context"], h["multipliers"][0], h["V"],
          h["O"], w.eos_token_id, w.heads_per_ngram)


def test_prefill_8k_full_size():
    w = wl.WORKLOADS["prefill8k"]
    h = wl.host_inputs(w)
    ids = check(h["input_ids"], h["query_start_loc"], None, h["multipliers"][0], h["V"], h["O"],
                w.eos_token_id, w.heads_per_ngram)
    V, O = h["V"], h["O"]
    assert np.all((ids >= O) & (ids < O + V))


@pytest.mark.parametrize("layer", [0, 7])
def test_prefill_32k_zipf_layers(layer):
    w = wl.WORKLOADS["fp8x8"]
    h = wl.host_inputs(w)
    check(h["input_ids"], h["query_start_loc"], None, h["multipliers"][layer], h["V"], h["O"],
          w.eos_token_id, w.heads_per_ngram)


def test_zero_tokens_carry_over():
    mult, V, O = [3, 5, 7], [7, 11], [0, 7]
    _, ctx_out, err = run_gpu([], [0, 0, 0], None, mult, V, O, 9, 1)
    assert err == 0 and np.array_equal(ctx_out, np.full((2, 2), 9))
    _, ctx_out, err = run_gpu([], [0, 0, 0], [[1, 2], [3, 4]], mult, V, O, 9, 1)
    assert np.array_equal(ctx_out, [[1, 2], [3, 4]])


def test_invalid_query_start_loc_is_flagged_not_faulted():
    mult, V, O = [3, 5, 7], [7, 11], [0, 7]
    for qsl in ([0, 5, 3, 8], [2, 4, 6, 8], [0, 4, 6, 12], [0, -3, 6, 8]):
        ids, _, err = run_gpu(list(range(8)), qsl, None, mult, V, O, 9, 1)
        assert err & _lib.PLE_DEVERR_QSL
        assert np.all((ids >= O) & (ids < np.add(O, V)))


def test_empty_head_shard_rejected():
    with pytest.raises(_lib.PleError):
        run_gpu([1, 2], [0, 2], None, [1, 2, 3], [], [], 2, 0)


def test_many_requests_search_outside_shared_memory():
    # more boundaries than the kernel stages in shared memory
    rng = np.random.default_rng(11)
    lengths = rng.integers(0, 4, size=5000)
    qsl = [0] + [int(x) for x in np.cumsum(lengths)]
    tokens = [int(t) for t in rng.integers(0, 50, size=qsl[-1])]
    ctx = rng.integers(0, 50, size=(5000, 2))
    check(tokens, qsl, ctx, [7, -11, 13], [101, 103], [0, 101], 2, 1)
