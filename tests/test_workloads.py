"""The synthetic workload recipe: sizes of the pages' workloads, seeded and
reproducible, ragged boundaries well formed, Zipf tokens heavy-headed."""

import numpy as np

from hashed_gram_embedding_gb300 import workloads as wl


def test_table_sizes_of_each_workload():
    rows = {n: wl.table_rows(w) for n, w in wl.WORKLOADS.items()}
    assert rows["tiny"] == 80368
    assert rows["prefill8k"] == rows["decode256x4"] == 32002074
    assert rows["uva32g"] == 134219512
    assert rows["fp8x8"] == 67110742
    V, O = wl.head_vocab(wl.WORKLOADS["tiny"])
    assert list(V) == [10007, 10009, 10037, 10039, 10061, 10067, 10069, 10079]
    assert list(O) == list(np.concatenate([[0], np.cumsum(V)[:-1]]))


def test_primes_are_prime_and_consecutive():
    ps = wl.consecutive_primes(2_000_000, 16)
    assert ps[0] == 2_000_003 and ps[-1] == 2_000_249
    for a, b in zip(ps, ps[1:]):
        for n in range(a + 1, b):
            assert any(n % f == 0 for f in range(2, int(n ** 0.5) + 1))


def test_host_inputs_are_seeded_and_well_formed():
    for name, w in wl.WORKLOADS.items():
        a = wl.host_inputs(w)
        b = wl.host_inputs(w)
        assert np.array_equal(a["input_ids"], b["input_ids"])
        q = a["query_start_loc"]
        assert q[0] == 0 and q[-1] == w.num_tokens and np.all(np.diff(q) >= 0)
        assert len(q) == w.num_reqs + 1
        assert a["input_ids"].dtype == np.int32 and a["input_ids"].min() >= 0
        assert a["input_ids"].max() < w.token_vocab
        m = a["multipliers"]
        assert m.shape == (w.num_layers, 3) and np.all(m % 2 == 1) and np.all(m >= 1 << 32)
        assert (a["ngram_context"] is not None) == w.decode


def test_ragged_lengths_positive_and_sum():
    rng = np.random.default_rng(0)
    L = wl.ragged_lengths(8192, 16, rng)
    assert sum(L) == 8192 and len(L) == 16 and min(L) >= 1


def test_zipf_tokens_are_heavy_headed():
    w = wl.WORKLOADS["fp8x8"]
    toks = wl.host_inputs(w)["input_ids"]
    _, counts = np.unique(toks, return_counts=True)
    counts = np.sort(counts)[::-1]
    # Zipf(1.1) over 128k: the most frequent token carries a few percent of mass
    assert counts[0] / len(toks) > 0.02
    assert len(counts) < len(toks) // 2
