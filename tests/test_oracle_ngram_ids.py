"""Pins of the n-gram ID oracle.

Against: hand-worked golden values (tests/golden/ngram_ids_hand.txt), a
second, independently written enumerator (explicit n-gram tuples from
EOS-filled per-request rows, numpy int64 wrap-around and numpy floor-mod
instead of Python big ints), closed forms, invariants (range, no leakage
across requests, chunked prefill with carry-over == one prefill), and
``torch.remainder`` on int64 as a library check of the floor-mod of wrapped
values.
"""

import bisect
import os

import numpy as np
import pytest
import torch

from oracle import ngram_ids
from oracle.ngram_ids import wrap_int64

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "ngram_ids_hand.txt")


def _parse_rows(text):
    if text.strip() == "none":
        return None
    return [[int(v) for v in part.split()] for part in text.split("|")]


def load_golden_cases():
    cases, cur = [], None
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(" ")
            if key == "case":
                cur = {"name": rest}
            elif key == "end":
                cases.append(cur)
                cur = None
            elif key in ("multipliers", "query_start_loc", "input_ids"):
                cur[key] = [int(v) for v in rest.split()]
            else:
                cur[key] = _parse_rows(rest)
    return cases


@pytest.mark.parametrize("case", load_golden_cases(), ids=lambda c: c["name"])
def test_hand_worked_golden(case):
    ids, ctx_out = ngram_ids(case["input_ids"], case["query_start_loc"], case["context"],
                             case["multipliers"], [7, 11], [0, 7], 9, 1)
    assert ids == case["ids"]
    assert ctx_out == case["context_out"]


# ---------------------------------------------------------------------------
# independent enumerator
# ---------------------------------------------------------------------------

def brute_force_ids(input_ids, qsl, ctx, mult, V, O, eos, hpn):
    """Explicit n-gram tuples, hashed with numpy int64 arithmetic."""
    T = len(input_ids)
    R = len(qsl) - 1
    L = len(mult) - 1
    # one EOS-filled row per request: L history columns, then T token columns
    rows = np.full((R, L + T), eos, dtype=np.int64)
    if ctx is not None:
        rows[:, :L] = np.asarray(ctx, dtype=np.int64)
    col_of = []
    for pos in range(T):
        req = min(bisect.bisect_right(list(qsl), pos) - 1, R - 1)
        col = L + pos - qsl[req]
        rows[req, col] = input_ids[pos]
        col_of.append((req, col))
    m = np.asarray(mult, dtype=np.int64)
    out = np.zeros((T, L * hpn), dtype=np.int64)
    for pos in range(T):
        req, col = col_of[pos]
        for n in range(2, L + 2):
            gram = [int(rows[req, col - s]) for s in range(n)]  # newest first
            # EOS crossing: tokens behind an EOS (lag >= 1) become EOS
            for s in range(2, n):
                if eos in gram[1:s]:
                    gram[s] = eos
            with np.errstate(over="ignore"):
                terms = np.asarray(gram, dtype=np.int64) * m[:n]
            h = np.int64(0)
            for term in terms:
                h = np.bitwise_xor(h, term)
            for j in range(hpn):
                head = (n - 2) * hpn + j
                out[pos, head] = np.remainder(h, np.int64(V[head])) + O[head]
    # the carry-over: last L columns of each request's row
    ctx_out = []
    for r in range(R):
        end = (qsl[r + 1] if r + 1 < R else T)
        length = max(0, end - qsl[r])
        ctx_out.append([int(v) for v in rows[r, length:length + L]])
    return out, ctx_out


def random_batch(rng, num_reqs, max_len, vocab, eos, with_ctx):
    lengths = rng.integers(0, max_len + 1, size=num_reqs)
    qsl = [0] + list(np.cumsum(lengths))
    T = int(qsl[-1])
    tokens = rng.integers(0, vocab, size=T)
    # inject EOS often
    tokens[rng.random(T) < 0.2] = eos
    ctx = rng.integers(0, vocab, size=(num_reqs, 2)) if with_ctx else None
    if ctx is not None:
        ctx[rng.random((num_reqs, 2)) < 0.2] = eos
    return [int(t) for t in tokens], [int(q) for q in qsl], ctx


@pytest.mark.parametrize("seed", range(40))
def test_matches_brute_force_on_tiny_batches(seed):
    rng = np.random.default_rng(seed)
    eos = 3
    hpn = int(rng.integers(1, 4))
    V = [int(v) for v in rng.integers(1, 50, size=2 * hpn)]
    O = [int(o) for o in np.concatenate([[0], np.cumsum(V)[:-1]])]
    # multipliers that overflow int64, of both signs
    mult = [int(v) for v in rng.integers(-(1 << 63), (1 << 63) - 1, size=3, dtype=np.int64)]
    tokens, qsl, ctx = random_batch(rng, int(rng.integers(1, 6)), 6, 8, eos, seed % 2 == 0)
    ids, ctx_out = ngram_ids(tokens, qsl, None if ctx is None else ctx.tolist(), mult, V, O, eos, hpn)
    bf_ids, bf_ctx = brute_force_ids(tokens, qsl, ctx, mult, V, O, eos, hpn)
    assert np.array_equal(np.asarray(ids, dtype=np.int64).reshape(len(tokens), 2 * hpn), bf_ids)
    assert ctx_out == bf_ctx


def test_padding_tokens_join_last_request():
    # query_start_loc[-1] < T: the trailing tokens continue the last request
    tokens = [5, 6, 7, 8, 9]
    qsl = [0, 2, 3]
    mult = [11, 13, 17]
    V, O = [101, 103], [0, 101]
    ids, ctx_out = ngram_ids(tokens, qsl, None, mult, V, O, 2, 1)
    bf_ids, bf_ctx = brute_force_ids(tokens, qsl, None, mult, V, O, 2, 1)
    assert np.array_equal(np.asarray(ids), bf_ids)
    assert ctx_out == bf_ctx == [[5, 6], [8, 9]]


# ---------------------------------------------------------------------------
# closed forms
# ---------------------------------------------------------------------------

def test_unit_multiplier_on_current_token():
    rng = np.random.default_rng(1)
    tokens, qsl, _ = random_batch(rng, 4, 10, 1000, 2, False)
    V = [97, 89, 83, 79]
    O = [0, 97, 186, 269]
    ids, _ = ngram_ids(tokens, qsl, None, [1, 0, 0], V, O, 2, 2)
    for t, row in enumerate(ids):
        assert row == [tokens[t] % V[h] + O[h] for h in range(4)]


def test_unit_multiplier_on_previous_token():
    tokens = [10, 20, 30, 40, 50]
    qsl = [0, 3, 5]
    eos = 2
    V, O = [7, 11], [0, 7]
    ids, _ = ngram_ids(tokens, qsl, None, [0, 1, 0], V, O, eos, 1)
    prev = [eos, 10, 20, eos, 40]  # request starts see EOS
    for t in range(5):
        assert ids[t] == [prev[t] % 7, prev[t] % 11 + 7]


def test_all_eos_is_constant_per_head():
    eos = 5
    mult = [(1 << 61) + 3, -(1 << 60) + 7, 12345]
    V, O = [13, 17, 19, 23], [0, 13, 30, 49]
    ids, _ = ngram_ids([eos] * 9, [0, 4, 9], None, mult, V, O, eos, 2)
    first = ids[0]
    assert all(row == first for row in ids)


# ---------------------------------------------------------------------------
# invariants
# ---------------------------------------------------------------------------

def test_ids_in_head_partition():
    rng = np.random.default_rng(2)
    tokens, qsl, ctx = random_batch(rng, 8, 30, 5000, 2, True)
    V = [10007, 10009, 10037, 10039]
    O = [0, 10007, 20016, 30053]
    mult = [int(v) for v in rng.integers(1 << 32, 1 << 62, size=3)]
    ids, _ = ngram_ids(tokens, qsl, ctx.tolist(), mult, V, O, 2, 2)
    for row in ids:
        for h, v in enumerate(row):
            assert O[h] <= v < O[h] + V[h]


def test_no_leakage_across_requests():
    rng = np.random.default_rng(3)
    tokens, qsl, ctx = random_batch(rng, 5, 12, 100, 2, True)
    mult = [int(v) for v in rng.integers(1 << 32, 1 << 62, size=3)]
    V, O = [31, 37], [0, 31]
    base, _ = ngram_ids(tokens, qsl, ctx.tolist(), mult, V, O, 2, 1)
    for r in range(5):
        changed = list(tokens)
        for t in range(qsl[r], qsl[r + 1]):
            changed[t] = (changed[t] + 7) % 100
        ids, _ = ngram_ids(changed, qsl, ctx.tolist(), mult, V, O, 2, 1)
        for t in range(len(tokens)):
            if not (qsl[r] <= t < qsl[r + 1]):
                assert ids[t] == base[t]


def test_chunked_prefill_with_carry_over_equals_single_pass():
    rng = np.random.default_rng(4)
    lengths = [17, 1, 9, 0, 25]
    eos = 2
    full_tokens = [list(rng.integers(0, 50, size=n)) for n in lengths]
    for toks in full_tokens:
        for i in range(len(toks)):
            if rng.random() < 0.15:
                toks[i] = eos
    mult = [int(v) for v in rng.integers(1 << 32, 1 << 62, size=3)]
    V, O = [53, 59, 61, 67], [0, 53, 112, 173]

    def run(chunks, ctx):
        qsl = [0] + list(np.cumsum([len(c) for c in chunks]))
        flat = [int(t) for c in chunks for t in c]
        return ngram_ids(flat, qsl, ctx, mult, V, O, eos, 2)

    one_ids, one_ctx = run(full_tokens, None)
    # split every request at a random point, run the two halves in sequence
    cut = [int(rng.integers(0, n + 1)) for n in lengths]
    a_ids, a_ctx = run([t[:c] for t, c in zip(full_tokens, cut)], None)
    b_ids, b_ctx = run([t[c:] for t, c in zip(full_tokens, cut)], a_ctx)
    # reassemble per request
    one_by_req, k = [], 0
    for n in lengths:
        one_by_req.append(one_ids[k:k + n])
        k += n
    ka = kb = 0
    for r, n in enumerate(lengths):
        first = a_ids[ka:ka + cut[r]]
        second = b_ids[kb:kb + n - cut[r]]
        ka += cut[r]
        kb += n - cut[r]
        assert first + second == one_by_req[r]
    assert b_ctx == one_ctx


def test_floor_mod_of_wrapped_values_matches_torch_remainder():
    rng = np.random.default_rng(5)
    mixed = list(rng.integers(-(1 << 63), (1 << 63) - 1, size=2000, dtype=np.int64))
    mixed += [-(1 << 63), (1 << 63) - 1, -1, 0, 1]
    divisors = [1, 2, 3, 7, 10007, 2_000_003, 8_388_617, (1 << 62) + 135, (1 << 63) - 25]
    t_mixed = torch.tensor([int(m) for m in mixed], dtype=torch.int64)
    for V in divisors:
        ref = torch.remainder(t_mixed, V).tolist()
        # the oracle's step: Python floor-mod of the wrapped int64 value
        ours = [wrap_int64(int(m)) % V for m in mixed]
        assert ours == ref


def test_wrap_int64_definition():
    assert wrap_int64(1 << 63) == -(1 << 63)
    assert wrap_int64((1 << 64) + 5) == 5
    assert wrap_int64(-(1 << 63) - 1) == (1 << 63) - 1
    # agrees with numpy's silent int64 wrap on products
    rng = np.random.default_rng(6)
    a = rng.integers(-(1 << 63), (1 << 63) - 1, size=500, dtype=np.int64)
    b = rng.integers(-(1 << 31), (1 << 31) - 1, size=500, dtype=np.int64)
    with np.errstate(over="ignore"):
        prod = a * b
    assert [wrap_int64(int(x) * int(y)) for x, y in zip(a, b)] == [int(p) for p in prod]
