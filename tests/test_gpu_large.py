"""Parity past 32-bit element offsets: one layer of 270,077 tokens (8 ragged
requests, 16 heads x 128 bf16, hidden 4096) through PLELayer, so that kv
[T, 2C] holds 2.2 x 10^9 elements (more than 2^31) and every kernel has to
index its rows with 64-bit offsets. Checked against the oracle on sampled
windows, a third of them in the rows past 2^31 / 2C = 262,144: the ids bit for
bit (the oracle run on each window with the two tokens before it as n-gram
context), the gathered rows bit for bit, the value half of kv and the gate
scalars within the projection's tolerance, and y within the chain tolerance
(the window's own conv history)."""

import numpy as np
import pytest
import torch

import oracle
from hashed_gram_embedding_gb300 import PLELayer
from hashed_gram_embedding_gb300 import workloads as wl

from _helpers import CHAIN_ATOL_FRAC, assert_close, bits, dev_err_word

pytestmark = pytest.mark.gpu

T_LARGE = 270_077
BLOCK = 64


def windows(qsl, T, W, rng, n_low=8, n_high=4, first=10):
    """[(lo, a, b)]: window [lo, b) fed to the oracle, tokens [a, b) checked:
    every request's first `first` tokens, n_low random blocks anywhere and
    n_high blocks past row 262,144, each block with its W tokens of conv
    history and two more tokens of n-gram context inside its request."""
    spans = [(int(qsl[r]), int(qsl[r + 1]) if r + 1 < len(qsl) - 1 else T)
             for r in range(len(qsl) - 1)]
    out = [(s, s, min(e, s + first)) for s, e in spans if e > s]
    taken = []

    def pick(lo_bound, count):
        cands = [(max(s + first + W + 2, lo_bound), e) for s, e in spans]
        cands = [(s, e) for s, e in cands if e - s >= BLOCK]
        n = 0
        while n < count:
            s, e = cands[rng.integers(len(cands))]
            a = int(rng.integers(s, e - BLOCK + 1))
            if all(a + BLOCK <= x or a >= x + BLOCK for x in taken):
                taken.append(a)
                out.append((a - W, a, a + BLOCK))
                n += 1

    pick(0, n_low)
    pick(262_144 + 1, n_high)
    return out


def oracle_window_ids(host, qsl, w, lo, b):
    """The oracle's ids of tokens [lo, b) of one request, the two tokens
    before lo (EOS before the request start) as the n-gram context."""
    r = int(np.searchsorted(qsl[:-1], lo, side="right")) - 1
    s = int(qsl[r])
    toks = host["input_ids"]
    before = list(toks[max(s, lo - w.ctx_len):lo])
    ctx = [w.eos_token_id] * (w.ctx_len - len(before)) + [int(x) for x in before]
    ids, _ = oracle.ngram_ids(toks[lo:b], np.array([0, b - lo], dtype=np.int32),
                              np.array([ctx], dtype=np.int32), host["multipliers"][0], host["V"],
                              host["O"], w.eos_token_id, w.heads_per_ngram)
    return np.asarray(ids, dtype=np.int64).reshape(b - lo, -1)


def test_layer_past_2_31_elements():
    w = wl.scaled(wl.WORKLOADS["prefill8k"], name="large270k", num_tokens=T_LARGE, num_reqs=8,
                  vocab_start=65_536, seed=11)
    assert w.num_tokens * 2 * w.hidden > 2 ** 31
    host = wl.host_inputs(w)
    table, _ = wl.make_table(torch, w, "cuda")
    dense = wl.dense_inputs(torch, w, "cuda", random_gamma=True)
    layer = PLELayer(table, None, host["multipliers"][0], host["V"], host["O"], w.eos_token_id,
                     w.heads_per_ngram, dense["w_kv"], dense["gamma_h"], dense["gamma_k"],
                     dense["conv_w"], w.dilation)
    qsl = host["query_start_loc"]
    err = dev_err_word()
    y = layer.forward(torch.from_numpy(host["input_ids"]).cuda(), torch.from_numpy(qsl).cuda(),
                      dense["hidden"], dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    buf = layer.buffers(w.num_tokens, y.device)
    C = w.hidden
    blocks = windows(qsl, w.num_tokens, (w.conv_k - 1) * w.dilation, np.random.default_rng(5))
    assert sum(1 for _, a, _ in blocks if a > 262_144) >= 4

    # ids and rows, window by window; the oracle's kv once for every window row
    rows = np.unique(np.concatenate([np.arange(lo, b) for lo, _, b in blocks]))
    pos = {int(t): i for i, t in enumerate(rows)}
    ids = np.empty((len(rows), w.num_heads), dtype=np.int64)
    gpu_ids = buf["ids"][torch.from_numpy(rows).cuda()].cpu().numpy()
    for lo, _, b in blocks:
        ids[[pos[t] for t in range(lo, b)]] = oracle_window_ids(host, qsl, w, lo, b)
    assert np.array_equal(gpu_ids, ids)
    uniq, inv = np.unique(ids, return_inverse=True)
    emb = oracle.lookup_bf16(inv.reshape(ids.shape), bits(table[torch.from_numpy(uniq).cuda()]))
    d_rows = torch.from_numpy(rows).cuda()
    assert np.array_equal(bits(buf["emb"][d_rows]), emb)
    kv = oracle.kv_proj(emb, bits(dense["w_kv"]))
    assert_close(bits(buf["kv"][d_rows][:, C:]), kv[:, C:], what="v past 2^31 elements")
    gh, gk, cw = (bits(dense[k]) for k in ("gamma_h", "gamma_k", "conv_w"))
    hid = bits(dense["hidden"][d_rows])
    _, ref_g = oracle.gate(hid, kv, gh, gk, 1e-6)
    assert np.max(np.abs(buf["gate"][d_rows].cpu().numpy().astype(np.float64) - ref_g)) < 5e-4

    # y on each window, with the window's own conv history
    checked = 0
    for lo, a, b in blocks:
        idx = [pos[t] for t in range(lo, b)]
        ref_y, _, _ = oracle.gate_conv(hid[idx], kv[idx], gh, gk, 1e-6, [0, b - lo], cw,
                                       w.dilation)
        assert_close(bits(y[a:b]), ref_y[a - lo:], atol_frac=CHAIN_ATOL_FRAC,
                     what=f"tokens {a}..{b}")
        checked += b - a
    assert checked >= 12 * BLOCK
    del table, dense, layer, y
    torch.cuda.empty_cache()
