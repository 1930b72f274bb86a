"""GPU parity of the whole per-layer chain (PLELayer.forward: ids -> gather ->
kv_proj -> gate + conv; by default the ids are hashed inside the gather
(ple_ngram_lookup; fuse_ids=False runs ple_ngram_ids + ple_lookup) and the
projection does the gate's reductions, ple_kv_proj_gate + ple_gated_conv
(fuse_gate=False runs ple_kv_proj + ple_gate_conv)) against the oracle's layer_forward: the tiny workload with a
bf16 and with an fp8 table (every token, both projections), the decode
workload's carry-over outputs, and the 8k prefill at full size (sampled
tokens with their conv windows); the four-layer chain (PLEChain, with and
without cross-layer prefetch) and layers over host tables against the same
oracle."""

import numpy as np
import pytest
import torch

import oracle
from hashed_gram_embedding_gb300 import PLELayer
from hashed_gram_embedding_gb300 import workloads as wl

from _helpers import CHAIN_ATOL_FRAC, assert_close, bits, dev_err_word, tiny_case

pytestmark = pytest.mark.gpu


def build_layer(w, host, dense, table, row_scale, layer=0, fuse_gate=None, fuse_ids=None):
    return PLELayer(table, row_scale, host["multipliers"][layer], host["V"], host["O"],
                    w.eos_token_id, w.heads_per_ngram, dense["w_kv"], dense["gamma_h"],
                    dense["gamma_k"], dense["conv_w"], w.dilation, fuse_gate=fuse_gate,
                    fuse_ids=fuse_ids)


@pytest.mark.parametrize("fuse_ids", [True, False])
@pytest.mark.parametrize("fuse_gate", [True, False])
@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_tiny_chain_every_token(dtype, fuse_gate, fuse_ids):
    w = wl.scaled(wl.WORKLOADS["tiny"], table_dtype=dtype)
    w, host, dense, table, row_scale = tiny_case(w)
    d_dense = {k: v.cuda() for k, v in dense.items()}
    layer = build_layer(w, host, d_dense, table.cuda(),
                        None if row_scale is None else row_scale.cuda(), fuse_gate=fuse_gate,
                        fuse_ids=fuse_ids)
    assert layer.fuse_gate == fuse_gate and layer.fuse_ids == fuse_ids
    err = dev_err_word()
    qsl = torch.from_numpy(host["query_start_loc"]).cuda()
    y = layer.forward(torch.from_numpy(host["input_ids"]).cuda(), qsl, d_dense["hidden"],
                      dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    host_table = bits(table) if row_scale is None else table.numpy()
    ref = oracle.layer_forward(host["input_ids"], host["query_start_loc"], None,
                               host["multipliers"][0], host["V"], host["O"], w.eos_token_id,
                               w.heads_per_ngram, host_table,
                               None if row_scale is None else row_scale.numpy(),
                               bits(dense["hidden"]), bits(dense["w_kv"]), bits(dense["gamma_h"]),
                               bits(dense["gamma_k"]), 1e-6, bits(dense["conv_w"]), w.dilation)
    b = layer.buffers(w.num_tokens, y.device)
    assert np.array_equal(b["ids"].cpu().numpy(), ref["ids"])
    assert np.array_equal(bits(b["emb"]), ref["emb"])
    tol = 1e-2 if dtype == "bf16" else 3e-2
    C = w.hidden
    cols = slice(C, 2 * C) if fuse_gate else slice(0, 2 * C)  # fused: k is never stored
    assert_close(bits(b["kv"])[:, cols], ref["kv"][:, cols], rtol=tol, atol_frac=tol, what="kv")
    assert_close(bits(y), ref["y"], rtol=tol, atol_frac=max(tol, CHAIN_ATOL_FRAC), what="y")


def test_decode_chain_carry_over():
    w = wl.scaled(wl.WORKLOADS["decode256x4"], hidden=256, vocab_start=5000, num_reqs=64,
                  num_tokens=256, fixed_lengths=(4,) * 64)
    host = wl.host_inputs(w)
    dense = wl.dense_inputs(torch, w, "cpu", random_gamma=True)
    rows = wl.table_rows(w)
    g = torch.Generator().manual_seed(5)
    table = (torch.randn((rows, w.head_dim), generator=g) * 0.02).to(torch.bfloat16)
    d = {k: v.cuda() for k, v in dense.items()}
    layer = build_layer(w, host, d, table.cuda(), None)
    ctx_in = torch.from_numpy(host["ngram_context"]).cuda()
    ctx_out = torch.empty_like(ctx_in)
    st_out = torch.empty_like(d["conv_state"])
    y = layer.forward(torch.from_numpy(host["input_ids"]).cuda(),
                      torch.from_numpy(host["query_start_loc"]).cuda(), d["hidden"],
                      ngram_context=ctx_in, ngram_context_out=ctx_out,
                      conv_state=d["conv_state"], conv_state_out=st_out)
    torch.cuda.synchronize()
    ref = oracle.layer_forward(host["input_ids"], host["query_start_loc"], host["ngram_context"],
                               host["multipliers"][0], host["V"], host["O"], w.eos_token_id,
                               w.heads_per_ngram, bits(table), None, bits(dense["hidden"]),
                               bits(dense["w_kv"]), bits(dense["gamma_h"]), bits(dense["gamma_k"]),
                               1e-6, bits(dense["conv_w"]), w.dilation, bits(dense["conv_state"]))
    assert np.array_equal(ctx_out.cpu().numpy(), np.asarray(ref["ngram_context_out"]))
    assert_close(bits(y), ref["y"], atol_frac=CHAIN_ATOL_FRAC, what="decode y")
    assert_close(bits(st_out), ref["conv_state_out"], atol_frac=CHAIN_ATOL_FRAC,
                 what="decode state")


def test_decode_256x4_full_size():
    """The decode workload at full size (256 requests x 4 tokens, n-gram
    context and conv state carried over, hidden 4096, the 8.2 GB table)
    through PLELayer (ids hashed inside the gather): ids, carry-over of both
    kinds and y of every token against the oracle."""
    w = wl.WORKLOADS["decode256x4"]
    host = wl.host_inputs(w)
    table, _ = wl.make_table(torch, w, "cuda")
    dense = wl.dense_inputs(torch, w, "cuda", random_gamma=True)
    layer = build_layer(w, host, dense, table, None)
    qsl = host["query_start_loc"]
    ctx_in = torch.from_numpy(host["ngram_context"]).cuda()
    ctx_out = torch.empty_like(ctx_in)
    st_out = torch.empty_like(dense["conv_state"])
    err = dev_err_word()
    y = layer.forward(torch.from_numpy(host["input_ids"]).cuda(), torch.from_numpy(qsl).cuda(),
                      dense["hidden"], ngram_context=ctx_in, ngram_context_out=ctx_out,
                      conv_state=dense["conv_state"], conv_state_out=st_out, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0 and layer.fused_ids_for(w.num_tokens)
    ids, ref_ctx = oracle.ngram_ids(host["input_ids"], qsl, host["ngram_context"],
                                    host["multipliers"][0], host["V"], host["O"],
                                    w.eos_token_id, w.heads_per_ngram)
    ids = np.asarray(ids, dtype=np.int64).reshape(w.num_tokens, -1)
    assert np.array_equal(layer.buffers(w.num_tokens, y.device)["ids"].cpu().numpy(), ids)
    assert np.array_equal(ctx_out.cpu().numpy(), np.asarray(ref_ctx).reshape(ctx_out.shape))
    uniq, inv = np.unique(ids, return_inverse=True)
    emb = oracle.lookup_bf16(inv.reshape(ids.shape), bits(table[torch.from_numpy(uniq).cuda()]))
    kv = oracle.kv_proj(emb, bits(dense["w_kv"]))
    ref_y, ref_st, _ = oracle.gate_conv(bits(dense["hidden"]), kv, bits(dense["gamma_h"]),
                                        bits(dense["gamma_k"]), 1e-6, qsl, bits(dense["conv_w"]),
                                        w.dilation, bits(dense["conv_state"]))
    assert_close(bits(y), ref_y, atol_frac=CHAIN_ATOL_FRAC, what="decode y")
    assert_close(bits(st_out), ref_st, atol_frac=CHAIN_ATOL_FRAC, what="decode conv state")
    del table
    torch.cuda.empty_cache()


def sampled_blocks(qsl, T, W, rng, n_blocks=30, block=64, first=10):
    """Token ranges checked at full size: every request's first `first`
    tokens, and `n_blocks` random blocks of `block` tokens inside requests,
    each with the W tokens of history before it (its window starts at the
    request start or W tokens earlier, so every checked token sees all its
    taps). Returns [(lo, a, b)]: window [lo, b), checked tokens [a, b)."""
    out = []
    for r in range(len(qsl) - 1):
        s, e = int(qsl[r]), int(qsl[r + 1]) if r + 1 < len(qsl) - 1 else T
        if e > s:
            out.append((s, s, min(e, s + first)))
    spans = [(int(qsl[r]), int(qsl[r + 1]) if r + 1 < len(qsl) - 1 else T)
             for r in range(len(qsl) - 1)]
    long_spans = [(s, e) for s, e in spans if e - s >= block + W + first]
    taken = []
    while len(taken) < n_blocks:  # blocks that do not overlap one another
        s, e = long_spans[rng.integers(len(long_spans))]
        a = int(rng.integers(s + first + W, e - block + 1))
        if all(a + block <= x or a >= x + block for x in taken):
            taken.append(a)
            out.append((a - W, a, a + block))
    return out


def check_chain_sampled(w, host, dense, table_bits_of, row_scale_of, y, ids, blocks):
    """The oracle's layer on the sampled windows (kv computed once for all
    their rows) against y, chain tolerance."""
    qsl = host["query_start_loc"]
    rows = np.unique(np.concatenate([np.arange(lo, b) for lo, _, b in blocks]))
    pos = {int(t): i for i, t in enumerate(rows)}
    win_ids = ids[rows]
    uniq, inv = np.unique(win_ids, return_inverse=True)
    if row_scale_of is None:
        emb = oracle.lookup_bf16(inv.reshape(win_ids.shape), table_bits_of(uniq))
    else:
        emb = oracle.lookup_fp8(inv.reshape(win_ids.shape), table_bits_of(uniq), row_scale_of(uniq))
    kv = oracle.kv_proj(emb, bits(dense["w_kv"]))
    gh, gk, cw = (bits(dense[k]) for k in ("gamma_h", "gamma_k", "conv_w"))
    hid = bits(dense["hidden"])
    yb = bits(y)
    checked = 0
    for lo, a, b in blocks:
        idx = [pos[t] for t in range(lo, b)]
        ref_y, _, _ = oracle.gate_conv(hid[lo:b], kv[idx], gh, gk, 1e-6, [0, b - lo], cw,
                                       w.dilation)
        assert_close(yb[a:b], ref_y[a - lo:], atol_frac=CHAIN_ATOL_FRAC, what=f"tokens {a}..{b}")
        checked += b - a
    return checked  # distinct tokens: the blocks do not overlap each other or the first ones


def test_prefill_8k_chain_sampled():
    """The 8k prefill at full size (8.2 GB table) through PLELayer: every id
    bit for bit, and y against the oracle on >= 2048 sampled tokens (every
    request's first 10 and 30 blocks of 64 with their conv history)."""
    w = wl.WORKLOADS["prefill8k"]
    host = wl.host_inputs(w)
    table, _ = wl.make_table(torch, w, "cuda")
    dense = wl.dense_inputs(torch, w, "cuda", random_gamma=True)
    layer = build_layer(w, host, dense, table, None)
    qsl = host["query_start_loc"]
    err = dev_err_word()
    y = layer.forward(torch.from_numpy(host["input_ids"]).cuda(), torch.from_numpy(qsl).cuda(),
                      dense["hidden"], dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ids, _ = oracle.ngram_ids(host["input_ids"], qsl, None, host["multipliers"][0], host["V"],
                              host["O"], w.eos_token_id, w.heads_per_ngram)
    ids = np.asarray(ids, dtype=np.int64).reshape(w.num_tokens, -1)
    assert np.array_equal(layer.buffers(w.num_tokens, y.device)["ids"].cpu().numpy(), ids)
    blocks = sampled_blocks(qsl, w.num_tokens, (w.conv_k - 1) * w.dilation,
                            np.random.default_rng(2))
    n = check_chain_sampled(w, host, dense,
                            lambda u: bits(table[torch.from_numpy(u).cuda()]), None, y, ids,
                            blocks)
    assert n >= 2048
    del table
    torch.cuda.empty_cache()


def test_fp8_32k_layer_sampled():
    """One layer of the 32k-token fp8 workload at full size (8 GiB e4m3 table
    with per-row scales, Zipf tokens): every id bit for bit, y against the
    oracle on >= 2048 sampled tokens."""
    w = wl.WORKLOADS["fp8x8"]
    host = wl.host_inputs(w)
    codes, scale = wl.make_table(torch, w, "cuda", layer=3)
    dense = wl.dense_inputs(torch, w, "cuda", layer=3, random_gamma=True)
    layer = build_layer(w, host, dense, codes, scale, layer=3)
    qsl = host["query_start_loc"]
    err = dev_err_word()
    y = layer.forward(torch.from_numpy(host["input_ids"]).cuda(), torch.from_numpy(qsl).cuda(),
                      dense["hidden"], dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ids, _ = oracle.ngram_ids(host["input_ids"], qsl, None, host["multipliers"][3], host["V"],
                              host["O"], w.eos_token_id, w.heads_per_ngram)
    ids = np.asarray(ids, dtype=np.int64).reshape(w.num_tokens, -1)
    assert np.array_equal(layer.buffers(w.num_tokens, y.device)["ids"].cpu().numpy(), ids)
    blocks = sampled_blocks(qsl, w.num_tokens, (w.conv_k - 1) * w.dilation,
                            np.random.default_rng(3), n_blocks=24)
    sel = lambda u: torch.from_numpy(u).cuda()
    n = check_chain_sampled(w, host, dense, lambda u: codes[sel(u)].cpu().numpy(),
                            lambda u: scale[sel(u)].cpu().numpy(), y, ids, blocks)
    assert n >= 2048
    del codes, scale
    torch.cuda.empty_cache()


@pytest.mark.parametrize("graphs", [True, False])
@pytest.mark.parametrize("depth", [1, 2, 3])
def test_host_pipeline_matches_layer(depth, graphs):
    """PLEHostPipeline over pinned host buffers (transfers overlapping
    compute) gives, step by step, exactly what PLELayer.forward gives on the
    same inputs; every step has its own tokens and hidden states. With
    graphs, each slot's steps after its first replay a captured graph."""
    from hashed_gram_embedding_gb300 import PLEHostPipeline
    w, host, dense, table, row_scale = tiny_case(wl.WORKLOADS["tiny"])
    d_dense = {k: v.cuda() for k, v in dense.items()}
    layer = build_layer(w, host, d_dense, table.cuda(), None)
    T, C = w.num_tokens, w.hidden
    steps = 8
    rng = np.random.default_rng(3)
    g = torch.Generator().manual_seed(4)
    h_ids = [torch.from_numpy(rng.integers(0, w.token_vocab, T).astype(np.int32)).pin_memory()
             for _ in range(steps)]
    h_qsl = torch.from_numpy(host["query_start_loc"]).pin_memory()
    h_hidden = [torch.randn((T, C), generator=g).to(torch.bfloat16).pin_memory()
                for _ in range(steps)]
    h_out = [torch.empty((T, C), dtype=torch.bfloat16).pin_memory() for _ in range(steps)]
    pipe = PLEHostPipeline(layer, T, len(host["query_start_loc"]) - 1, "cuda", depth=depth,
                           graphs=graphs)
    err = dev_err_word()
    for k in range(steps):
        pipe.submit(h_ids[k], h_qsl, h_hidden[k], h_out[k], dev_err=err)
    pipe.synchronize()
    assert int(err.item()) == 0
    d_qsl = h_qsl.cuda()
    for k in range(steps):
        want = layer.forward(h_ids[k].cuda(), d_qsl, h_hidden[k].cuda()).clone()
        torch.cuda.synchronize()
        assert torch.equal(h_out[k].view(torch.int16), want.cpu().view(torch.int16)), f"step {k}"


def test_host_pipeline_carry_over_ping_pong():
    """Decode-style steps through PLEHostPipeline: the n-gram context and the
    conv state alternate between two device buffers (step k reads set k % 2
    and writes the other), so the argument tensors, and with them the
    captured graphs, alternate too. From the fifth step on every step is one
    native ple_step call replaying a graph. Step by step the host outputs and
    the final carry-over equal sequential PLELayer.forward calls."""
    from hashed_gram_embedding_gb300 import PLEHostPipeline
    w, host, dense, table, _ = tiny_case(decode=True)
    d_dense = {k: v.cuda() for k, v in dense.items()}
    layer = build_layer(w, host, d_dense, table.cuda(), None)
    T, C, R = w.num_tokens, w.hidden, w.num_reqs
    steps = 10
    rng = np.random.default_rng(8)
    g = torch.Generator().manual_seed(9)
    h_ids = [torch.from_numpy(rng.integers(0, w.token_vocab, T).astype(np.int32)).pin_memory()
             for _ in range(steps)]
    h_qsl = torch.from_numpy(host["query_start_loc"]).pin_memory()
    h_hidden = [torch.randn((T, C), generator=g).to(torch.bfloat16).pin_memory()
                for _ in range(steps)]
    h_out = [torch.empty((T, C), dtype=torch.bfloat16).pin_memory() for _ in range(steps)]

    def carry():
        ctx0 = torch.from_numpy(host["ngram_context"]).cuda()
        st0 = d_dense["conv_state"].clone()
        return [ctx0, torch.empty_like(ctx0)], [st0, torch.empty_like(st0)]

    ctx, st = carry()
    pipe = PLEHostPipeline(layer, T, R, "cuda", depth=2)
    err = dev_err_word()
    done = None
    for k in range(steps):
        a, b = k % 2, (k + 1) % 2
        done = pipe.submit(h_ids[k], h_qsl, h_hidden[k], h_out[k], ngram_context=ctx[a],
                           ngram_context_out=ctx[b], conv_state=st[a], conv_state_out=st[b],
                           dev_err=err)
    done.synchronize()  # the last step's read-back
    assert int(err.item()) == 0
    assert len(pipe._graphs) == 2
    rctx, rst = carry()
    d_qsl = h_qsl.cuda()
    for k in range(steps):
        a, b = k % 2, (k + 1) % 2
        want = layer.forward(h_ids[k].cuda(), d_qsl, h_hidden[k].cuda(), ngram_context=rctx[a],
                             ngram_context_out=rctx[b], conv_state=rst[a],
                             conv_state_out=rst[b]).clone()
        torch.cuda.synchronize()
        assert torch.equal(h_out[k].view(torch.int16), want.cpu().view(torch.int16)), f"step {k}"
    assert torch.equal(ctx[steps % 2], rctx[steps % 2])
    assert torch.equal(st[steps % 2].view(torch.int16), rst[steps % 2].view(torch.int16))
    pipe.close()


def test_host_pipeline_rejects_mismatched_host_buffers():
    from hashed_gram_embedding_gb300 import PLEHostPipeline
    w, host, dense, table, _ = tiny_case()
    layer = build_layer(w, host, {k: v.cuda() for k, v in dense.items()}, table.cuda(), None)
    T, C = w.num_tokens, w.hidden
    pipe = PLEHostPipeline(layer, T, w.num_reqs, "cuda", depth=1)
    ids = torch.zeros((T,), dtype=torch.int32)
    qsl = torch.from_numpy(host["query_start_loc"])
    out = torch.empty((T, C), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="host input 2"):
        pipe.submit(ids, qsl, torch.zeros((T, C), dtype=torch.float32), out)
    with pytest.raises(ValueError, match="host input 0"):
        pipe.submit(ids[:-1], qsl, torch.zeros((T, C), dtype=torch.bfloat16), out)
    with pytest.raises(ValueError, match="host output"):
        pipe.submit(ids, qsl, torch.zeros((T, C), dtype=torch.bfloat16), out.cuda())
    pipe.close()
    with pytest.raises(RuntimeError, match="after close"):
        pipe.submit(ids, qsl, torch.zeros((T, C), dtype=torch.bfloat16), out)


@pytest.mark.parametrize("prefetch", [True, False])
@pytest.mark.parametrize("on_host", [False, True])
def test_chain_matches_layers(prefetch, on_host):
    """PLEChain over four layers (own multipliers, tables, weights, hidden
    states, conv states) gives each layer's PLELayer.forward output bit for
    bit, with the next layers' ids and gathers prefetched on a side stream or
    run in line; tables in HBM, or in host memory (ordered gather)."""
    from hashed_gram_embedding_gb300 import PLEChain, _lib
    L = 4
    w = wl.scaled(wl.WORKLOADS["tiny"], num_layers=L, decode=True)
    layers, hiddens, states, owners = [], [], [], []
    host = None
    for i in range(L):
        w_i, host_i, dense, table, _ = tiny_case(w, seed_step=i)
        host = host or host_i
        d = {k: v.cuda() for k, v in dense.items()}
        if on_host:
            owner = _lib.HostTable(table.shape[0], table.shape[1], torch.bfloat16)
            owner.tensor.copy_(table)
            owners.append(owner)
            tab = owner.tensor
        else:
            tab = table.cuda()
        layers.append(PLELayer(tab, None, host["multipliers"][i], host["V"], host["O"],
                               w.eos_token_id, w.heads_per_ngram, d["w_kv"], d["gamma_h"],
                               d["gamma_k"], d["conv_w"], w.dilation))
        hiddens.append(d["hidden"])
        states.append(d["conv_state"])
    T, C = w.num_tokens, w.hidden
    ids = torch.from_numpy(host["input_ids"]).cuda()
    qsl = torch.from_numpy(host["query_start_loc"]).cuda()
    ctx = torch.from_numpy(host["ngram_context"]).cuda()
    outs = [torch.empty((T, C), dtype=torch.bfloat16, device="cuda") for _ in range(L)]
    st_out = [torch.empty_like(s) for s in states]
    ctx_out = torch.empty_like(ctx)
    err = dev_err_word()
    PLEChain(layers, prefetch=prefetch, prefetch_ctas=76).forward(
        ids, qsl, hiddens, outs, ngram_context=ctx, ngram_context_out=ctx_out,
        conv_states=states, conv_states_out=st_out, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for i in range(L):
        so = torch.empty_like(states[i])
        co = torch.empty_like(ctx)
        want = layers[i].forward(ids, qsl, hiddens[i], ngram_context=ctx, ngram_context_out=co,
                                 conv_state=states[i], conv_state_out=so).clone()
        torch.cuda.synchronize()
        assert torch.equal(outs[i].view(torch.int16), want.view(torch.int16)), f"layer {i}"
        assert torch.equal(st_out[i].view(torch.int16), so.view(torch.int16)), f"state {i}"
        if i == 0:
            assert torch.equal(ctx_out, co)
    for o in owners:
        o.close()


@pytest.mark.parametrize("on_host", [False, True])
def test_layer_in_cuda_graph_matches_eager(on_host):
    """PLELayer.forward captured once into a CUDA graph and replayed gives the
    eager result bit for bit; replays pick up new inputs written into the
    captured buffers."""
    from hashed_gram_embedding_gb300 import _lib
    w, host, dense, table, _ = tiny_case(wl.WORKLOADS["tiny"])
    d = {k: v.cuda() for k, v in dense.items()}
    owner = None
    if on_host:
        owner = _lib.HostTable(table.shape[0], table.shape[1], torch.bfloat16)
        owner.tensor.copy_(table)
        tab = owner.tensor
    else:
        tab = table.cuda()
    layer = build_layer(w, host, d, tab, None)
    ids = torch.from_numpy(host["input_ids"]).cuda()
    qsl = torch.from_numpy(host["query_start_loc"]).cuda()
    hidden = d["hidden"].clone()
    out = torch.empty_like(hidden)
    err = dev_err_word()
    layer.forward(ids, qsl, hidden, out=out, dev_err=err)  # buffers exist before capture
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        layer.forward(ids, qsl, hidden, out=out, dev_err=err, stream=s)
    for k in range(2):
        ids.copy_(torch.from_numpy(np.random.default_rng(k).integers(
            0, w.token_vocab, w.num_tokens).astype(np.int32)))
        hidden.copy_(torch.randn(hidden.shape, generator=torch.Generator().manual_seed(k))
                     .to(torch.bfloat16))
        g.replay()
        torch.cuda.synchronize()
        want = layer.forward(ids, qsl, hidden).clone()
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert torch.equal(out.view(torch.int16), want.view(torch.int16)), f"replay {k}"
    if owner is not None:
        owner.close()


@pytest.mark.parametrize("prefetch", [True, False])
@pytest.mark.parametrize("on_host", [False, True])
@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_chain_matches_oracle(prefetch, on_host, dtype):
    """PLEChain over four layers against the oracle's layer_forward for each
    layer (its own multipliers, table, weights, hidden state and conv state;
    the n-gram context shared by all layers): ids of the carried context bit
    for bit, every layer's y and conv-state carry-over within the chain
    tolerance; next layers' gathers prefetched on a side stream or run in
    line, tables in HBM or in pinned host memory (table-order gather)."""
    from hashed_gram_embedding_gb300 import PLEChain, _lib
    L = 4
    tol = 1e-2 if dtype == "bf16" else 3e-2
    w = wl.scaled(wl.WORKLOADS["tiny"], num_layers=L, decode=True, table_dtype=dtype)
    layers, hiddens, states, owners, refs = [], [], [], [], []
    host = None
    for i in range(L):
        _, host_i, dense, table, row_scale = tiny_case(w, seed_step=i)
        host = host or host_i
        d = {k: v.cuda() for k, v in dense.items()}
        if on_host and dtype == "bf16":
            owner = _lib.HostTable(table.shape[0], table.shape[1], torch.bfloat16)
            owner.tensor.copy_(table)
            owners.append(owner)
            tab = owner.tensor
        elif on_host:
            tab = table.pin_memory()
        else:
            tab = table.cuda()
        rs = None if row_scale is None else row_scale.cuda()
        layers.append(PLELayer(tab, rs, host["multipliers"][i], host["V"], host["O"],
                               w.eos_token_id, w.heads_per_ngram, d["w_kv"], d["gamma_h"],
                               d["gamma_k"], d["conv_w"], w.dilation))
        hiddens.append(d["hidden"])
        states.append(d["conv_state"])
        refs.append(oracle.layer_forward(
            host["input_ids"], host["query_start_loc"], host["ngram_context"],
            host["multipliers"][i], host["V"], host["O"], w.eos_token_id, w.heads_per_ngram,
            bits(table) if row_scale is None else table.numpy(),
            None if row_scale is None else row_scale.numpy(), bits(dense["hidden"]),
            bits(dense["w_kv"]), bits(dense["gamma_h"]), bits(dense["gamma_k"]), 1e-6,
            bits(dense["conv_w"]), w.dilation, bits(dense["conv_state"])))
    T, C = w.num_tokens, w.hidden
    ids = torch.from_numpy(host["input_ids"]).cuda()
    qsl = torch.from_numpy(host["query_start_loc"]).cuda()
    ctx = torch.from_numpy(host["ngram_context"]).cuda()
    outs = [torch.empty((T, C), dtype=torch.bfloat16, device="cuda") for _ in range(L)]
    st_out = [torch.empty_like(s) for s in states]
    ctx_out = torch.empty_like(ctx)
    err = dev_err_word()
    PLEChain(layers, prefetch=prefetch, prefetch_ctas=76).forward(
        ids, qsl, hiddens, outs, ngram_context=ctx, ngram_context_out=ctx_out,
        conv_states=states, conv_states_out=st_out, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(ctx_out.cpu().numpy(), np.asarray(refs[0]["ngram_context_out"]))
    for i in range(L):
        assert_close(bits(outs[i]), refs[i]["y"], rtol=tol, atol_frac=max(tol, CHAIN_ATOL_FRAC),
                     what=f"layer {i} y")
        assert_close(bits(st_out[i]), refs[i]["conv_state_out"], rtol=tol,
                     atol_frac=max(tol, CHAIN_ATOL_FRAC), what=f"layer {i} conv state")
    for o in owners:
        o.close()


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_host_table_layer_every_token(dtype):
    """PLELayer.forward over a table in pinned host memory (read over the
    host link in table order) against the oracle's layer_forward: ids and
    gathered rows bit for bit, y of every token in tolerance."""
    from hashed_gram_embedding_gb300 import _lib
    w = wl.scaled(wl.WORKLOADS["tiny"], table_dtype=dtype)
    w, host, dense, table, row_scale = tiny_case(w)
    d = {k: v.cuda() for k, v in dense.items()}
    owner = None
    if dtype == "bf16":
        owner = _lib.HostTable(table.shape[0], table.shape[1], torch.bfloat16)
        owner.tensor.copy_(table)
        tab = owner.tensor
    else:
        tab = table.pin_memory()
    layer = build_layer(w, host, d, tab, None if row_scale is None else row_scale.cuda())
    err = dev_err_word()
    y = layer.forward(torch.from_numpy(host["input_ids"]).cuda(),
                      torch.from_numpy(host["query_start_loc"]).cuda(), d["hidden"], dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = oracle.layer_forward(host["input_ids"], host["query_start_loc"], None,
                               host["multipliers"][0], host["V"], host["O"], w.eos_token_id,
                               w.heads_per_ngram,
                               bits(table) if row_scale is None else table.numpy(),
                               None if row_scale is None else row_scale.numpy(),
                               bits(dense["hidden"]), bits(dense["w_kv"]), bits(dense["gamma_h"]),
                               bits(dense["gamma_k"]), 1e-6, bits(dense["conv_w"]), w.dilation)
    b = layer.buffers(w.num_tokens, y.device)
    assert np.array_equal(b["ids"].cpu().numpy(), ref["ids"])
    assert np.array_equal(bits(b["emb"]), ref["emb"])
    tol = 1e-2 if dtype == "bf16" else 3e-2
    assert_close(bits(y), ref["y"], rtol=tol, atol_frac=max(tol, CHAIN_ATOL_FRAC), what="y")
    if owner is not None:
        owner.close()


def test_uva32g_layer_sampled():
    """The host-table workload at full size (a 32 GiB bf16 table in pinned
    host memory, 8192 tokens) through PLELayer.forward: every id bit for
    bit, every gathered row of the sampled tokens bit for bit, and y against
    the oracle on >= 2048 sampled tokens with their conv history."""
    w = wl.WORKLOADS["uva32g"]
    host = wl.host_inputs(w)
    table, _ = wl.make_table(torch, w, "cuda")
    assert not table.is_cuda
    dense = wl.dense_inputs(torch, w, "cuda", random_gamma=True)
    layer = build_layer(w, host, dense, table, None)
    qsl = host["query_start_loc"]
    err = dev_err_word()
    y = layer.forward(torch.from_numpy(host["input_ids"]).cuda(), torch.from_numpy(qsl).cuda(),
                      dense["hidden"], dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ids, _ = oracle.ngram_ids(host["input_ids"], qsl, None, host["multipliers"][0], host["V"],
                              host["O"], w.eos_token_id, w.heads_per_ngram)
    ids = np.asarray(ids, dtype=np.int64).reshape(w.num_tokens, -1)
    b = layer.buffers(w.num_tokens, y.device)
    assert np.array_equal(b["ids"].cpu().numpy(), ids)
    blocks = sampled_blocks(qsl, w.num_tokens, (w.conv_k - 1) * w.dilation,
                            np.random.default_rng(4))
    rows = np.unique(np.concatenate([np.arange(lo, e) for lo, _, e in blocks]))
    want = oracle.lookup_bf16(ids[rows], bits(table))
    assert np.array_equal(bits(b["emb"])[rows], want)
    n = check_chain_sampled(w, host, dense, lambda u: bits(table[torch.from_numpy(u)]), None, y,
                            ids, blocks)
    assert n >= 2048
    del layer, b, table
    torch.cuda.empty_cache()
