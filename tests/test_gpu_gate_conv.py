"""GPU parity of ple_gate, ple_conv and ple_gate_conv against the oracle:
ragged requests with empty requests and padding tokens, zero / given
history, carry-over state (ping-pong over two steps), kernel sizes 1..8 and
dilations up to a 63-token halo, the tiny and the decode (256 x 4, hidden
4096) workloads, the 8k prefill at full size (sampled tokens), and the fused
kernel against the two separate ones."""

import numpy as np
import pytest
import torch

from oracle import gate as oracle_gate, conv as oracle_conv, gate_conv as oracle_gate_conv
from hashed_gram_embedding_gb300 import _lib
from hashed_gram_embedding_gb300 import workloads as wl

from _helpers import assert_close, bits, from_bits, dev_err_word

pytestmark = pytest.mark.gpu


def rand_bf16(shape, std, seed, mean=0.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * std + mean).to(torch.bfloat16)


def qsl_of(lengths):
    return np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)


def dev_qsl(q):
    return torch.from_numpy(np.asarray(q, dtype=np.int32)).cuda()


@pytest.mark.parametrize("T,C", [(1, 8), (37, 64), (65, 520), (512, 1024), (300, 4096),
                                 (40, 8192), (17, 16384)])
def test_gate_matches_oracle(T, C):
    h = rand_bf16((T, C), 1.0, 1)
    kv = rand_bf16((T, 2 * C), 0.02, 2)
    gh = rand_bf16((C,), 0.1, 3, mean=1.0)
    gk = rand_bf16((C,), 0.1, 4, mean=1.0)
    u = torch.empty((T, C), dtype=torch.bfloat16, device="cuda")
    g = torch.empty((T,), dtype=torch.float32, device="cuda")
    _lib.ple_gate(h.cuda(), kv.cuda(), gh.cuda(), gk.cuda(), u, eps=1e-6, gate_out=g)
    torch.cuda.synchronize()
    ref_u, ref_g = oracle_gate(bits(h), bits(kv), bits(gh), bits(gk), 1e-6)
    assert np.max(np.abs(g.cpu().numpy() - ref_g)) < 1e-4
    assert np.all((g.cpu().numpy() > 0) & (g.cpu().numpy() < 1))
    assert_close(bits(u), ref_u, what="gate u")


CONV_CASES = [
    # lengths, C, K, dilation
    ([64, 100, 150, 198], 64, 4, 3),
    ([5, 0, 17, 1, 0, 40], 32, 4, 3),
    ([3, 9, 1], 16, 1, 1),
    ([70, 2, 33], 24, 8, 9),
    ([10, 20], 40, 2, 5),
    ([1] * 50, 8, 4, 3),
    # decode-like: every token's taps reach into the carry-over state; C not a
    # multiple of the 256-channel slice (idle lanes in the last slice)
    ([1] * 300, 264, 4, 3),
    # hundreds of empty requests around a few non-empty ones
    ([0] * 40 + [5] + [0] * 300 + [7, 0, 0, 3], 48, 3, 2),
    # one long request over many token tiles
    ([2000], 72, 4, 3),
    # several 256-channel slices
    ([64, 100, 150, 198], 512, 4, 3),
    # the largest window (W = 63 rows before each tile)
    ([70, 2, 33], 256, 8, 9),
    # a ragged last slice (C % 256 = 64) and empty requests
    ([5, 0, 17, 1, 0, 40], 320, 3, 2),
]


# conv pass variants: the one-shot tiled kernel (default tile, the 112-token
# tile of large steps, an odd 5-token tile; the window staged as the default
# chooses, by per-lane loads, and by one TMA copy wherever that fits the
# source tensor) and the streaming kernel (default launch shape, one token
# range per slice, seven ranges)
CONV_MODES = {"tile": {}, "tile-112": {"PLE_CONV_TILE": "112"}, "tile-5": {"PLE_CONV_TILE": "5"},
              "tile-noTMA": {"PLE_CONV_TMA": "0"}, "tile-TMA": {"PLE_CONV_TMA": "1"},
              "stream": {"PLE_CONV_MODE": "stream"},
              "stream-1range": {"PLE_CONV_MODE": "stream", "PLE_CONV_RANGES": "1"},
              "stream-7ranges": {"PLE_CONV_MODE": "stream", "PLE_CONV_RANGES": "7"}}


@pytest.fixture(params=list(CONV_MODES))
def conv_mode(request, monkeypatch):
    for k, v in CONV_MODES[request.param].items():
        monkeypatch.setenv(k, v)
    return request.param


@pytest.mark.parametrize("with_state", [False, True])
@pytest.mark.parametrize("case", CONV_CASES, ids=lambda c: f"{len(c[0])}req-C{c[1]}-K{c[2]}-d{c[3]}")
def test_conv_matches_oracle(case, with_state, conv_mode):
    lengths, C, K, d = case
    q = qsl_of(lengths)
    T = int(q[-1])
    W = (K - 1) * d
    x = rand_bf16((T, C), 1.0, T + C)
    w = rand_bf16((C, K), 0.5, K)
    state = rand_bf16((len(lengths), W, C), 0.3, 9) if with_state else None
    y = torch.empty((T, C), dtype=torch.bfloat16, device="cuda")
    st_out = torch.full((len(lengths), W, C), 3.0, dtype=torch.bfloat16, device="cuda")
    err = dev_err_word()
    _lib.ple_conv(x.cuda(), dev_qsl(q), w.cuda(), d, y,
                  conv_state=None if state is None else state.cuda(), conv_state_out=st_out,
                  dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref_y, ref_st = oracle_conv(bits(x), q, bits(w), d, None if state is None else bits(state))
    assert_close(bits(y), ref_y, what="conv y")
    assert np.array_equal(bits(st_out), ref_st)


def test_conv_padding_tokens_join_last_request():
    q = np.array([0, 4, 9], dtype=np.int32)
    T, C, K, d = 14, 16, 4, 3
    x = rand_bf16((T, C), 1.0, 5)
    w = rand_bf16((C, K), 0.5, 6)
    y = torch.empty((T, C), dtype=torch.bfloat16, device="cuda")
    st = torch.empty((2, 9, C), dtype=torch.bfloat16, device="cuda")
    _lib.ple_conv(x.cuda(), dev_qsl(q), w.cuda(), d, y, conv_state_out=st)
    torch.cuda.synchronize()
    ref_y, ref_st = oracle_conv(bits(x), q, bits(w), d, None, num_tokens=T)
    assert_close(bits(y), ref_y, what="conv y tail")
    assert np.array_equal(bits(st), ref_st)


@pytest.mark.parametrize("tile", [None, "112", "37", "5"])
@pytest.mark.parametrize("gated", [False, True])
@pytest.mark.parametrize("case", CONV_CASES, ids=lambda c: f"{len(c[0])}req-C{c[1]}-K{c[2]}-d{c[3]}")
def test_tiled_and_streaming_conv_same_bits(case, gated, tile, monkeypatch):
    """The tiled kernel (taps and window as bf16 pairs, mixed-precision FMA;
    window staged by TMA where it fits, and by per-lane loads) and the
    streaming kernel (float32 ring, two-wide float32 FMA) take the same taps
    in the same order with one rounding per tap: y and the carry-over state
    agree bit for bit."""
    lengths, C, K, d = case
    q = qsl_of(lengths)
    T, R, W = int(q[-1]), len(lengths), (K - 1) * d
    src = rand_bf16((T, 2 * C if gated else C), 1.0, T + 7 * C)
    w = rand_bf16((C, K), 0.5, K + 1).cuda()
    state = rand_bf16((R, W, C), 0.3, 11).cuda()
    g = torch.rand((T,), generator=torch.Generator().manual_seed(5)).cuda() if gated else None
    outs = []
    tile_env = {} if tile is None else {"PLE_CONV_TILE": tile}
    for env in (tile_env, {**tile_env, "PLE_CONV_TMA": "0"}, {**tile_env, "PLE_CONV_TMA": "1"},
                {"PLE_CONV_MODE": "stream"}):
        monkeypatch.delenv("PLE_CONV_MODE", raising=False)
        monkeypatch.delenv("PLE_CONV_TILE", raising=False)
        for k, v in env.items():
            monkeypatch.setenv(k, v)
        y = torch.full((T, C), float("nan"), dtype=torch.bfloat16, device="cuda")
        st = torch.full((R, W, C), float("nan"), dtype=torch.bfloat16, device="cuda")
        if gated:
            _lib.ple_gated_conv(src.cuda(), g, dev_qsl(q), w, d, y, conv_state=state,
                                conv_state_out=st)
        else:
            _lib.ple_conv(src.cuda(), dev_qsl(q), w, d, y, conv_state=state, conv_state_out=st)
        torch.cuda.synchronize()
        outs.append((y.view(torch.int16).cpu(), st.view(torch.int16).cpu()))
    for y, st in outs[1:]:
        assert torch.equal(outs[0][0], y)
        assert torch.equal(outs[0][1], st)


def _gate_conv_inputs(lengths, C, seed):
    q = qsl_of(lengths)
    T = int(q[-1])
    h = rand_bf16((T, C), 1.0, seed)
    kv = rand_bf16((T, 2 * C), 0.02, seed + 1)
    gh = rand_bf16((C,), 0.1, seed + 2, mean=1.0)
    gk = rand_bf16((C,), 0.1, seed + 3, mean=1.0)
    w = rand_bf16((C, 4), 0.5, seed + 4)
    return q, T, h, kv, gh, gk, w


@pytest.mark.parametrize("lengths,C", [([64, 100, 150, 198], 1024), ([7, 0, 30, 2, 0, 61], 256),
                                       ([1] * 40, 64), ([300], 4096),
                                       ([1] * 70 + [3, 0, 9], 264)])
def test_gate_conv_matches_oracle_and_separate_kernels(lengths, C, conv_mode):
    q, T, h, kv, gh, gk, w = _gate_conv_inputs(lengths, C, 20)
    R = len(lengths)
    state = rand_bf16((R, 9, C), 0.01, 30)
    args = [t.cuda() for t in (h, kv, gh, gk)]
    y = torch.empty((T, C), dtype=torch.bfloat16, device="cuda")
    g = torch.empty((T,), dtype=torch.float32, device="cuda")
    st_out = torch.empty((R, 9, C), dtype=torch.bfloat16, device="cuda")
    err = dev_err_word()
    _lib.ple_gate_conv(*args, dev_qsl(q), w.cuda(), 3, y, eps=1e-6, conv_state=state.cuda(),
                       conv_state_out=st_out, gate_out=g, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref_y, ref_st, ref_g = oracle_gate_conv(bits(h), bits(kv), bits(gh), bits(gk), 1e-6, q,
                                            bits(w), 3, bits(state))
    assert np.max(np.abs(g.cpu().numpy() - ref_g)) < 1e-4
    assert_close(bits(y), ref_y, what="gate_conv y")
    assert_close(bits(st_out), ref_st, what="gate_conv state")
    # the fused kernel equals gate followed by conv, bit for bit
    u = torch.empty((T, C), dtype=torch.bfloat16, device="cuda")
    _lib.ple_gate(*args, u, eps=1e-6)
    y2 = torch.empty_like(y)
    st2 = torch.empty_like(st_out)
    _lib.ple_conv(u, dev_qsl(q), w.cuda(), 3, y2, conv_state=state.cuda(), conv_state_out=st2)
    torch.cuda.synchronize()
    assert torch.equal(y, y2) and torch.equal(st_out, st2)


def test_gate_conv_decode_two_steps_ping_pong(conv_mode):
    w_ = wl.WORKLOADS["decode256x4"]
    R, C = w_.num_reqs, w_.hidden
    lengths = [4] * R
    q = qsl_of(lengths)
    dense0 = wl.dense_inputs(torch, w_, "cpu", step=0, random_gamma=True)
    state0 = dense0["conv_state"]
    states = [state0.cuda(), torch.empty_like(state0, device="cuda")]
    ref_state = bits(state0)
    for step in range(2):
        _, T, h, kv, gh, gk, _ = _gate_conv_inputs(lengths, C, 40 + step)
        y = torch.empty((T, C), dtype=torch.bfloat16, device="cuda")
        _lib.ple_gate_conv(h.cuda(), kv.cuda(), gh.cuda(), gk.cuda(), dev_qsl(q),
                           dense0["conv_w"].cuda(), 3, y, conv_state=states[step % 2],
                           conv_state_out=states[(step + 1) % 2])
        torch.cuda.synchronize()
        ref_y, ref_state, _ = oracle_gate_conv(bits(h), bits(kv), bits(gh), bits(gk), 1e-6, q,
                                               bits(dense0["conv_w"]), 3, ref_state)
        assert_close(bits(y), ref_y, what=f"decode y step {step}")
        assert_close(bits(states[(step + 1) % 2]), ref_state, what=f"decode state step {step}")


def test_zero_tokens_copy_state_through():
    C = 64
    state = rand_bf16((3, 9, C), 1.0, 50).cuda()
    out_state = torch.zeros_like(state)
    y = torch.empty((0, C), dtype=torch.bfloat16, device="cuda")
    x = torch.empty((0, C), dtype=torch.bfloat16, device="cuda")
    w = rand_bf16((C, 4), 0.5, 51).cuda()
    _lib.ple_conv(x, dev_qsl([0, 0, 0, 0]), w, 3, y, conv_state=state, conv_state_out=out_state)
    torch.cuda.synchronize()
    assert torch.equal(state, out_state)


def test_gate_conv_prefill_8k_sampled(conv_mode):
    w_ = wl.WORKLOADS["prefill8k"]
    host = wl.host_inputs(w_)
    q = host["query_start_loc"]
    T, C = w_.num_tokens, w_.hidden
    g = torch.Generator(device="cuda").manual_seed(3)
    h = torch.randn((T, C), generator=g, device="cuda").to(torch.bfloat16)
    kv = (torch.randn((T, 2 * C), generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    gh = (torch.randn((C,), generator=g, device="cuda") * 0.1 + 1).to(torch.bfloat16)
    gk = (torch.randn((C,), generator=g, device="cuda") * 0.1 + 1).to(torch.bfloat16)
    cw = (torch.randn((C, 4), generator=g, device="cuda") * 0.5).to(torch.bfloat16)
    y = torch.empty((T, C), dtype=torch.bfloat16, device="cuda")
    st = torch.empty((len(q) - 1, 9, C), dtype=torch.bfloat16, device="cuda")
    _lib.ple_gate_conv(h, kv, gh, gk, dev_qsl(q), cw, 3, y, conv_state_out=st)
    torch.cuda.synchronize()
    rng = np.random.default_rng(1)
    starts = q[:-1]
    sample = np.unique(np.concatenate([s + np.arange(10) for s in starts] +
                                      [rng.integers(0, T, 100), [T - 1]]))
    req_of = np.searchsorted(q, sample, side="right") - 1
    hb, kvb, ghb, gkb, cwb, yb = bits(h), bits(kv), bits(gh), bits(gk), bits(cw), bits(y)
    for t, r in zip(sample, req_of):
        lo = max(int(q[r]), int(t) - 9)  # the token's window inside its request
        win = slice(lo, int(t) + 1)
        ref_y, _, _ = oracle_gate_conv(hb[win], kvb[win], ghb, gkb, 1e-6,
                                       [0, int(t) + 1 - lo], cwb, 3)
        assert_close(yb[t:t + 1], ref_y[-1:], what=f"token {t}")
