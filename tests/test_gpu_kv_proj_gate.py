"""GPU parity of the fused projection + gate reductions (ple_kv_proj_gate) and
of the conv pass on given gate scalars (ple_gated_conv).

Checked against the oracle (kv_proj, gate, gate_conv in float64) and against
the unfused kernels: the value half of kv equals ple_kv_proj's bit for bit
(same tensor-core arithmetic), the key half is left untouched, the gate
scalars agree with ple_gate run on ple_kv_proj's kv (same bf16 k; only the
float32 summation order differs), and ple_gated_conv on ple_gate's scalars
equals ple_gate_conv bit for bit. Shapes cover ragged row counts (a partial
32-row group, M = 1), several key-tile counts, both CTA-pair kernels with 4
and 8 epilogue warps and both tile orders, and the 8k-prefill shape in the
launch configuration the benchmark times."""

import numpy as np
import pytest
import torch

from oracle import gate as oracle_gate
from oracle import gate_conv as oracle_gate_conv
from oracle import kv_proj as oracle_kv_proj

from _helpers import CHAIN_ATOL_FRAC, assert_close, bits, dev_err_word
from hashed_gram_embedding_gb300 import _lib
from hashed_gram_embedding_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def rand_bf16(shape, std, seed, mean=0.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * std + mean).to(torch.bfloat16)


def inputs(M, E, C, seed):
    emb = rand_bf16((M, E), 0.5, seed)
    w = rand_bf16((2 * C, E), 0.05, seed + 1)
    h = rand_bf16((M, C), 1.0, seed + 2)
    gh = rand_bf16((C,), 0.1, seed + 3, mean=1.0)
    gk = rand_bf16((C,), 0.1, seed + 4, mean=1.0)
    return emb, w, h, gh, gk


def workspace(M, C):
    n = _lib.ple_kv_proj_gate_workspace(M, C)
    assert n > 0
    return torch.zeros((n,), dtype=torch.uint8, device="cuda")  # zero-filled before first use


def counters_zero(ws):
    # the arrival counters (the buffer's last bytes) are zero after every
    # completed call
    n = ws.numel()
    tail = ((n // 16 + 31) // 32) * 4
    return bool(torch.all(ws[n - tail:] == 0))


def run_fused(emb, w, h, gh, gk, eps=1e-6, ws=None):
    M, C = h.shape
    kv = torch.full((M, 2 * C), float("nan"), dtype=torch.bfloat16, device="cuda")
    g = torch.full((M,), float("nan"), dtype=torch.float32, device="cuda")
    err = dev_err_word()
    _lib.ple_kv_proj_gate(emb, w, h, gh, gk, kv, g, ws if ws is not None else workspace(M, C),
                          eps=eps, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return kv, g


CASES = [(512, 512, 1024), (1, 64, 256), (129, 200, 256), (300, 2048, 4096), (1000, 128, 512),
         (257, 72, 768), (33, 64, 512)]


@pytest.mark.parametrize("epi,order", [("4", "natural"), ("8", "natural"), ("4", "keyfirst"),
                                       ("8", "keyfirst")])
@pytest.mark.parametrize("mode", ["pair", "pair-nosplit"])
@pytest.mark.parametrize("M,E,C", CASES)
def test_kv_proj_gate_matches_oracle_and_unfused(M, E, C, mode, epi, order, monkeypatch):
    """The CTA-pair kernel; "pair" splits the last round's tiles into
    128-column halves where that shortens it (every case here but 300 x 4096
    and 1000 x 512), "pair-nosplit" never does; epi: 4 or 8 epilogue warps;
    order: row blocks in turn, or every key tile before the value tiles. The
    gate scalars and v are the same bits with every epilogue width and order."""
    monkeypatch.setenv("PLE_KVPROJ_MODE", mode.split("-")[0])
    monkeypatch.setenv("PLE_KVPROJ_SPLIT", "0" if mode.endswith("nosplit") else "1")
    monkeypatch.setenv("PLE_KVPROJ_EPI", "8" if epi == "4" else "4")
    monkeypatch.setenv("PLE_KVPROJ_ORDER", "keyfirst" if order == "natural" else "natural")
    emb, w, h, gh, gk = (t.cuda() for t in inputs(M, E, C, M + C))
    kv_other, g_other = run_fused(emb, w, h, gh, gk)
    monkeypatch.setenv("PLE_KVPROJ_EPI", epi)
    monkeypatch.setenv("PLE_KVPROJ_ORDER", order)
    kv, g = run_fused(emb, w, h, gh, gk)
    assert torch.equal(g.view(torch.int32), g_other.view(torch.int32))
    assert torch.equal(kv[:, C:].view(torch.int16), kv_other[:, C:].view(torch.int16))
    # value half: the unfused projection's bits; key half: never written
    kv_ref = torch.empty_like(kv)
    _lib.ple_kv_proj(emb, w, kv_ref)
    u = torch.empty((M, C), dtype=torch.bfloat16, device="cuda")
    g_ref = torch.empty((M,), dtype=torch.float32, device="cuda")
    _lib.ple_gate(h, kv_ref, gh, gk, u, eps=1e-6, gate_out=g_ref)
    torch.cuda.synchronize()
    assert torch.equal(kv[:, C:].view(torch.int16), kv_ref[:, C:].view(torch.int16))
    assert torch.isnan(kv[:, :C].float()).all()
    assert float((g - g_ref).abs().max()) < 1e-5
    # the gate scalars do not depend on how the tiles were split
    monkeypatch.setenv("PLE_KVPROJ_SPLIT", "0")
    _, g_nosplit = run_fused(emb, w, h, gh, gk)
    assert torch.equal(g.view(torch.int32), g_nosplit.view(torch.int32))
    # against the oracle: kv in float64, the gate on the oracle's kv
    ref_kv = oracle_kv_proj(bits(emb), bits(w))
    assert_close(bits(kv[:, C:]), ref_kv[:, C:], what=f"v {M}x{E}x{2 * C}")
    _, ref_g = oracle_gate(bits(h), ref_kv, bits(gh), bits(gk), 1e-6)
    gg = g.cpu().numpy().astype(np.float64)
    assert np.all((gg > 0) & (gg < 1))
    assert np.max(np.abs(gg - ref_g)) < 5e-4


@pytest.mark.parametrize("vn", ["192", "128"])
@pytest.mark.parametrize("M,E,C", CASES + [(1024, 256, 4096), (2000, 64, 1024)])
def test_kv_proj_gate_strip_schedule_same_bits(M, E, C, vn, monkeypatch):
    """The strip schedule (value half in vn-column strips, the narrower
    remainder strips first, then the key tiles) gives the default schedule's
    v and gate scalars bit for bit, and the oracle's within tolerance."""
    monkeypatch.setenv("PLE_KVPROJ_ORDER", "keyfirst")
    monkeypatch.setenv("PLE_KVPROJ_VN", "0")
    emb, w, h, gh, gk = (t.cuda() for t in inputs(M, E, C, M + 3 * C))
    kv_ref, g_ref = run_fused(emb, w, h, gh, gk)
    monkeypatch.setenv("PLE_KVPROJ_VN", vn)
    kv, g = run_fused(emb, w, h, gh, gk)
    assert torch.equal(g.view(torch.int32), g_ref.view(torch.int32))
    assert torch.equal(kv[:, C:].view(torch.int16), kv_ref[:, C:].view(torch.int16))
    assert torch.isnan(kv[:, :C].float()).all()
    ref_kv = oracle_kv_proj(bits(emb), bits(w))
    assert_close(bits(kv[:, C:]), ref_kv[:, C:], what=f"v strips {vn} {M}x{E}x{2 * C}")


def test_kv_proj_gate_is_deterministic_with_a_reused_workspace():
    M, E, C = 700, 256, 512
    emb, w, h, gh, gk = (t.cuda() for t in inputs(M, E, C, 5))
    ws = workspace(M, C)
    kv1, g1 = run_fused(emb, w, h, gh, gk, ws=ws)
    assert counters_zero(ws)
    kv2, g2 = run_fused(emb, w, h, gh, gk, ws=ws)
    assert counters_zero(ws)
    assert torch.equal(g1.view(torch.int32), g2.view(torch.int32))
    assert torch.equal(kv1[:, C:].view(torch.int16), kv2[:, C:].view(torch.int16))


def test_one_workspace_serves_varying_token_counts_and_hidden_sizes():
    """Serving reuses one workspace sized for the largest step: calls with
    other token counts and hidden sizes find their counters zeroed and get
    the unfused kernels' gate scalars."""
    ws = workspace(1000, 1024)
    for k, (M, C) in enumerate([(1000, 1024), (100, 1024), (1, 256), (513, 512), (1000, 1024),
                                (33, 768), (1000, 256)]):
        emb, w, h, gh, gk = (t.cuda() for t in inputs(M, 128, C, 70 + k))
        kv, g = run_fused(emb, w, h, gh, gk, ws=ws)
        assert counters_zero(ws)
        kv_ref = torch.empty_like(kv)
        _lib.ple_kv_proj(emb, w, kv_ref)
        u = torch.empty((M, C), dtype=torch.bfloat16, device="cuda")
        g_ref = torch.empty((M,), dtype=torch.float32, device="cuda")
        _lib.ple_gate(h, kv_ref, gh, gk, u, gate_out=g_ref)
        torch.cuda.synchronize()
        assert float((g - g_ref).abs().max()) < 1e-5, (M, C)


def test_kv_proj_gate_degenerate_gate_inputs():
    # h = 0 for one token: the dot is 0, so g = sigmoid(0) = 1/2 exactly;
    # gamma_k = 0: every score is 0
    M, E, C = 70, 64, 256
    emb, w, h, gh, gk = inputs(M, E, C, 9)
    h[3] = 0
    kv, g = run_fused(emb.cuda(), w.cuda(), h.cuda(), gh.cuda(), gk.cuda())
    assert float(g[3]) == 0.5
    _, g0 = run_fused(emb.cuda(), w.cuda(), h.cuda(), gh.cuda(), torch.zeros_like(gk).cuda())
    assert torch.all(g0 == 0.5)


def qsl_of(lengths):
    return np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)


@pytest.mark.parametrize("lengths,C", [([64, 100, 150, 198], 1024), ([7, 0, 30, 2, 0, 61], 256),
                                       ([1] * 40, 512), ([300], 4096)])
def test_fused_chain_matches_oracle_gate_conv(lengths, C):
    q = qsl_of(lengths)
    T, E, R = int(q[-1]), 256, len(lengths)
    emb, w, h, gh, gk = inputs(T, E, C, 40)
    cw = rand_bf16((C, 4), 0.5, 45)
    state = rand_bf16((R, 9, C), 0.01, 46)
    dq = torch.from_numpy(q).cuda()
    kv, g = run_fused(emb.cuda(), w.cuda(), h.cuda(), gh.cuda(), gk.cuda())
    y = torch.empty((T, C), dtype=torch.bfloat16, device="cuda")
    st = torch.empty((R, 9, C), dtype=torch.bfloat16, device="cuda")
    err = dev_err_word()
    _lib.ple_gated_conv(kv, g, dq, cw.cuda(), 3, y, conv_state=state.cuda(), conv_state_out=st,
                        dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref_kv = oracle_kv_proj(bits(emb), bits(w))
    ref_y, ref_st, _ = oracle_gate_conv(bits(h), ref_kv, bits(gh), bits(gk), 1e-6, q, bits(cw),
                                        3, bits(state))
    assert_close(bits(y), ref_y, atol_frac=CHAIN_ATOL_FRAC, what="fused chain y")
    assert_close(bits(st), ref_st, atol_frac=CHAIN_ATOL_FRAC, what="fused chain state")


@pytest.mark.parametrize("lengths,C", [([64, 100, 150, 198], 1024), ([1] * 70 + [3, 0, 9], 264)])
def test_gated_conv_equals_gate_conv(lengths, C):
    """ple_gated_conv on ple_gate_conv's own gate scalars gives its y and
    state bit for bit (any C, not only multiples of 256)."""
    q = qsl_of(lengths)
    T, R = int(q[-1]), len(lengths)
    h = rand_bf16((T, C), 1.0, 60).cuda()
    kv = rand_bf16((T, 2 * C), 0.02, 61).cuda()
    gh = rand_bf16((C,), 0.1, 62, mean=1.0).cuda()
    gk = rand_bf16((C,), 0.1, 63, mean=1.0).cuda()
    cw = rand_bf16((C, 4), 0.5, 64).cuda()
    state = rand_bf16((R, 9, C), 0.01, 65).cuda()
    dq = torch.from_numpy(q).cuda()
    y1, y2 = (torch.empty((T, C), dtype=torch.bfloat16, device="cuda") for _ in range(2))
    s1, s2 = (torch.empty((R, 9, C), dtype=torch.bfloat16, device="cuda") for _ in range(2))
    g = torch.empty((T,), dtype=torch.float32, device="cuda")
    _lib.ple_gate_conv(h, kv, gh, gk, dq, cw, 3, y1, conv_state=state, conv_state_out=s1,
                       gate_out=g)
    _lib.ple_gated_conv(kv, g, dq, cw, 3, y2, conv_state=state, conv_state_out=s2)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2) and torch.equal(s1, s2)


def test_kv_proj_gate_prefill_8k():
    """The 8k-prefill shape (8192 tokens, 2048 -> 2 x 4096) in the launch
    configuration the benchmark times: all rows against the unfused kernels
    and cuBLAS, 2060 sampled rows (tile edges included) against the oracle."""
    w_ = wl.WORKLOADS["prefill8k"]
    M, E, C = w_.num_tokens, w_.emb_dim, w_.hidden
    gen = torch.Generator(device="cuda").manual_seed(21)
    emb = (torch.randn((M, E), generator=gen, device="cuda") * 0.02).to(torch.bfloat16)
    w = (torch.randn((2 * C, E), generator=gen, device="cuda") * 0.02).to(torch.bfloat16)
    h = torch.randn((M, C), generator=gen, device="cuda").to(torch.bfloat16)
    gh = (torch.randn((C,), generator=gen, device="cuda") * 0.1 + 1).to(torch.bfloat16)
    gk = (torch.randn((C,), generator=gen, device="cuda") * 0.1 + 1).to(torch.bfloat16)
    kv, g = run_fused(emb, w, h, gh, gk)
    kv_ref = torch.empty_like(kv)
    _lib.ple_kv_proj(emb, w, kv_ref)
    u = torch.empty((M, C), dtype=torch.bfloat16, device="cuda")
    g_ref = torch.empty((M,), dtype=torch.float32, device="cuda")
    _lib.ple_gate(h, kv_ref, gh, gk, u, gate_out=g_ref)
    torch.cuda.synchronize()
    assert torch.equal(kv[:, C:].view(torch.int16), kv_ref[:, C:].view(torch.int16))
    assert float((g - g_ref).abs().max()) < 1e-5
    lib_v = (emb.float() @ w[C:].float().T).to(torch.bfloat16)
    assert_close(bits(kv[:, C:]), bits(lib_v), what="v vs cuBLAS")
    edges = [0, 1, 31, 32, 127, 128, 255, 256, 4095, 4096, 8190, 8191]
    rest = np.setdiff1d(np.arange(M), edges)
    rows = np.concatenate([edges, np.random.default_rng(2).choice(rest, 2048, replace=False)])
    sel = torch.from_numpy(rows).cuda()
    ref_kv = oracle_kv_proj(bits(emb[sel]), bits(w))
    assert_close(bits(kv[sel][:, C:]), ref_kv[:, C:], what="v, sampled rows")
    _, ref_g = oracle_gate(bits(h[sel]), ref_kv, bits(gh), bits(gk), 1e-6)
    assert np.max(np.abs(g[sel].cpu().numpy() - ref_g)) < 5e-4


def test_kv_proj_gate_largest_hidden():
    """hidden = 16384 (ple_gate's largest): 128 partial-sum blocks per row."""
    M, E, C = 96, 64, 16384
    emb, w, h, gh, gk = (t.cuda() for t in inputs(M, E, C, 17))
    kv, g = run_fused(emb, w, h, gh, gk)
    kv_ref = torch.empty_like(kv)
    _lib.ple_kv_proj(emb, w, kv_ref)
    u = torch.empty((M, C), dtype=torch.bfloat16, device="cuda")
    g_ref = torch.empty((M,), dtype=torch.float32, device="cuda")
    _lib.ple_gate(h, kv_ref, gh, gk, u, gate_out=g_ref)
    torch.cuda.synchronize()
    assert torch.equal(kv[:, C:].view(torch.int16), kv_ref[:, C:].view(torch.int16))
    assert float((g - g_ref).abs().max()) < 1e-5
    _, ref_g = oracle_gate(bits(h), oracle_kv_proj(bits(emb), bits(w)), bits(gh), bits(gk), 1e-6)
    assert np.max(np.abs(g.cpu().numpy() - ref_g)) < 5e-4
