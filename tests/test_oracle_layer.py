"""Pins of the kv_proj, gate and short-conv oracles.

Against: brute-force triple loops on tiny non-square shapes, PyTorch's CPU
matmul and ``torch.nn.functional.conv1d`` (library routines), closed forms of
the gate (sigmoid(sqrt(C)) when h == k, sign flip, orthogonality, gamma
scaling, scale invariance), hand-worked conv values, tap shifts, K = 1, and
decode-with-state == suffix of one prefill.
"""

import math

import numpy as np
import pytest
import torch

from oracle import kv_proj, gate, conv, gate_conv, bf16_bits_to_f64, f64_to_bf16_bits


def bf16(x):
    return f64_to_bf16_bits(np.asarray(x, dtype=np.float64))


def rand_bf16(rng, shape, std=1.0):
    return bf16(rng.standard_normal(shape) * std)


# ---------------------------------------------------------------------------
# kv_proj
# ---------------------------------------------------------------------------

def test_kv_proj_brute_force_nonsquare():
    rng = np.random.default_rng(0)
    emb = rand_bf16(rng, (3, 5))
    w = rand_bf16(rng, (4, 5))  # [2C, E] with C = 2
    got = bf16_bits_to_f64(kv_proj(emb, w))
    e = bf16_bits_to_f64(emb)
    wf = bf16_bits_to_f64(w)
    for t in range(3):
        for n in range(4):
            s = sum(e[t, k] * wf[n, k] for k in range(5))
            assert got[t, n] == bf16_bits_to_f64(bf16([s]))[0]


def test_kv_proj_one_hot_weight_selects_columns():
    rng = np.random.default_rng(1)
    emb = rand_bf16(rng, (6, 8))
    pick = [3, 0, 7, 7, 1, 5]
    w = np.zeros((6, 8))
    for n, k in enumerate(pick):
        w[n, k] = 1.0
    out = kv_proj(emb, bf16(w))
    assert np.array_equal(out, emb[:, pick])


def test_kv_proj_matches_torch_matmul():
    rng = np.random.default_rng(2)
    emb = rand_bf16(rng, (40, 96), 0.02)
    w = rand_bf16(rng, (64, 96), 0.02)
    ref = (torch.from_numpy(bf16_bits_to_f64(emb)) @ torch.from_numpy(bf16_bits_to_f64(w)).T).numpy()
    got = bf16_bits_to_f64(kv_proj(emb, w))
    # bf16 rounding: |got - ref| <= half an ulp = 2^-9 |ref| (relative)
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-30)


# ---------------------------------------------------------------------------
# gate
# ---------------------------------------------------------------------------

def _kv(k, v):
    return np.concatenate([k, v], axis=1)


def test_gate_closed_form_equal_rows():
    rng = np.random.default_rng(3)
    C = 64
    h = rand_bf16(rng, (5, C))
    v = rand_bf16(rng, (5, C))
    ones = bf16(np.ones(C))
    _, g = gate(h, _kv(h, v), ones, ones, 0.0)
    assert np.allclose(g, 1.0 / (1.0 + math.exp(-math.sqrt(C))), rtol=0, atol=1e-12)


def test_gate_closed_form_negated_and_gamma_scaled():
    rng = np.random.default_rng(4)
    C = 16
    h = rand_bf16(rng, (3, C))
    v = rand_bf16(rng, (3, C))
    neg = bf16(-bf16_bits_to_f64(h))
    ones = bf16(np.ones(C))
    _, g = gate(h, _kv(neg, v), ones, ones, 0.0)
    assert np.allclose(g, 1.0 / (1.0 + math.exp(math.sqrt(C))), atol=1e-12)
    # gamma_h = 0.5, gamma_k = 0.25 everywhere: score scales by 1/8
    _, g2 = gate(h, _kv(h, v), bf16(np.full(C, 0.5)), bf16(np.full(C, 0.25)), 0.0)
    assert np.allclose(g2, 1.0 / (1.0 + math.exp(-math.sqrt(C) / 8)), atol=1e-12)


def test_gate_orthogonal_rows_give_half():
    C = 4
    h = bf16([[1.0, 1.0, 0.0, 0.0]])
    k = bf16([[0.0, 0.0, 3.0, -2.0]])
    v = bf16([[2.0, -4.0, 8.0, 0.5]])
    ones = bf16(np.ones(C))
    u, g = gate(h, _kv(k, v), ones, ones, 1e-6)
    assert g[0] == 0.5
    assert list(bf16_bits_to_f64(u)[0]) == [1.0, -2.0, 4.0, 0.25]


def test_gate_hand_value():
    # h = k = [3, 4], gamma = 1, eps = 0: mean(h^2) = 12.5, <rms h, rms k> = 25/12.5 = 2,
    # divided by sqrt(C) = sqrt(2): score sqrt(2), g = 1/(1+e^-1.41421356...) = 0.80443...
    h = bf16([[3.0, 4.0]])
    ones = bf16([1.0, 1.0])
    _, g = gate(h, _kv(h, bf16([[1.0, 1.0]])), ones, ones, 0.0)
    assert abs(g[0] - 0.8044296825) < 1e-9


def test_gate_scale_invariance_and_zero_v():
    rng = np.random.default_rng(5)
    C = 32
    h = rand_bf16(rng, (4, C))
    k = rand_bf16(rng, (4, C))
    gh = rand_bf16(rng, (C,), 0.1)
    gk = rand_bf16(rng, (C,), 0.1)
    zero_v = bf16(np.zeros((4, C)))
    u, g = gate(h, _kv(k, zero_v), gh, gk, 0.0)
    assert np.all(u == 0)
    h8 = bf16(bf16_bits_to_f64(h) * 8.0)  # exact in bf16
    _, g8 = gate(h8, _kv(k, zero_v), gh, gk, 0.0)
    assert np.allclose(g, g8, atol=1e-12)
    assert np.all((g > 0) & (g < 1))


# ---------------------------------------------------------------------------
# conv
# ---------------------------------------------------------------------------

def test_conv_hand_values():
    # C = 1, K = 2, d = 2, taps w = [0.5, 2] (tap 1 = current token)
    # request 0: x = [1, 2, 3, 4], zero history:
    #   y0 = 2*1 = 2, y1 = 2*2 = 4, y2 = 0.5*1 + 2*3 = 6.5, y3 = 0.5*2 + 2*4 = 9
    # request 1: x = [5], zero history: y = 10
    x = bf16([[1.0], [2.0], [3.0], [4.0], [5.0]])
    w = bf16([[0.5, 2.0]])
    y, state = conv(x, [0, 4, 5], w, 2)
    assert list(bf16_bits_to_f64(y)[:, 0]) == [2.0, 4.0, 6.5, 9.0, 10.0]
    st = bf16_bits_to_f64(state)
    assert list(st[0, :, 0]) == [3.0, 4.0]
    assert list(st[1, :, 0]) == [0.0, 5.0]
    # with history [7, 8] for request 1: y = 0.5*7 + 2*5 = 13.5
    hist = bf16(np.array([[[0.0], [0.0]], [[7.0], [8.0]]]))
    y2, state2 = conv(x, [0, 4, 5], w, 2, hist)
    assert bf16_bits_to_f64(y2)[4, 0] == 13.5
    assert list(bf16_bits_to_f64(state2)[1, :, 0]) == [8.0, 5.0]


def test_conv_matches_torch_conv1d_per_request():
    rng = np.random.default_rng(6)
    C, K, d = 12, 4, 3
    lengths = [7, 0, 19, 1, 11]
    qsl = [0] + list(np.cumsum(lengths))
    T = qsl[-1]
    x = rand_bf16(rng, (T, C))
    w = rand_bf16(rng, (C, K), 0.5)
    y, _ = conv(x, qsl, w, d)
    xf = torch.from_numpy(bf16_bits_to_f64(x))
    wf = torch.from_numpy(bf16_bits_to_f64(w)).unsqueeze(1)  # [C, 1, K]
    for r in range(len(lengths)):
        seg = xf[qsl[r]:qsl[r + 1]].T.unsqueeze(0)  # [1, C, L]
        if seg.shape[-1] == 0:
            continue
        ref = torch.nn.functional.conv1d(seg, wf, padding=(K - 1) * d, dilation=d, groups=C)
        ref = ref[0, :, :seg.shape[-1]].T.numpy()
        assert np.array_equal(y[qsl[r]:qsl[r + 1]], bf16(ref))


def test_conv_one_hot_tap_shifts():
    rng = np.random.default_rng(7)
    C, K, d = 5, 4, 3
    x = rand_bf16(rng, (30, C))
    for i in range(K):
        w = np.zeros((C, K))
        w[:, i] = 1.0
        y, _ = conv(x, [0, 30], bf16(w), d)
        shift = (K - 1 - i) * d
        expect = np.zeros((30, C), np.uint16)
        expect[shift:] = x[:30 - shift]
        assert np.array_equal(y, expect)


def test_conv_k1_is_elementwise_scale():
    rng = np.random.default_rng(8)
    x = rand_bf16(rng, (9, 6))
    w = bf16(np.full((6, 1), 0.5))
    y, state = conv(x, [0, 4, 9], w, 1)
    assert np.array_equal(bf16_bits_to_f64(y), bf16_bits_to_f64(x) * 0.5)
    assert state.shape == (2, 0, 6)


def test_conv_decode_with_state_equals_prefill_suffix():
    rng = np.random.default_rng(9)
    C, K, d = 8, 4, 3
    lengths = [20, 3, 14]
    x = rand_bf16(rng, (sum(lengths), C))
    w = rand_bf16(rng, (C, K), 0.5)
    qsl = [0] + list(np.cumsum(lengths))
    y_full, st_full = conv(x, qsl, w, d)
    cut = [11, 1, 14]
    first = np.concatenate([x[qsl[r]:qsl[r] + cut[r]] for r in range(3)])
    second = np.concatenate([x[qsl[r] + cut[r]:qsl[r + 1]] for r in range(3)])
    q1 = [0] + list(np.cumsum(cut))
    q2 = [0] + list(np.cumsum([n - c for n, c in zip(lengths, cut)]))
    y1, st1 = conv(first, q1, w, d)
    y2, st2 = conv(second, q2, w, d, st1)
    for r in range(3):
        assert np.array_equal(y1[q1[r]:q1[r + 1]], y_full[qsl[r]:qsl[r] + cut[r]])
        assert np.array_equal(y2[q2[r]:q2[r + 1]], y_full[qsl[r] + cut[r]:qsl[r + 1]])
    assert np.array_equal(st2, st_full)


def test_gate_conv_is_conv_of_gate():
    rng = np.random.default_rng(10)
    C = 16
    h = rand_bf16(rng, (12, C))
    kv = rand_bf16(rng, (12, 2 * C))
    g1 = rand_bf16(rng, (C,), 0.1)
    w = rand_bf16(rng, (C, 4), 0.5)
    u, g = gate(h, kv, g1, g1, 1e-6)
    y, st = conv(u, [0, 5, 12], w, 3)
    y2, st2, g2 = gate_conv(h, kv, g1, g1, 1e-6, [0, 5, 12], w, 3)
    assert np.array_equal(y, y2) and np.array_equal(st, st2) and np.array_equal(g, g2)
