"""Oracle for the dense part of the PLE layer: kv_proj, gate, short conv.

TEST INFRASTRUCTURE (see the package docstring).

All arithmetic is float64 on the exact values of bf16 inputs; each step's
output is rounded to bf16 (nearest even) at the step's boundary, the rounding
points the CUDA path also has (ids -> rows -> kv -> gated u -> conv y).

Sources and readings:
  * ``kv_proj``: PR#54517 report ("Fuse Qwen4Exp PLE kernels"), 实现拆解
    item 1 -- ``key_proj`` and ``value_proj`` merged into one
    ``MergedColumnParallelLinear``. Merged weight ``W = [W_k; W_v]`` of shape
    [2C, E] (key rows first), ``kv = emb @ W^T`` with no bias, so
    ``kv[:, :C]`` is k and ``kv[:, C:]`` is v.
  * ``gate``: same report, 实现拆解 item 2, "PLE gating and normalisation";
    the pages give no formula. Reading: per token a scalar gate
    ``g = sigmoid(<rms(h) * gamma_h, rms(k) * gamma_k> / sqrt(C))`` with
    ``rms(x) = x / sqrt(mean(x^2) + eps)``, and ``u = g * v``. No residual, no
    activation. Parity against the real model is unpinned (the pages hold no
    numbers); the formula as read is pinned by closed forms in the tests.
  * ``conv``: same report, 实现拆解 items 2, 4 and 5 -- a dilated short conv
    with prefill and decode paths and a cached state. Reading: causal,
    depthwise (one filter per channel), ``torch.nn.functional.conv1d``
    orientation with left history, no bias, no activation:
    ``y_t[c] = sum_i w[c, i] * u_{t - (K-1-i)*d}[c]`` over each request's
    virtual sequence ``state ++ segment``; a missing state is zeros. The new
    state is the last (K-1)*d inputs of that virtual sequence.
"""

import math

import numpy as np

from .numerics import bf16_bits_to_f64, f64_to_bf16_bits
from .ngram_ids import request_spans


def kv_proj(emb_bits, w_bits):
    """kv = round_bf16(emb @ W^T) in float64.

    Args: emb_bits [T, E] uint16, w_bits [2C, E] uint16 (bf16 bits).
    Returns: [T, 2C] uint16.
    """
    emb = bf16_bits_to_f64(emb_bits)
    w = bf16_bits_to_f64(w_bits)
    return f64_to_bf16_bits(emb @ w.T)


def _rms_normalise(x, eps):
    return x / math.sqrt(float(np.mean(x * x)) + eps)


def gate(hidden_bits, kv_bits, gamma_h_bits, gamma_k_bits, eps):
    """RMSNorm + sigmoid gate of every token.

    Args:
      hidden_bits: [T, C] uint16; kv_bits: [T, 2C] uint16 (k then v);
      gamma_h_bits, gamma_k_bits: [C] uint16; eps: float.
    Returns:
      (u_bits [T, C] uint16 = round_bf16(g_t * v_t), g [T] float64).
    """
    h = bf16_bits_to_f64(hidden_bits)
    kv = bf16_bits_to_f64(kv_bits)
    T, C = h.shape
    assert kv.shape == (T, 2 * C)
    k = kv[:, :C]
    v = kv[:, C:]
    gh = bf16_bits_to_f64(gamma_h_bits)
    gk = bf16_bits_to_f64(gamma_k_bits)
    g = np.empty(T, dtype=np.float64)
    u = np.empty((T, C), dtype=np.float64)
    for t in range(T):
        hn = _rms_normalise(h[t], eps) * gh
        kn = _rms_normalise(k[t], eps) * gk
        score = float(np.dot(hn, kn)) / math.sqrt(C)
        g[t] = 1.0 / (1.0 + math.exp(-score))
        u[t] = g[t] * v[t]
    return f64_to_bf16_bits(u), g


def conv(x_bits, query_start_loc, w_bits, dilation, conv_state_bits=None,
         num_tokens=None):
    """Dilated causal depthwise short conv over ragged requests.

    Args:
      x_bits: [T, C] uint16 conv inputs.
      query_start_loc: [R+1] request boundaries (tokens past the last boundary
        continue the last request).
      w_bits: [C, K] uint16 taps; tap K-1 multiplies the current token.
      dilation: d >= 1.
      conv_state_bits: [R, (K-1)*d, C] uint16 history (oldest first) or None.
    Returns:
      (y_bits [T, C] uint16, state_out_bits [R, (K-1)*d, C] uint16).
    """
    x = bf16_bits_to_f64(x_bits)
    T, C = x.shape
    if num_tokens is None:
        num_tokens = T
    w = bf16_bits_to_f64(w_bits)
    Cw, K = w.shape
    assert Cw == C and K >= 1 and dilation >= 1
    W = (K - 1) * dilation
    spans = request_spans(query_start_loc, num_tokens)
    y = np.zeros((T, C), dtype=np.float64)
    state_out = np.zeros((len(spans), W, C), dtype=np.float64)
    for r, (start, end) in enumerate(spans):
        if conv_state_bits is None:
            history = np.zeros((W, C), dtype=np.float64)
        else:
            history = bf16_bits_to_f64(conv_state_bits[r])
        seq = np.concatenate([history, x[start:end]], axis=0)
        for p in range(W, seq.shape[0]):
            acc = np.zeros(C, dtype=np.float64)
            for i in range(K):
                acc += w[:, i] * seq[p - (K - 1 - i) * dilation]
            y[start + p - W] = acc
        if W > 0:
            state_out[r] = seq[seq.shape[0] - W:]
    return f64_to_bf16_bits(y), f64_to_bf16_bits(state_out)


def gate_conv(hidden_bits, kv_bits, gamma_h_bits, gamma_k_bits, eps,
              query_start_loc, w_bits, dilation, conv_state_bits=None):
    """Gate followed by the short conv on the gated values (u rounded to bf16).

    Returns (y_bits, state_out_bits, g).
    """
    u_bits, g = gate(hidden_bits, kv_bits, gamma_h_bits, gamma_k_bits, eps)
    y_bits, state_bits = conv(u_bits, query_start_loc, w_bits, dilation,
                              conv_state_bits)
    return y_bits, state_bits, g


def layer_forward(input_ids, query_start_loc, ngram_context, layer_multipliers,
                  vocab_sizes, offsets, eos_token_id, heads_per_ngram,
                  table, row_scale, hidden_bits, w_kv_bits, gamma_h_bits,
                  gamma_k_bits, eps, conv_w_bits, dilation, conv_state_bits=None):
    """The whole per-layer chain: ids -> gather -> kv_proj -> gate -> conv.

    ``table`` is uint16 bf16 bits, or uint8 e4m3 codes when ``row_scale`` is
    given. Returns a dict of every intermediate.
    """
    from .ngram_ids import ngram_ids
    from .lookup import lookup_bf16, lookup_fp8

    ids, ctx_out = ngram_ids(input_ids, query_start_loc, ngram_context,
                             layer_multipliers, vocab_sizes, offsets,
                             eos_token_id, heads_per_ngram)
    ids = np.asarray(ids, dtype=np.int64).reshape(len(input_ids), -1)
    if row_scale is None:
        emb = lookup_bf16(ids, table)
    else:
        emb = lookup_fp8(ids, table, row_scale)
    kv = kv_proj(emb, w_kv_bits)
    y, state_out, g = gate_conv(hidden_bits, kv, gamma_h_bits, gamma_k_bits,
                                eps, query_start_loc, conv_w_bits, dilation,
                                conv_state_bits)
    return {"ids": ids, "ngram_context_out": ctx_out, "emb": emb, "kv": kv,
            "gate": g, "y": y, "conv_state_out": state_out}
