"""PLELayer: one per-layer n-gram embedding step through libple.

The user-facing call of the path: n-gram ids -> row gather -> kv_proj ->
gate + short conv, four libple calls on one stream with reusable
intermediate buffers (a table in host memory is gathered in table order). Device memory comes from PyTorch; all arithmetic is in
libple's kernels.
"""

import torch

from . import _lib


class PLELayer:
    """Weights and hash constants of one PLE layer.

    Args:
      table: [rows, D] bf16, or uint8 e4m3 codes (with ``row_scale``), on the
        device or pinned on the host (read over UVA).
      row_scale: [rows] float32 on the device (fp8 tables only).
      layer_multipliers, vocab_sizes, offsets: host int64 hash constants.
      w_kv: [2C, H*D] bf16 merged key/value weight (key rows first).
      gamma_h, gamma_k: [C] bf16 RMSNorm weights; conv_w: [C, K] bf16.
    """

    def __init__(self, table, row_scale, layer_multipliers, vocab_sizes, offsets,
                 eos_token_id, heads_per_ngram, w_kv, gamma_h, gamma_k, conv_w,
                 dilation, eps=1e-6, max_ctas=0):
        self.table = table
        self.row_scale = row_scale
        self.mult = [int(m) for m in layer_multipliers]
        self.V = [int(v) for v in vocab_sizes]
        self.O = [int(o) for o in offsets]
        self.eos = int(eos_token_id)
        self.hpn = int(heads_per_ngram)
        self.ctx_len = len(self.mult) - 1
        self.num_heads = self.ctx_len * self.hpn
        self.head_dim = table.shape[1]
        self.w_kv = w_kv
        self.gamma_h = gamma_h
        self.gamma_k = gamma_k
        self.conv_w = conv_w
        self.dilation = int(dilation)
        self.eps = float(eps)
        self.max_ctas = int(max_ctas)
        self.hidden = w_kv.shape[0] // 2
        self._bufs = {}

    def buffers(self, num_tokens, device):
        key = (num_tokens, str(device))
        b = self._bufs.get(key)
        if b is None:
            E = self.num_heads * self.head_dim
            ws = 0
            if not self.table.is_cuda:  # host table: gather in table order
                ws = _lib.ple_lookup_ordered_workspace(num_tokens, self.num_heads, self.table,
                                                       self.row_scale)
            b = {
                "order_ws": torch.empty((ws,), dtype=torch.uint8, device=device) if ws else None,
                "ids": torch.empty((num_tokens, self.num_heads), dtype=torch.int64, device=device),
                "emb": torch.empty((num_tokens, E), dtype=torch.bfloat16, device=device),
                "kv": torch.empty((num_tokens, 2 * self.hidden), dtype=torch.bfloat16, device=device),
                "y": torch.empty((num_tokens, self.hidden), dtype=torch.bfloat16, device=device),
                "gate": torch.empty((num_tokens,), dtype=torch.float32, device=device),
            }
            self._bufs = {key: b}
        return b

    def forward(self, input_ids, query_start_loc, hidden, ngram_context=None,
                ngram_context_out=None, conv_state=None, conv_state_out=None,
                dev_err=None, stream=None, out=None):
        """Run the layer; returns y [T, C] bf16 (a reused buffer unless ``out``)."""
        T = input_ids.numel()
        b = self.buffers(T, hidden.device)
        y = out if out is not None else b["y"]
        _lib.ple_ngram_ids(input_ids, query_start_loc, ngram_context, self.mult, self.V, self.O,
                           self.eos, self.hpn, b["ids"], ngram_context_out, dev_err, stream)
        if b["order_ws"] is not None:
            _lib.ple_lookup_ordered(b["ids"], self.table, b["emb"], b["order_ws"],
                                    row_scale=self.row_scale, max_ctas=self.max_ctas,
                                    dev_err=dev_err, stream=stream)
        else:
            _lib.ple_lookup(b["ids"], self.table, b["emb"], row_scale=self.row_scale,
                            max_ctas=self.max_ctas, dev_err=dev_err, stream=stream)
        _lib.ple_kv_proj(b["emb"], self.w_kv, b["kv"], dev_err=dev_err, stream=stream)
        _lib.ple_gate_conv(hidden, b["kv"], self.gamma_h, self.gamma_k, query_start_loc,
                           self.conv_w, self.dilation, y, eps=self.eps, conv_state=conv_state,
                           conv_state_out=conv_state_out, gate_out=b["gate"],
                           dev_err=dev_err, stream=stream)
        return y

    # launches of libple kernels per forward (ids, gather, kv_proj, gate, conv);
    # a host table's ordered gather adds three (count, scan, scatter)
    LAUNCHES_PER_FORWARD = 5
    ORDERED_GATHER_EXTRA = 3

    def launches_per_forward(self):
        return self.LAUNCHES_PER_FORWARD + (0 if self.table.is_cuda else self.ORDERED_GATHER_EXTRA)
