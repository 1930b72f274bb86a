"""PLELayer: one per-layer n-gram embedding step through libple.

The user-facing call of the path: n-gram ids -> row gather -> kv_proj ->
gate + short conv, four libple calls on one stream with reusable
intermediate buffers (a table in host memory is gathered in table order). Device memory comes from PyTorch; all arithmetic is in
libple's kernels.
"""

import ctypes

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
                 dilation, eps=1e-6, max_ctas=0, fuse_gate=None, fuse_ids=None):
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
        # gate reductions inside the projection (ple_kv_proj_gate +
        # ple_gated_conv) where the hidden size allows it (a multiple of 256),
        # else ple_kv_proj + ple_gate_conv
        can_fuse = self.hidden % 256 == 0
        self.fuse_gate = can_fuse if fuse_gate is None else bool(fuse_gate)
        if self.fuse_gate and not can_fuse:
            raise ValueError(f"fuse_gate needs a hidden size that is a multiple of 256, "
                             f"not {self.hidden}")
        # ids hashed inside the gather (ple_ngram_lookup) for a table in HBM:
        # None = for steps of up to FUSED_IDS_MAX_TOKENS tokens; a host table
        # is gathered in table order, after the ids
        self.fuse_ids = None if fuse_ids is None else bool(fuse_ids) and table.is_cuda
        self._bufs = {}

    # Measured on a GB300 inside CUDA graphs: the fused lookup saves 4 us of a
    # 1024-token decode step and is level with the two kernels at 8192 tokens.
    FUSED_IDS_MAX_TOKENS = 4096

    def fused_ids_for(self, num_tokens):
        """Whether embed hashes the ids inside the gather for this step."""
        if not self.table.is_cuda:
            return False
        if self.fuse_ids is None:
            return num_tokens <= self.FUSED_IDS_MAX_TOKENS
        return self.fuse_ids

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
                # zero-filled once: each completed call leaves it zeroed
                "gate_ws": (torch.zeros((_lib.ple_kv_proj_gate_workspace(num_tokens, self.hidden),),
                                        dtype=torch.uint8, device=device)
                            if self.fuse_gate and num_tokens > 0 else None),
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
        self.embed(input_ids, query_start_loc, b["ids"], b["emb"], b["order_ws"],
                   ngram_context=ngram_context, ngram_context_out=ngram_context_out,
                   dev_err=dev_err, stream=stream)
        self.mix(b["emb"], hidden, query_start_loc, y, conv_state=conv_state,
                 conv_state_out=conv_state_out, dev_err=dev_err, stream=stream)
        return y

    def embed(self, input_ids, query_start_loc, ids, emb, order_ws=None, ngram_context=None,
              ngram_context_out=None, dev_err=None, stream=None, max_ctas=None):
        """n-gram ids -> row gather into ``emb`` [T, H*D] (``order_ws``: the
        ordered gather's workspace, required for a host table)."""
        ctas = self.max_ctas if max_ctas is None else int(max_ctas)
        if not self.fused_ids_for(input_ids.numel()):  # ids, then the gather (table order for a host table)
            _lib.ple_ngram_ids(input_ids, query_start_loc, ngram_context, self.mult, self.V,
                               self.O, self.eos, self.hpn, ids, ngram_context_out, dev_err, stream)
            if not self.table.is_cuda:
                _lib.ple_lookup_ordered(ids, self.table, emb, order_ws, row_scale=self.row_scale,
                                        max_ctas=ctas, dev_err=dev_err, stream=stream)
            else:
                _lib.ple_lookup(ids, self.table, emb, row_scale=self.row_scale, max_ctas=ctas,
                                dev_err=dev_err, stream=stream)
        else:  # HBM table: ids hashed inside the gather (ids still written to ``ids``)
            _lib.ple_ngram_lookup(input_ids, query_start_loc, ngram_context, self.mult, self.V,
                                  self.O, self.eos, self.hpn, self.table, emb,
                                  row_scale=self.row_scale, ids_out=ids,
                                  ngram_context_out=ngram_context_out, max_ctas=ctas,
                                  dev_err=dev_err, stream=stream)

    def mix(self, emb, hidden, query_start_loc, out, conv_state=None, conv_state_out=None,
            dev_err=None, stream=None):
        """kv_proj of ``emb`` -> gate with ``hidden`` -> short conv into ``out``."""
        self.project(emb, hidden, dev_err=dev_err, stream=stream)
        self.convolve(hidden, query_start_loc, out, conv_state=conv_state,
                      conv_state_out=conv_state_out, dev_err=dev_err, stream=stream)

    def project(self, emb, hidden, dev_err=None, stream=None):
        """The projection of ``emb`` into the layer's kv buffer; fused, it
        writes v and the gate scalars (k stays on chip)."""
        b = self.buffers(hidden.shape[0], hidden.device)
        if self.fuse_gate:
            _lib.ple_kv_proj_gate(emb, self.w_kv, hidden, self.gamma_h, self.gamma_k, b["kv"],
                                  b["gate"], b["gate_ws"], eps=self.eps, dev_err=dev_err,
                                  stream=stream)
        else:
            _lib.ple_kv_proj(emb, self.w_kv, b["kv"], dev_err=dev_err, stream=stream)

    def convolve(self, hidden, query_start_loc, out, conv_state=None, conv_state_out=None,
                 dev_err=None, stream=None):
        """Gate (unless the projection did its reductions) and short conv of
        the layer's kv buffer into ``out``."""
        b = self.buffers(hidden.shape[0], hidden.device)
        if self.fuse_gate:
            _lib.ple_gated_conv(b["kv"], b["gate"], query_start_loc, self.conv_w, self.dilation,
                                out, conv_state=conv_state, conv_state_out=conv_state_out,
                                dev_err=dev_err, stream=stream)
        else:
            _lib.ple_gate_conv(hidden, b["kv"], self.gamma_h, self.gamma_k, query_start_loc,
                               self.conv_w, self.dilation, out, eps=self.eps,
                               conv_state=conv_state, conv_state_out=conv_state_out,
                               gate_out=b["gate"], dev_err=dev_err, stream=stream)

    def launches_per_forward(self, num_tokens):
        """libple kernels per forward: the n-gram lookup (ids hashed inside the
        gather; a host table: ids, then count, scan, scatter and the ordered
        gather), then kv_proj_gate and the gated conv (unfused: kv_proj, the
        gate pass and the conv pass)."""
        embed = 1 if self.fused_ids_for(num_tokens) else (2 if self.table.is_cuda else 5)
        return embed + (2 if self.fuse_gate else 3)


class PLEHostPipeline:
    """PLELayer over pinned host buffers, with each step's transfers
    overlapping its neighbours' compute.

    ``submit`` enqueues one step: the inputs (token ids, query_start_loc,
    hidden) go to the device on a copy-in stream, the layer runs on the
    compute stream, and the output comes back on a copy-out stream into the
    caller's pinned buffer. ``depth`` device buffer sets rotate, so step k's
    upload and step k-1's download run while step k-1 / k computes; a buffer
    set is reused only after the step that last used it has been read back.
    Three sets (the default) leave the transfers a step of slack: at 256 x 4
    decode the end-to-end rate is 15.6 M tokens/s/layer against 14.9 M with
    two and 15.4 M with four (measured). The copies run asynchronously: a
    step's host inputs must not be changed, nor its host output read or
    reused, before ``synchronize`` (or the ``synchronize()`` of the object
    ``submit`` returns). The streams are PyTorch's; the copies, the events
    ordering them and the graph launches are issued by libple's step
    runtime (ple_step_begin / ple_step_end / ple_step); all arithmetic is in
    libple.

    With ``graphs`` (the default) a slot's layer calls are captured into a
    CUDA graph (ple_graph_begin / ple_graph_end) the second time the slot
    runs with the same argument tensors (the first run is launched directly
    and warms the library up); from then on a step is one ple_step call: its
    uploads, the graph launch and its read-back with their event waits,
    without a Python call per copy, wait or kernel. Small steps (decode) are
    otherwise bound by the host. A change of argument tensors captures
    another graph.
    """

    class Done:
        """Completion of one submitted step (its read-back)."""

        def __init__(self, event):
            self.event = event

        def synchronize(self):
            _lib.ple_event_synchronize(self.event)

    def __init__(self, layer, num_tokens, num_reqs, device, depth=3, graphs=True):
        self.layer = layer
        self.device = torch.device(device)
        self.graphs = bool(graphs)
        self._graphs = {}   # (slot, argument tensors) -> ple_graph handle
        self._seen = set()  # (slot, argument tensors) run once directly
        self._capture = torch.cuda.Stream(self.device) if self.graphs else None
        layer.buffers(num_tokens, self.device)  # allocated outside any capture
        self.copy_in = torch.cuda.Stream(self.device)
        self.compute = torch.cuda.Stream(self.device)
        self.copy_out = torch.cuda.Stream(self.device)
        self._h = [ctypes.c_void_p(st.cuda_stream) for st in (self.copy_in, self.compute, self.copy_out)]
        C = layer.hidden
        self.slots = []
        for _ in range(depth):
            s = {
                "ids": torch.empty((num_tokens,), dtype=torch.int32, device=self.device),
                "qsl": torch.empty((num_reqs + 1,), dtype=torch.int32, device=self.device),
                "hidden": torch.empty((num_tokens, C), dtype=torch.bfloat16, device=self.device),
                "y": torch.empty((num_tokens, C), dtype=torch.bfloat16, device=self.device),
            }
            # events: inputs on the device / the layer read the inputs and wrote
            # y / y back on the host
            s["events"] = [ctypes.c_void_p(_lib.ple_event_create()) for _ in range(3)]
            s["up"] = _lib.copies([(s[n].data_ptr(), None, s[n].numel() * s[n].element_size())
                                   for n in ("ids", "qsl", "hidden")])
            s["down"] = _lib.copies([(None, s["y"].data_ptr(),
                                      s["y"].numel() * s["y"].element_size())])
            s["done"] = PLEHostPipeline.Done(s["events"][2])
            self.slots.append(s)
        self.k = 0

    def submit(self, h_input_ids, h_query_start_loc, h_hidden, h_out, **forward_kwargs):
        """Enqueue one step; ``forward_kwargs`` go to PLELayer.forward (device
        carry-over buffers, dev_err). Returns the step's completion (an
        object with ``synchronize()``)."""
        if not self.slots:
            raise RuntimeError("PLEHostPipeline.submit after close()")
        slot = self.k % len(self.slots)
        s = self.slots[slot]
        self.k += 1
        up, down = s["up"], s["down"]
        for i, (h, d) in enumerate(((h_input_ids, s["ids"]), (h_query_start_loc, s["qsl"]),
                                    (h_hidden, s["hidden"]))):
            if h.dtype != d.dtype or h.shape != d.shape or h.is_cuda:
                raise ValueError(f"host input {i}: expected a host {d.dtype} tensor of shape "
                                 f"{tuple(d.shape)}, got {h.dtype} {tuple(h.shape)} "
                                 f"on {h.device}")
            up[i].src = h.data_ptr()
        y = s["y"]
        if h_out.dtype != y.dtype or h_out.shape != y.shape or h_out.is_cuda:
            raise ValueError(f"host output: expected a host {y.dtype} tensor of shape "
                             f"{tuple(y.shape)}")
        down[0].dst = h_out.data_ptr()
        ci, cp, co = self._h
        loaded, computed, returned = s["events"]
        key = (slot,) + tuple((n, v.data_ptr() if torch.is_tensor(v) else v)
                              for n, v in forward_kwargs.items())
        g = self._graphs.get(key)
        if g is not None:
            _lib._check("ple_step", _lib.lib().ple_step(ci, cp, co, up, 3, g, down, 1,
                                                        loaded, computed, returned))
            return s["done"]
        _lib._check("ple_step_begin", _lib.lib().ple_step_begin(ci, cp, up, 3, loaded, computed,
                                                                returned))
        self._forward(key, s, forward_kwargs)
        _lib._check("ple_step_end", _lib.lib().ple_step_end(cp, co, down, 1, computed, returned))
        return s["done"]

    def _forward(self, key, s, kwargs):
        def run(stream):
            self.layer.forward(s["ids"], s["qsl"], s["hidden"], stream=stream, out=s["y"],
                               **kwargs)
        if not self.graphs or key not in self._seen:
            if self.graphs:
                self._seen.add(key)
            run(self.compute)
            return
        # capture with nothing else in flight; the graph does not run now
        torch.cuda.synchronize(self.device)
        _lib.ple_graph_begin(self._capture)
        try:
            run(self._capture)
        except BaseException:
            _lib.ple_graph_destroy(_lib.ple_graph_end(self._capture))  # end the capture, drop it
            raise
        g = _lib.ple_graph_end(self._capture)
        self._graphs[key] = g
        _lib.ple_graph_launch(g, self.compute)

    def synchronize(self):
        self.copy_out.synchronize()

    def close(self):
        """Wait for every submitted step, then release the graphs and events."""
        if not self.slots:
            return
        torch.cuda.synchronize(self.device)
        for g in self._graphs.values():
            _lib.ple_graph_destroy(g)
        self._graphs.clear()
        for s in self.slots:
            for ev in s["events"]:
                _lib.ple_event_destroy(ev)
        self.slots = []

    def __del__(self):
        try:
            self.close()
        except Exception:  # interpreter shutdown: the library or CUDA may be gone
            pass


class PLEChain:
    """Several PLE layers over the same tokens, with the next layers' n-gram
    ids and row gathers prefetched on a side stream.

    Layer i+1's ids and gather (its embed stage) only need the tokens, so
    they run on a side stream into one of two staging buffers while layer i's
    kv_proj, gate and conv (its mix stage) run on the main stream; a staging
    buffer is refilled once the layer that read it has finished, so the
    gather overlaps the next layer's projection. With ``prefetch=False`` the
    layers run one after the other on the main stream. Results are the same
    either way.

    prefetch_ctas caps the side-stream gathers' grid: None = one CTA per SM
    for tables in HBM (a gather CTA fits beside the projection's CTA on the
    same SM, so the two run together) and the full grid for host tables; 0 =
    the full grid.
    """

    def __init__(self, layers, prefetch=True, prefetch_ctas=None):
        self.layers = list(layers)
        self.prefetch = bool(prefetch)
        if prefetch_ctas is None:
            on_device = all(l.table.is_cuda for l in self.layers)
            prefetch_ctas = (torch.cuda.get_device_properties(
                torch.cuda.current_device()).multi_processor_count if on_device else 0)
        self.prefetch_ctas = int(prefetch_ctas)
        self._bufs = {}
        self._side = {}

    def _staging(self, num_tokens, device):
        key = (num_tokens, str(device))
        st = self._bufs.get(key)
        if st is None:
            l0 = self.layers[0]
            E = l0.num_heads * l0.head_dim
            st = []
            for _ in range(2):
                ws = None
                host = [l for l in self.layers if not l.table.is_cuda]
                if host:
                    n = max(_lib.ple_lookup_ordered_workspace(num_tokens, l.num_heads, l.table,
                                                              l.row_scale) for l in host)
                    ws = torch.empty((n,), dtype=torch.uint8, device=device)
                st.append({
                    "ids": torch.empty((num_tokens, l0.num_heads), dtype=torch.int64, device=device),
                    "emb": torch.empty((num_tokens, E), dtype=torch.bfloat16, device=device),
                    "ws": ws, "ready": torch.cuda.Event(), "free": torch.cuda.Event(),
                })
            self._bufs = {key: st}
        return st

    def forward(self, input_ids, query_start_loc, hiddens, outs, ngram_context=None,
                ngram_context_out=None, conv_states=None, conv_states_out=None, dev_err=None,
                stream=None):
        """Run every layer: layer i reads hiddens[i] and writes outs[i];
        conv_states / conv_states_out are per-layer lists (or None);
        ngram_context_out is written once (the tokens are the same for all
        layers)."""
        L = len(self.layers)
        device = input_ids.device
        main = stream if stream is not None else torch.cuda.current_stream(device)
        st = self._staging(input_ids.numel(), device)
        cs = conv_states or [None] * L
        cso = conv_states_out or [None] * L

        def embed(i, s):
            slot = st[i % 2]
            self.layers[i].embed(input_ids, query_start_loc, slot["ids"], slot["emb"], slot["ws"],
                                 ngram_context=ngram_context,
                                 ngram_context_out=ngram_context_out if i == 0 else None,
                                 dev_err=dev_err, stream=s,
                                 max_ctas=self.prefetch_ctas if s is not main else None)

        if not self.prefetch:
            for i in range(L):
                embed(i, main)
                self.layers[i].mix(st[i % 2]["emb"], hiddens[i], query_start_loc, outs[i],
                                   conv_state=cs[i], conv_state_out=cso[i], dev_err=dev_err,
                                   stream=main)
            return outs
        side = self._side.get(str(device))
        if side is None:
            side = self._side[str(device)] = torch.cuda.Stream(device)
        side.wait_stream(main)  # inputs written on the main stream
        for i in range(min(2, L)):
            embed(i, side)
            st[i % 2]["ready"].record(side)
        for i in range(L):
            slot = st[i % 2]
            main.wait_event(slot["ready"])
            layer = self.layers[i]
            layer.project(slot["emb"], hiddens[i], dev_err=dev_err, stream=main)
            layer.convolve(hiddens[i], query_start_loc, outs[i], conv_state=cs[i],
                           conv_state_out=cso[i], dev_err=dev_err, stream=main)
            # The projection has read this staging buffer; refill it with layer
            # i+2's rows once the conv is done too, so that the gather runs
            # beside layer i+1's projection (tensor-bound, one CTA per SM)
            # rather than beside this layer's conv (memory-bound, SMs full).
            slot["free"].record(main)
            if i + 2 < L:
                side.wait_event(slot["free"])
                embed(i + 2, side)
                slot["ready"].record(side)
        main.wait_stream(side)
        return outs
