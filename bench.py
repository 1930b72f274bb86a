#!/usr/bin/env python
"""Benchmark of the per-layer n-gram embedding (PLE / Engram) path on GB300.

One step = one pass of the whole hot path over one batch for one layer:
n-gram ids -> row gather -> kv_proj (with the gate's reductions) -> gated
short conv (libple launches only). Metric: PLE tokens/sec/layer.

The default run measures every workload of the input recipe in one go and
prints ONE JSON line: the headline is the largest workload, fp8x8 (8 layers,
each with its own 8 GiB fp8 e4m3 table and per-row scales, 32768-token
prefill over 64 ragged requests, Zipf tokens, hidden 4096; one step = one
layer, rotating over the 8 layers), and "configs" holds the same figures for
every workload: tiny (512 tokens), prefill8k (8192 tokens, 8.2 GB bf16 table
in HBM), decode256x4 (256 x 4 decode tokens with carried context and conv
state) and uva32g (8192 tokens over a 32 GiB bf16 table in pinned host
memory read over the host link, reported against the measured link rate and
the PCIe5 x16 nominal).

Steps rotate over independent layer parameter sets (table, kv_proj weight,
gammas, conv taps, hash multipliers, hidden states, token ids): one rotation
touches far more than the 129 MB L2, so no step finds its inputs cached by an
earlier one and no L2 flush is needed.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload all|fp8x8|prefill8k|decode256x4|tiny|uva32g]

Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(the path has no exchange step on one node's replicas); rank 0 prints one
JSON line with the whole-job rate, timed as the max over ranks.
"""

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "PLE tokens/sec/layer"
UNIT = "tokens/s/layer"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
E2E_MIN_STEPS = 100  # end-to-end steps timed at least (host buffers, three streams)
NUM_SETS = 4
# the oracle's stages (cpu_baseline and the reference arm)
ORACLE_STAGES = ("ngram_ids", "lookup", "kv_proj", "gate_conv")
# Timed kernels per step. The ids and the gather: one kernel (ngram_lookup)
# for a table in HBM, else the ids, then the table-order gather. The dense
# part: the projection with the gate's reductions, then the gated conv (hidden
# sizes that are multiples of 256), else the projection, then gate_conv's two
# passes (gate reduction, gated conv).


# ---------------------------------------------------------------------------
# distributed plumbing (replicas: barrier + max-over-ranks timing only)
# ---------------------------------------------------------------------------

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def dist_setup(backend):
    import torch.distributed as dist
    rank, world, _ = dist_env()
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return rank, world


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(value, device="cpu"):
    """Max of a float over all ranks (identity when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# peaks, clocks, ncu traffic
# ---------------------------------------------------------------------------

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            data = json.load(f)
        peaks = {}
        for key in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained"):
            v = data.get(key)
            if isinstance(v, dict):
                v = v.get("value")
            if v is not None:
                peaks[key] = float(v)
        if "hbm_gbs" in peaks and "bf16_tflops" in peaks:
            return peaks, "measured"
    except (OSError, ValueError, TypeError):
        pass
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []
        self._thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self._thread = threading.Thread(target=self._read, daemon=True)
        self._thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self._thread is not None:
            self._thread.join(timeout=2)
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, flag in zip(names, parts[5:9]):
                if flag.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_median": float(np.median(power)) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def source_hash(path):
    """sha256 prefix of a kernel source's code: comments and whitespace are
    removed first, so an edit of comments alone keeps a profile valid."""
    import re
    text = open(path, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    text = re.sub(r"\s+", "", text)
    return hashlib.sha256(text.encode()).hexdigest()[:16]


def ncu_traffic(kernel, workload, field="dram_bytes_per_launch"):
    """bytes per launch (``field``: DRAM bytes, or for a kernel bound by the
    host link the bytes L2 read from host memory) from the committed ncu
    summary of ``kernel`` on ``workload``, or None when the summary is
    missing or the kernel source changed since."""
    summary = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    src = os.path.join(ROOT, "hashed_gram_embedding_gb300", "csrc",
                       {"kv_proj": "kv_proj.cu", "kv_proj_gate": "kv_proj.cu",
                        "ngram_lookup": "lookup.cu",
                        "lookup": "lookup.cu", "gate_conv": "gate_conv.cu",
                        "conv": "gate_conv.cu", "ngram_ids": "ngram_ids.cu"}[kernel])
    try:
        text = open(summary).read()
    except OSError:
        return None
    fields = {}
    for line in text.splitlines():
        if ":" in line and line.strip().startswith(("source_sha256", field)):
            k, _, v = line.strip().partition(":")
            fields[k.strip()] = v.strip().strip("`")
    if fields.get("source_sha256") != source_hash(src):
        return None
    try:
        return float(fields[field])
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------------------
# workload set-up
# ---------------------------------------------------------------------------

def algorithmic_work(w):
    """Bytes (or flops) one launch of each kernel must move (or do)."""
    T, H, D, C, E = w.num_tokens, w.num_heads, w.head_dim, w.hidden, w.emb_dim
    elem = 1 if w.table_dtype == "fp8" else 2
    # decode steps also read and write every request's conv state [(K-1)d, C]
    state = 2 * w.num_reqs * (w.conv_k - 1) * w.dilation * C * 2 if w.decode else 0
    row_read = H * D * elem + (H * 4 if w.table_dtype == "fp8" else 0)
    lookup = (("link", T * row_read) if w.table_loc == "host"
              else ("hbm", T * (H * 8 + row_read + H * D * 2)))
    return {
        "ngram_ids": ("hbm", T * 4 + T * H * 8 + (w.num_reqs + 1) * 4),
        # token ids in, rows read, rows and ids written
        "ngram_lookup": ("hbm", T * (4 + row_read + H * D * 2 + H * 8)),
        "lookup": lookup,
        "kv_proj": ("tensor", 2.0 * T * E * 2 * C),
        "gate_conv": ("hbm", T * (C * 2 + 2 * C * 2 + C * 2) + state),
        # the gate reductions ride in the projection's epilogue: tensor-bound
        "kv_proj_gate": ("tensor", 2.0 * T * E * 2 * C),
        # v and g in, y out (+ the carried conv state)
        "conv": ("hbm", T * (C * 2 + 4 + C * 2) + state),
    }


def make_sets(torch, w, device, num_sets):
    from hashed_gram_embedding_gb300 import workloads as wl
    sets = []
    for s in range(num_sets):
        host = wl.host_inputs(w, step=s)
        dense = wl.dense_inputs(torch, w, device, layer=s, step=s, random_gamma=True)
        table, row_scale = wl.make_table(torch, w, device, layer=s)
        sets.append({
            "host": host,
            "input_ids": torch.from_numpy(host["input_ids"]).to(device),
            "qsl": torch.from_numpy(host["query_start_loc"]).to(device),
            "ctx": None if host["ngram_context"] is None else torch.from_numpy(host["ngram_context"]).to(device),
            "mult": wl.layer_multipliers(w, s),
            "table": table, "row_scale": row_scale, **dense,
        })
    return sets


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

# The default run: the headline on the largest workload (8 fp8 layers, 32k
# tokens), then every other workload measured in the same run and reported
# under "configs" in the same line.
HEADLINE = "fp8x8"
ALL_WORKLOADS = ("fp8x8", "tiny", "prefill8k", "decode256x4", "uva32g")
PCIE5_X16_GBS = 63.0  # nominal per direction, context for host-table gathers


def run_ours(args):
    import gc
    import torch
    from hashed_gram_embedding_gb300 import build as build_mod
    from hashed_gram_embedding_gb300 import _lib

    rank, world, local_rank = dist_env()
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    dist_setup("nccl")
    if rank == 0 or not os.path.exists(_lib.LIB_PATH):
        build_mod.build()
    barrier()

    names = ALL_WORKLOADS if args.workload == "all" else (args.workload,)
    sampler = ClockSampler(local_rank)
    sampler.start()
    lines = {}
    for i, name in enumerate(names):
        lines[name] = measure_workload(torch, args, name, device, rank, world, headline=i == 0)
        gc.collect()  # host tables hold their owner in a reference cycle
        torch.cuda.empty_cache()
    clocks = sampler.stop()
    if rank != 0:
        return None
    line = lines[names[0]]
    line["clocks"] = clocks
    if len(names) > 1:
        line["configs"] = {n: config_summary(lines[n]) for n in names}
    return line


def config_summary(line):
    """The per-workload figures reported side by side under "configs"."""
    out = {"value": line["value"], "unit": line["unit"], "ms_per_step": line["ms_per_step"],
           "mode": line["config"]["mode"], "num_tokens": line["config"]["num_tokens"],
           "table_loc": line["config"]["table_loc"], "table_dtype": line["config"]["table_dtype"],
           "e2e": line["e2e"]["value"], "gather": line["gather"],
           "roofline": {k: line["roofline"][k] for k in ("kernel", "bound", "achieved", "peak",
                                                         "unit", "frac", "traffic",
                                                         "traffic_counters")},
           "kernels": {k: {"us": v["us"], "achieved": v["achieved"], "unit": v["unit"],
                           "peak": v["peak"], "frac": v["frac"]}
                       for k, v in line["kernels"].items()}}
    if "chain" in line:
        out["chain"] = line["chain"]
    if "overlap" in line:
        out["overlap"] = line["overlap"]
    if "sharded" in line:
        out["sharded"] = line["sharded"]
    return out


def measure_workload(torch, args, name, device, rank, world, headline):
    """Set up one workload's layer sets, time its steps (per-kernel events,
    then CUDA-graph replays), its end-to-end steps from pinned host buffers,
    and return its JSON line (rank 0; None elsewhere)."""
    from hashed_gram_embedding_gb300 import _lib
    from hashed_gram_embedding_gb300 import workloads as wl
    from hashed_gram_embedding_gb300 import PLELayer

    w = wl.WORKLOADS[name]
    if args.vocab_start:
        w = wl.scaled(w, vocab_start=args.vocab_start)  # smaller table (profiling cases)
    # one step = one layer; multi-layer workloads rotate over their layers
    num_sets = w.num_layers if w.num_layers > 1 else (NUM_SETS if w.table_loc == "hbm" else 1)
    if args.layer_sets:
        num_sets = args.layer_sets
    sets = make_sets(torch, w, device, num_sets)
    T, H, C = w.num_tokens, w.num_heads, w.hidden
    fuse = C % 256 == 0 and not args.no_fuse_gate
    fuse_ids = w.table_loc == "hbm" and (
        args.fuse_ids == "on" or (args.fuse_ids == "auto" and T <= PLELayer.FUSED_IDS_MAX_TOKENS))
    KERNELS = ((("ngram_lookup",) if fuse_ids else ("ngram_ids", "lookup")) +
               (("kv_proj_gate", "conv") if fuse else ("kv_proj", "gate_conv")))
    gate_ws = (torch.zeros((_lib.ple_kv_proj_gate_workspace(T, C),), dtype=torch.uint8,
                           device=device) if fuse else None)
    # activation buffers shared by the steps (as an engine reuses them), except
    # the gather's ids and rows: one buffer each per layer set, so that the
    # gather timed alone over the rotating sets reads each set's own rows and
    # writes its own output (cold in L2, as in a step)
    shared = {"kv": torch.empty((T, 2 * C), dtype=torch.bfloat16, device=device),
              "y": torch.empty((T, C), dtype=torch.bfloat16, device=device),
              "gate": torch.empty((T,), dtype=torch.float32, device=device),
              "ctx_out": torch.empty((w.num_reqs, w.ctx_len), dtype=torch.int32, device=device),
              "st_out": torch.empty_like(sets[0]["conv_state"]) if w.decode else None}
    bufs = [dict(shared, ids=torch.empty((T, H), dtype=torch.int64, device=device),
                 emb=torch.empty((T, w.emb_dim), dtype=torch.bfloat16, device=device))
            for _ in range(num_sets)]
    ids, emb, ctx_out, st_out = (bufs[0][k] for k in ("ids", "emb", "ctx_out", "st_out"))
    err = torch.zeros(1, dtype=torch.int32, device=device)
    stream = torch.cuda.current_stream(device)
    order_ws = None
    if w.table_loc == "host":  # a host table is gathered in table order
        order_ws = torch.empty((_lib.ple_lookup_ordered_workspace(
            T, H, sets[0]["table"], sets[0]["row_scale"]),), dtype=torch.uint8, device=device)

    def gather(p, b, st):
        if order_ws is not None:
            _lib.ple_lookup_ordered(b["ids"], p["table"], b["emb"], order_ws,
                                    row_scale=p["row_scale"], dev_err=err, stream=st)
        else:
            _lib.ple_lookup(b["ids"], p["table"], b["emb"], row_scale=p["row_scale"], dev_err=err,
                            stream=st)

    def stages_of(s, st):
        """The step's libple calls for layer set s, one callable per kernel."""
        p = sets[s % num_sets]
        b = bufs[s % num_sets]
        ids, emb, kv, y, gate = (b[k] for k in ("ids", "emb", "kv", "y", "gate"))
        st_out = b["st_out"]
        ctx_o = b["ctx_out"] if w.decode else None
        stages = []
        if fuse_ids:
            stages.append(lambda: _lib.ple_ngram_lookup(
                p["input_ids"], p["qsl"], p["ctx"], p["mult"], p["host"]["V"], p["host"]["O"],
                w.eos_token_id, w.heads_per_ngram, p["table"], emb, row_scale=p["row_scale"],
                ids_out=ids, ngram_context_out=ctx_o, dev_err=err, stream=st))
        else:
            stages.append(lambda: _lib.ple_ngram_ids(
                p["input_ids"], p["qsl"], p["ctx"], p["mult"], p["host"]["V"], p["host"]["O"],
                w.eos_token_id, w.heads_per_ngram, ids, ctx_o, err, st))
            stages.append(lambda: gather(p, b, st))
        if fuse:
            stages.append(lambda: _lib.ple_kv_proj_gate(
                emb, p["w_kv"], p["hidden"], p["gamma_h"], p["gamma_k"], kv, gate, gate_ws,
                dev_err=err, stream=st))
            stages.append(lambda: _lib.ple_gated_conv(
                kv, gate, p["qsl"], p["conv_w"], w.dilation, y, conv_state=p.get("conv_state"),
                conv_state_out=st_out, dev_err=err, stream=st))
        else:
            stages.append(lambda: _lib.ple_kv_proj(emb, p["w_kv"], kv, dev_err=err, stream=st))
            stages.append(lambda: _lib.ple_gate_conv(
                p["hidden"], kv, p["gamma_h"], p["gamma_k"], p["qsl"], p["conv_w"], w.dilation, y,
                conv_state=p.get("conv_state"), conv_state_out=st_out, gate_out=gate, dev_err=err,
                stream=st))
        return stages

    def step(s, ev=None, st=None):
        st = stream if st is None else st
        stages = stages_of(s, st)
        if ev is not None:
            ev[0].record(st)
        for j, run in enumerate(stages):
            run()
            if ev is not None:
                ev[j + 1].record(st)

    for i in range(max(args.warmup, num_sets)):  # every set's buffers hold its step's results
        step(i)
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise RuntimeError(f"{name}: device error word {int(err.item())} during warm-up")

    # ---- eager steps with events between the kernels (per-kernel times) ----
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(len(KERNELS) + 1)]
              for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    for i in range(args.steps):
        step(i, events[i])
    torch.cuda.synchronize()
    barrier()
    eager_ms = events[0][0].elapsed_time(events[-1][-1])
    per_kernel = {k: [] for k in KERNELS}
    for ev in events:
        for j, k in enumerate(KERNELS):
            per_kernel[k].append(ev[j].elapsed_time(ev[j + 1]))
    eager_ms = max_over_ranks(eager_ms, device)
    if int(err.item()) != 0:
        raise RuntimeError(f"{name}: device error word {int(err.item())} in the timed region")

    # ---- timed region: K steps replayed from CUDA graphs (one per layer
    # set, captured once), device events on the replay stream ----
    graphs, graph_error = capture_graphs(torch, step, num_sets, device)
    if graphs is not None:
        for i in range(max(args.warmup, len(graphs))):
            graphs[i % len(graphs)].replay()
        torch.cuda.synchronize()
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        replay = torch.cuda.current_stream(device)
        barrier()
        torch.cuda.synchronize()
        g0.record(replay)
        for i in range(args.steps):
            graphs[i % num_sets].replay()
        g1.record(replay)
        torch.cuda.synchronize()
        barrier()
        total_ms = max_over_ranks(g0.elapsed_time(g1), device)
        if int(err.item()) != 0:
            raise RuntimeError(f"{name}: device error word {int(err.item())} in the graph replays")
        mode = "cuda_graph"
    else:
        total_ms, mode = eager_ms, "eager"
    del graphs

    # ---- each kernel alone (after the timed region, so that its extra GPU
    # work does not warm the board before it): K back-to-back launches over
    # the rotating layer sets between two events on the launching stream, so that a short
    # kernel's launch latency overlaps the previous launch (the events
    # between the kernels of the eager steps above add it to every kernel);
    # the per-launch average is the kernel's duration for the roofline ----
    # (the K launches are replayed from one CUDA graph, so that the host's
    # submission rate does not bound the short kernels)
    alone = {}
    for j, k in enumerate(KERNELS):
        def launches(st, j=j):
            for i in range(args.steps):
                stages_of(i, st)[j]()
        g_alone, why = capture_graphs(torch, lambda s, st=None: launches(st), 1, device)
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        if g_alone is not None:
            g_alone[0].replay()
            torch.cuda.synchronize()
            a0.record(stream)
            g_alone[0].replay()
            a1.record(stream)
        else:
            launches(stream)
            torch.cuda.synchronize()
            a0.record(stream)
            launches(stream)
            a1.record(stream)
        torch.cuda.synchronize()
        alone[k] = a0.elapsed_time(a1) / args.steps
        del g_alone
    if int(err.item()) != 0:
        raise RuntimeError(f"{name}: device error word {int(err.item())} in the per-kernel timing")

    # ---- end to end through PLEHostPipeline with pinned host buffers ----
    # Every step uploads its inputs (token ids, query_start_loc, hidden) from
    # pinned host memory and reads y back into pinned host memory; uploads,
    # compute (each slot's layer calls replayed from a CUDA graph) and
    # read-backs of neighbouring steps overlap on three streams.
    from hashed_gram_embedding_gb300 import PLEHostPipeline
    p0 = sets[0]
    layer = PLELayer(p0["table"], p0["row_scale"], p0["mult"], p0["host"]["V"], p0["host"]["O"],
                     w.eos_token_id, w.heads_per_ngram, p0["w_kv"], p0["gamma_h"], p0["gamma_k"],
                     p0["conv_w"], w.dilation, fuse_gate=fuse, fuse_ids=fuse_ids)
    depth = args.e2e_depth
    pipe = PLEHostPipeline(layer, T, w.num_reqs, device, depth=depth)
    h_ids = torch.from_numpy(p0["host"]["input_ids"]).pin_memory()
    h_qsl = torch.from_numpy(p0["host"]["query_start_loc"]).pin_memory()
    h_hidden = p0["hidden"].cpu().pin_memory()
    h_ys = [torch.empty((T, C), dtype=torch.bfloat16).pin_memory() for _ in range(depth)]
    h2d = h_ids.numel() * 4 + h_qsl.numel() * 4 + h_hidden.numel() * 2
    d2h = h_ys[0].numel() * 2
    fwd = dict(ngram_context=p0["ctx"], ngram_context_out=ctx_out if w.decode else None,
               conv_state=p0.get("conv_state"), conv_state_out=st_out, dev_err=err)

    # warm-up: every slot runs once directly, then is captured into its graph
    for i in range(max(min(args.warmup, 3), 2 * depth)):
        pipe.submit(h_ids, h_qsl, h_hidden, h_ys[i % depth], **fwd)
    pipe.synchronize()
    torch.cuda.synchronize()
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    # at least E2E_MIN_STEPS steps: one hiccup of the host thread (scheduling,
    # a page fault) moves a 20-step region of 8 ms by tens of percent
    e2e_steps = max(args.steps, E2E_MIN_STEPS)
    e_start.record(pipe.copy_in)
    for i in range(e2e_steps):
        pipe.submit(h_ids, h_qsl, h_hidden, h_ys[i % depth], **fwd)
    e_end.record(pipe.copy_out)
    torch.cuda.synchronize()
    barrier()
    e2e_ms = max_over_ranks(e_start.elapsed_time(e_end), device)
    pipe.close()
    del pipe, layer

    extra = {}
    if rank == 0 and w.table_loc == "host":
        extra["overlap"] = uva_overlap(torch, _lib, sets[0], ids, emb, w, device, order_ws)
    if rank == 0 and w.name == "prefill8k" and w.table_loc == "hbm" and not args.vocab_start:
        extra["sharded"] = sharded_timing(torch, _lib, w, sets[0], bufs[0]["ids"], device)
    chain_layers = args.chain_layers or (w.num_layers if w.num_layers > 1 else 0)
    if chain_layers > 1:
        extra["chain"] = chain_timing(torch, w, sets, device, err, fuse, chain_layers)
    if rank != 0:
        return None
    peaks, peak_kind = load_peaks()
    link_gbs = measure_link_gbs(torch, device) if w.table_loc == "host" else None
    work = algorithmic_work(w)
    kernels = {}
    step_kernels_ms = float(np.mean([sum(per_kernel[x][i] for x in KERNELS)
                                     for i in range(args.steps)]))
    alone_total = sum(alone[x] for x in KERNELS)
    # a tensor-bound kernel whose alone loop ran for a second or more ran under
    # the power cap: its denominator is the sustained bf16 rate, else the burst
    def tensor_peak(avg_ms):
        sustained = args.steps * avg_ms >= 1000.0
        return (peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"],
                "bf16 sustained: the kernel's timed loop ran %.1f s" % (args.steps * avg_ms / 1e3)
                if sustained else "bf16 burst")
    for k in KERNELS:
        avg_ms = alone[k]
        bound, amount = work[k]
        if bound == "tensor":
            achieved = amount / (avg_ms * 1e-3) / 1e12
            peak = tensor_peak(avg_ms)[0]
            unit = "TFLOP/s"
        elif bound == "link":  # rows read over the host link
            achieved = amount / (avg_ms * 1e-3) / 1e9
            peak = link_gbs
            unit = "GB/s"
        else:
            achieved = amount / (avg_ms * 1e-3) / 1e9
            peak = peaks["hbm_gbs"]
            unit = "GB/s"
        in_step_ms = float(np.mean(per_kernel[k]))
        kernels[k] = {"us": round(avg_ms * 1e3, 2), "bound": bound, "achieved": round(achieved, 1),
                      "unit": unit, "peak": round(peak, 1), "frac": round(achieved / peak, 4),
                      "us_in_step": round(in_step_ms * 1e3, 2),
                      "share": round(avg_ms / alone_total, 4),
                      "share_in_step": round(in_step_ms / step_kernels_ms, 4)}
    dominant = max(KERNELS, key=lambda k: kernels[k]["us"])
    dk = kernels[dominant]
    bound, amount = work[dominant]
    traffic = None if args.vocab_start else ncu_traffic(
        dominant, w.name, "link_bytes_per_launch" if dk["bound"] == "link" else
        "dram_bytes_per_launch")
    dpeak = {"tensor": tensor_peak(alone[dominant])[0],
             "link": link_gbs}.get(dk["bound"], peaks["hbm_gbs"])
    roofline = {"bound": dk["bound"], "kernel": dominant, "achieved": dk["achieved"],
                "peak": dpeak, "unit": dk["unit"], "frac": dk["frac"],
                "peak_source": ("pinned host-to-device copy measured in this run"
                                if dk["bound"] == "link" else
                                f"{peak_kind} ({tensor_peak(alone[dominant])[1] if dk['bound'] == 'tensor' else 'HBM copy'})"),
                "algorithmic_per_launch": amount, "traffic": traffic,
                "traffic_counters": ("syslts__t_sectors_aperture_sysmem_op_read x 32 B"
                                     if dk["bound"] == "link" else
                                     "dram__bytes_read + dram__bytes_write")}
    gk = "lookup" if not fuse_ids else "ngram_lookup"
    if w.table_loc == "host":
        gather_line = {"kernel": gk, "gbs": kernels[gk]["achieved"], "link_gbs": link_gbs,
                       "frac_link": kernels[gk]["frac"],
                       "pcie5_x16_nominal_gbs": PCIE5_X16_GBS,
                       "frac_pcie5_x16_nominal": round(kernels[gk]["achieved"] / PCIE5_X16_GBS, 3)}
    else:
        gather_line = {"kernel": gk, "gbs": kernels[gk]["achieved"], "frac_hbm": kernels[gk]["frac"],
                       "note": ("algorithmic bytes; Zipf tokens hit L2 for repeated rows"
                                if w.token_dist == "zipf" else "algorithmic bytes")}
    value = world * args.steps * T / (total_ms * 1e-3)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded workload recipe; no dataset)",
        "config": {"workload": w.name, "mode": mode, "num_tokens": T, "num_reqs": w.num_reqs,
                   "heads": H, "head_dim": w.head_dim,
                   "table_rows": int(sets[0]["table"].shape[0]), "table_loc": w.table_loc,
                   "table_dtype": ("fp8 e4m3 + float32 row scale" if w.table_dtype == "fp8"
                                   else "bf16"),
                   "hidden": C, "conv_kernel": w.conv_k, "dilation": w.dilation,
                   "layers": w.num_layers, "fuse_gate": fuse, "fuse_ids": fuse_ids,
                   "layer_sets": num_sets,
                   "l2": f"inputs rotate over {num_sets} layer sets (> 129 MB L2 per rotation); no flush",
                   "parallelism": "replicas" if world > 1 else "single"},
        "roofline": roofline,
        "kernels": kernels,
        "gather": gather_line,
        "e2e": {"value": round(world * e2e_steps * T / (e2e_ms * 1e-3), 1), "unit": UNIT,
                "steps": e2e_steps,
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "pipeline_depth": depth},
        "gpu_launches": launches_per_step(w, fuse, fuse_ids) * args.steps,
    }
    line.update(extra)
    line["eager"] = {"ms_per_step": round(eager_ms / args.steps, 4),
                     "value": round(world * args.steps * T / (eager_ms * 1e-3), 1),
                     "note": "same steps launched one by one, events between kernels "
                             "(kernels.*.us_in_step, share_in_step: these also time the host's "
                             "submission); kernels.*.us and share: each kernel alone, "
                             f"{args.steps} back-to-back launches over the rotating layer sets"}
    if graph_error:
        line["eager"]["graph_capture_error"] = graph_error
    if headline and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, sets[0], budget_s=args.cpu_seconds)
    return line


def launches_per_step(w, fuse, fuse_ids):
    """libple kernels one step launches: the n-gram lookup (1; or ids and
    gather, 2; a host table's ordered gather adds its count, scan and scatter
    kernels), then the fused projection and the gated conv (2), or the
    projection and the gate and conv passes (3)."""
    embed = 1 if fuse_ids else 2 + (3 if w.table_loc == "host" else 0)
    return embed + (2 if fuse else 3)


def capture_graphs(torch, step, num_sets, device):
    """Each layer set's step captured once into a CUDA graph (the libple calls
    on a capture stream); (graphs, None), or (None, reason) if capture fails."""
    try:
        capture = torch.cuda.Stream(device)
        capture.wait_stream(torch.cuda.current_stream(device))
        graphs = []
        for s in range(num_sets):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=capture):
                step(s, st=capture)
            graphs.append(g)
        torch.cuda.synchronize()
        return graphs, None
    except Exception as e:  # report it; the eager timing then stands
        torch.cuda.synchronize()
        return None, str(e)[:300]


def chain_timing(torch, w, sets, device, err, fuse, L, reps=10):
    """L layers over the same tokens through PLEChain: with the next layers'
    ids and gathers prefetched on a side stream, and in line. Layer i uses
    layer set i; past the resident sets (one 32 GiB table for the host-table
    workload) layer i reuses set i mod sets' table and weights with its own
    layer multipliers, so each layer gathers its own rows."""
    from hashed_gram_embedding_gb300 import PLELayer, PLEChain
    from hashed_gram_embedding_gb300 import workloads as wl
    layers = []
    for i in range(L):
        p = sets[i % len(sets)]
        mult = p["mult"] if i < len(sets) else wl.layer_multipliers(w, i)
        layers.append(PLELayer(p["table"], p["row_scale"], mult, p["host"]["V"], p["host"]["O"],
                               w.eos_token_id, w.heads_per_ngram, p["w_kv"], p["gamma_h"],
                               p["gamma_k"], p["conv_w"], w.dilation, fuse_gate=fuse))
    p0 = sets[0]
    T, C = w.num_tokens, w.hidden
    hiddens = [sets[i % len(sets)]["hidden"] for i in range(L)]
    outs = [torch.empty((T, C), dtype=torch.bfloat16, device=device) for _ in range(L)]
    stream = torch.cuda.current_stream(device)
    res = {"layers": L}
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    variants = [("prefetch", True, None), ("prefetch_full_grid", True, 0),
                ("inline", False, 0)]
    if w.table_loc == "host":  # the pages cap the side-stream gather at half the SMs
        variants.insert(1, ("prefetch_half_grid", True, sms // 2))

    def timed(run):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(reps):
            run()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    for name, prefetch, ctas in variants:
        chain = PLEChain(layers, prefetch=prefetch, prefetch_ctas=ctas)

        def fwd(st=stream, chain=chain):
            chain.forward(p0["input_ids"], p0["qsl"], hiddens, outs, ngram_context=p0["ctx"],
                          dev_err=err, stream=st)
        for _ in range(2):
            fwd()
        ms = timed(fwd)
        res[f"{name}_ms"] = round(ms, 4)
        res[f"{name}_tokens_per_s_per_layer"] = round(T * L / (ms * 1e-3), 1)
        # the same chain captured once into a CUDA graph (side stream forked
        # and joined inside the capture) and replayed
        graphs, why = capture_graphs(torch, lambda s, st=None: fwd(st), 1, device)
        if graphs is not None:
            graphs[0].replay()
            gms = timed(graphs[0].replay)
            res[f"{name}_graph_ms"] = round(gms, 4)
            res[f"{name}_graph_tokens_per_s_per_layer"] = round(T * L / (gms * 1e-3), 1)
            del graphs
        else:
            res[f"{name}_graph_error"] = why
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item())} in the chain timing")
    return res


def measure_link_gbs(torch, device, nbytes=512 << 20, reps=5):
    """Host-to-device copy rate from pinned memory (the host link's usable
    peak, the denominator of a gather from a host table)."""
    src = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    dst = torch.empty(nbytes, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    dst.copy_(src, non_blocking=True)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        dst.copy_(src, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    return round(nbytes * reps / (e0.elapsed_time(e1) * 1e-3) / 1e9, 1)


def sharded_timing(torch, _lib, w, p, ids, device, tp=2, dp=2, reps=20):
    """The per-rank kernels of a sharded lookup, for a tp x dp group emulated
    on this GPU over the workload's table and ids (the step's tokens split
    into dp replicas): each rank's head-shard gather (its H / (tp dp) heads
    for every gathered token) and the select of one replica's window; and for
    a row-sharded table, one rank's raw-row gather (its row range, zeros
    elsewhere) and the select. Collectives are not timed (one GPU). Checks
    that the emulated group rebuilds the plain lookup's rows bit for bit."""
    from hashed_gram_embedding_gb300 import sharded
    T, H, D = w.num_tokens, w.num_heads, w.head_dim
    G = tp * dp
    table = p["table"]
    V, O = p["host"]["V"], p["host"]["O"]
    stream = torch.cuda.current_stream(device)

    def timed(fn):
        """us per call of fn: reps calls replayed from one CUDA graph (so that
        the host's submission does not bound these short kernels)."""
        fn()
        torch.cuda.synchronize()
        graphs, _ = capture_graphs(torch, lambda s_, st=None: [fn() for _ in range(reps)], 1,
                                   device)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        if graphs is not None:
            graphs[0].replay()
            torch.cuda.synchronize()
            e0.record(stream)
            graphs[0].replay()
            e1.record(stream)
        else:
            e0.record(stream)
            for _ in range(reps):
                fn()
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps * 1e3  # us

    slot = T // dp
    heads = {}
    for r in range(G):
        d, t = divmod(r, tp)
        _, hb, n = sharded.head_shard(H, tp, t, dp, d)
        r0, r1 = sharded.head_rows(V, O, hb, n)
        heads[r] = sharded.HeadShardedLookup(table[r0:r1], None, V, O, tp, t, dp, d)
    rows_out = torch.stack([heads[r].gather(ids) for r in range(G)])
    out = heads[0].select(rows_out, slot, slot)
    ref = torch.empty((T, H * D), dtype=torch.bfloat16, device=device)
    _lib.ple_lookup(ids, table, ref)
    ok_heads = bool(torch.equal(out.view(torch.int16), ref[:slot].view(torch.int16)))
    hs = heads[G - 1]
    g_us = timed(lambda: hs.gather(ids))
    s_us = timed(lambda: heads[0].select(rows_out, slot, slot, out=out))
    # row shards of the same table
    r0, r1 = sharded.row_shard(table.shape[0], G, 1)
    rl = sharded.RowShardedLookup(table[r0:r1], None, r0, H, dp, 0)
    raw, _ = rl.gather(ids)
    rg_us = timed(lambda: rl.gather(ids))
    rs_us = timed(lambda: rl.select(raw, None, slot, slot, out=out))
    n = H // G
    peak = load_peaks()[0]["hbm_gbs"]
    # bytes: head shard: T x n ids read, T x n rows read + written; select: slot x H rows
    # read + written; row shard: T x H ids, the owned rows read (~1/G), T x H rows written
    gb = {"head_gather": T * n * (8 + 2 * D * 2), "select": slot * H * D * 2 * 2,
          "row_gather": T * H * (8 + D * 2) + T * H * D * 2 // G}
    us = {"head_gather": g_us, "select": s_us, "row_gather": rg_us, "row_select": rs_us}
    gb["row_select"] = gb["select"]
    res = {"group": f"tp{tp} x dp{dp} emulated on one GPU (collectives not timed)",
           "tokens": T, "heads_per_shard": n, "rows_equal_plain_lookup": ok_heads}
    for k, v in us.items():
        ach = gb[k] / (v * 1e-6) / 1e9
        res[k] = {"us": round(v, 2), "gbs": round(ach, 1), "frac_hbm": round(ach / peak, 4)}
    return res


def uva_overlap(torch, _lib, p, ids, emb, w, device, order_ws, reps=10):
    """The pinned-host gather (in table order) prefetched on a side stream
    (half the SMs) while a 4096^3 bf16 GEMM -- a stand-in for the previous
    layer, run by cuBLAS through torch -- occupies the main stream: each
    alone, then both. Gather times come from events on the side stream,
    totals from events on the main stream, which joins the side stream at
    the end."""
    main = torch.cuda.current_stream(device)
    side = torch.cuda.Stream(device)
    half = max(1, torch.cuda.get_device_properties(device).multi_processor_count // 2)
    a = torch.randn((4096, 4096), device=device, dtype=torch.bfloat16)
    b = torch.randn((4096, 4096), device=device, dtype=torch.bfloat16)
    c = torch.empty((4096, 4096), device=device, dtype=torch.bfloat16)

    def run(with_gather, with_gemm, ordered=True):
        g_us, t_us = [], []
        for rep in range(reps + 2):
            torch.cuda.synchronize()
            s0, s1, m0, m1 = (torch.cuda.Event(enable_timing=True) for _ in range(4))
            m0.record(main)
            side.wait_stream(main)
            s0.record(side)
            if with_gather:
                if ordered:
                    _lib.ple_lookup_ordered(ids, p["table"], emb, order_ws, max_ctas=half,
                                            stream=side)
                else:
                    _lib.ple_lookup(ids, p["table"], emb, max_ctas=half, stream=side)
            s1.record(side)
            if with_gemm:
                torch.matmul(a, b, out=c)
            main.wait_stream(side)
            m1.record(main)
            torch.cuda.synchronize()
            if rep >= 2:
                g_us.append(s0.elapsed_time(s1) * 1e3)
                t_us.append(m0.elapsed_time(m1) * 1e3)
        return float(np.mean(g_us)), float(np.mean(t_us))

    g_alone, _ = run(True, False)
    _, m_alone = run(False, True)
    g_over, t_over = run(True, True)
    u_alone, _ = run(True, False, ordered=False)
    row_bytes = w.num_tokens * w.num_heads * w.head_dim * 2
    return {"gather_alone_us": round(g_alone, 1), "gemm_alone_us": round(m_alone, 1),
            "overlapped_total_us": round(t_over, 1), "overlapped_gather_us": round(g_over, 1),
            "saved_us": round(g_alone + m_alone - t_over, 1),
            "hidden_fraction": round((g_alone + m_alone - t_over) / min(g_alone, m_alone), 3),
            "gather_link_gbs": round(row_bytes / (g_alone * 1e-6) / 1e9, 1),
            "gather_unordered_alone_us": round(u_alone, 1),
            "gather_ctas": half, "gemm": "4096x4096x4096 bf16 (cuBLAS via torch.matmul)"}


# ---------------------------------------------------------------------------
# the oracle on the host cores (cpu_baseline leg and the reference arm)
# ---------------------------------------------------------------------------

def oracle_sample(w, p, req_range, max_tokens, bits):
    """Time the oracle over requests req_range (truncated to max_tokens tokens)."""
    import torch
    import oracle

    host = p["host"]
    qsl = host["query_start_loc"]
    r0, r1 = req_range
    start, end = int(qsl[r0]), int(min(qsl[r1], qsl[r0] + max_tokens))
    sub_qsl = [q - start for q in qsl[r0:r1 + 1]]
    sub_qsl = [min(q, end - start) for q in sub_qsl]
    tokens = host["input_ids"][start:end]
    ctx = None if host["ngram_context"] is None else host["ngram_context"][r0:r1]
    t = {}
    t0 = time.perf_counter()
    ids, _ = oracle.ngram_ids(tokens, sub_qsl, ctx, p["mult"], host["V"], host["O"],
                              w.eos_token_id, w.heads_per_ngram)
    t["ngram_ids"] = time.perf_counter() - t0
    ids = np.asarray(ids, dtype=np.int64).reshape(len(tokens), -1)
    # input staging, not timed: the rows the sample names, as a compact table
    uniq, inv = np.unique(ids, return_inverse=True)
    rows = p["table"][torch.from_numpy(uniq).to(p["table"].device)]
    hidden = bits(p["hidden"][start:end])
    w_kv, gh, gk, cw = (bits(p[k]) for k in ("w_kv", "gamma_h", "gamma_k", "conv_w"))
    t0 = time.perf_counter()
    if p["row_scale"] is None:
        emb = oracle.lookup_bf16(inv.reshape(ids.shape), bits(rows))
    else:
        scale = p["row_scale"][torch.from_numpy(uniq).to(p["row_scale"].device)].cpu().numpy()
        emb = oracle.lookup_fp8(inv.reshape(ids.shape), rows.cpu().numpy(), scale)
    t["lookup"] = time.perf_counter() - t0
    t0 = time.perf_counter()
    kv = oracle.kv_proj(emb, w_kv)
    t["kv_proj"] = time.perf_counter() - t0
    state = None if p.get("conv_state") is None else bits(p["conv_state"][r0:r1])
    t0 = time.perf_counter()
    oracle.gate_conv(hidden, kv, gh, gk, 1e-6, sub_qsl, cw, w.dilation, state)
    t["gate_conv"] = time.perf_counter() - t0
    return len(tokens), t


def _bits(t):
    import torch
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def cpu_baseline(w, p, budget_s=15.0):
    """The oracle as it stands on this host, over whole requests until the
    time budget is spent (at least one request)."""
    qsl = p["host"]["query_start_loc"]
    tokens = 0
    stages = {k: 0.0 for k in ORACLE_STAGES}
    r = 0
    while r < len(qsl) - 1:
        n, t = oracle_sample(w, p, (r, r + 1), 1 << 30, _bits)
        tokens += n
        for k in ORACLE_STAGES:
            stages[k] += t[k]
        r += 1
        if sum(stages.values()) > budget_s:
            break
    total = sum(stages.values())
    return {"value": round(tokens / total, 2), "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
            "sample": f"requests 0..{r - 1} of {w.name} ({tokens} of {w.num_tokens} tokens), "
                      f"float64 NumPy / Python-int oracle, inputs staged outside the timed region",
            "stage_seconds": {k: round(v, 3) for k, v in stages.items()}}


def run_reference(args):
    """The reference arm: the oracle timed on the host cores, rank 0 only."""
    import torch
    from hashed_gram_embedding_gb300 import workloads as wl

    rank, world, local_rank = dist_env()
    if rank != 0:
        return None
    device = torch.device("cuda", local_rank) if torch.cuda.is_available() else torch.device("cpu")
    w = wl.WORKLOADS[HEADLINE if args.workload == "all" else args.workload]
    p = make_sets(torch, w, device, 1)[0]
    qsl = p["host"]["query_start_loc"]
    max_tokens = args.ref_tokens
    times = []
    toks = []
    for i in range(args.warmup + args.steps):
        r = i % (len(qsl) - 1)
        n, t = oracle_sample(w, p, (r, r + 1), max_tokens, _bits)
        if i >= args.warmup:
            times.append(sum(t.values()))
            toks.append(n)
    total_s = sum(times)
    value = sum(toks) / total_s
    sample = (f"per step one request of {w.name} truncated to {max_tokens} tokens "
              f"({int(np.mean(toks))} tokens on average)")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(total_s * 1e3 / args.steps, 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded workload recipe; no dataset)",
            "config": {"workload": w.name, "num_tokens": w.num_tokens, "num_reqs": w.num_reqs,
                       "parallelism": "single"},
            "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": cpu_cores(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="all",
                    help="all (default: the fp8x8 headline, then every other workload under "
                         "\"configs\") or one of " + ", ".join(ALL_WORKLOADS))
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-tokens", type=int, default=256)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--chain-layers", type=int, default=0,
                    help="also time a chain of this many layers through PLEChain (prefetch vs "
                         "in line; 0 = the workload's layer count when it has several)")
    ap.add_argument("--fuse-ids", choices=["auto", "on", "off"], default="auto",
                    help="ple_ngram_lookup (ids hashed in the gather) for HBM tables: auto = as "
                         "PLELayer chooses (steps of up to 4096 tokens)")
    ap.add_argument("--no-fuse-gate", action="store_true",
                    help="time ple_kv_proj + ple_gate_conv instead of the fused projection")
    ap.add_argument("--layer-sets", type=int, default=0,
                    help="layer parameter sets to rotate over (0 = workload default)")
    ap.add_argument("--e2e-depth", type=int, default=3,
                    help="device buffer sets rotating in the end-to-end pipeline")
    ap.add_argument("--vocab-start", type=int, default=0,
                    help="first per-head vocab prime (smaller table for profiling cases)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    line = run_reference(args) if args.impl == "reference" else run_ours(args)
    if line is not None:
        print(json.dumps(line), flush=True)
    try:
        import torch.distributed as dist
        if dist.is_initialized():
            dist.destroy_process_group()
    except Exception:
        pass


if __name__ == "__main__":
    main()
