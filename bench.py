"""Benchmark: calibrated E4M3 paged decode attention on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload decode|decode32k|long|verify|mixed|prefill]
                    [--no-cpu-baseline] [--no-fp16] [--no-workloads]

One step = one pass of the whole hot path over one batch, for every layer
of the workload: quantise-on-append of the step's new K/V tokens into the
layer's page-4 cache, split-K decode / verify attention over it, and the
log-sum-exp combine.  Inputs are seeded synthetic tensors (see
fp8_paged_kv_e4m3_gb300.inputs).  The headline workload is batch 32 x 4096
context, 32 query / 4 kv heads, head_dim 128, q_len 1, split-K 4, one layer.

Reported (one JSON line on rank 0): achieved HBM GB/s of algorithmic bytes
per step (KV bytes read + Q + output + block tables + append traffic; the
FP32 split workspace is not counted), its fraction of the measured HBM
peak, sequence-steps/s, and the same for the fp16-KV arm with the
fp16/E4M3 step-time ratio.  L2 is defeated by rotating through copies of
the KV pools whose total exceeds twice the L2 size (the 24-layer steps move
far more than that by themselves).  Without --workload, the line also
carries a "workloads" object with the same figures for decode at 32K
context, the long-context batch, the 24-layer MTP3 verify step, the
24-layer mixed step and the chunked-prefill call.

N > 1 (torchrun): every rank runs an independent replica on its own GPU
with its own seeded batch (the path shards by sequence with no exchange),
timing is max-over-ranks, and the value is the aggregate.

--impl reference: the CPU oracle (the only other implementation of the
method here) timed on this host's cores on the step's (sequence, kv head)
units, printed in the same format with "impl": "reference".
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "E4M3 paged decode-attn achieved HBM GB/s (% of peak) and seq-steps/s vs FP16"
L2_BYTES_DEFAULT = 129 * 1024 * 1024
GRAPH_STEPS = 10   # steps captured in one CUDA graph


# source files each attention kernel is compiled from (for the profile hash)
KERNEL_SOURCES = {
    "prefill_attn_kernel": ["kvq_prefill.cu", "kvq_tcgen05.cuh", "kvq_device.cuh"],
    "attn_split_kernel": ["kvq_attn_kernel.cuh", "kvq_merge.cuh", "kvq_device.cuh"],
    "attn_tc_kernel": ["kvq_attn_tc.cu", "kvq_attn_kernel.cuh", "kvq_merge.cuh", "kvq_tcgen05.cuh", "kvq_device.cuh"],
}


def kernel_source_hash(kernel: str) -> str:
    """sha256 over the kernel's source files, in the listed order."""
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        h.update(open(os.path.join(ROOT, "fp8_paged_kv_e4m3_gb300", "csrc", f), "rb").read())
    return h.hexdigest()


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of the attention kernel from the committed ncu
    summary profiles/<kernel>_<workload>.md, or None when that summary was
    taken on other kernel source."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    try:
        text = open(path).read()
        digest = kernel_source_hash(kernel)
    except OSError:
        return None
    fields = dict(line.strip("- ").split(": ", 1) for line in text.splitlines()
                  if line.startswith("- ") and ": " in line)
    if fields.get("kernel_source_sha256") != digest:
        return None
    try:
        return int(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def _tensor_peak():
    """Dense fp16 tensor peak in TFLOP/s: the measured bf16 burst figure (fp16
    runs at the bf16 rate), else the recipe's fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            v = float(json.load(f)["bf16_tflops"])
        if v > 0:
            return v, "measured (bf16 dense burst; fp16 at the same rate)"
    except (OSError, KeyError, ValueError):
        pass
    return 1900.0, "fallback"


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ---------------------------------------------------------------------------
# workload accounting

def algorithmic_bytes(w, kv_elem_bytes: int, lens, topk=(None, None)):
    """Bytes the step must move at minimum: every K and V element attended
    once (all cached tokens of a dense sequence; the listed tokens of a top-k
    sequence, plus its list and block-table entries), Q, the output, the
    block-table entries of the pages read, the context lengths, and the
    append of the step's B * q_len tokens and of a prefill chunk (fp16 in,
    cache dtype out, slot ids).  "attention_kernel" is the split attention
    kernel's share."""
    Hkv, D = w.num_kv_heads, w.head_dim
    lens = np.asarray(lens, np.int64)
    ti, tl = topk
    dense = np.ones(lens.shape, bool) if tl is None else (np.asarray(tl) == 0)
    tokens = int(lens[dense].sum())
    pages = int(((lens[dense] + 3) // 4).sum())
    kv = 2 * tokens * Hkv * D * kv_elem_bytes
    listed = 0 if tl is None else int(np.asarray(tl)[~dense].sum())     # per kv head
    kv += 2 * listed * Hkv * D * kv_elem_bytes
    lists = listed * Hkv * 4 * 2
    q = w.batch * w.q_len * w.num_q_heads * D * 2
    out = q
    bt = pages * 4 + w.batch * 4
    appended = w.batch * w.q_len + w.prefill_chunk
    append = appended * (Hkv * D * 2 * (2 + kv_elem_bytes) + 4)
    attn = kv + q + bt + lists
    return {"step": attn + out + append, "attention_kernel": attn}


def describe(w, splits) -> str:
    kind, *rest = w.lens.split(":")
    ctx = {"fixed": lambda: f"{rest[0]} context", "list": lambda: f"contexts {rest[0]}",
           "loguniform": lambda: f"contexts log-uniform {rest[0]}-{rest[1]}",
           "uniform": lambda: f"contexts uniform {rest[0]}-{rest[1]}"}[kind]()
    extra = ""
    if w.topk:
        extra += f", {int(round(w.topk_fraction * 100))}% of sequences over top-{w.topk} lists"
    if w.prefill_chunk:
        extra += f", {w.prefill_chunk}-token prefill chunk appended"
    split = f"split-K {splits}" + (f" of {w.split_pages} pages" if w.split_pages else "")
    if not w.lens.startswith("fixed"):
        split += ", longest first"
    layers = "one layer" if w.layers <= 1 else f"{w.layers} layers per step, each with its own pools and scales"
    return (f"{w.name}: batch {w.batch}, {ctx}, {w.num_q_heads} q / {w.num_kv_heads} kv heads, "
            f"head_dim {w.head_dim}, q_len {w.q_len}, {split}, page 4{extra}; {layers}")


# ---------------------------------------------------------------------------
# clocks sampled while timing

class ClockSampler:
    """nvidia-smi samples (SM clock, its maximum, throttle reasons) every 100 ms
    while the timed region runs.  The raw samples go to KVQ_CLOCKS_DIR when
    that is set (kept), else to a temporary file (removed after the summary)."""

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.keep = bool(os.environ.get("KVQ_CLOCKS_DIR"))
        base = os.environ.get("KVQ_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(base, f"kvq_clocks_{os.getpid()}_{id(self)}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx),
                 "--query-gpu=clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                 "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                 "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()
        return False

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        rows = []
        with open(self.path) as fh:
            lines = fh.readlines()
        if not self.keep:
            os.remove(self.path)
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[4:8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, flags in rows for i, f in enumerate(flags)
                          if f.lower() in ("active", "1", "0x1")})
        under = [r[0] for r in rows]
        return {"sm_mhz": statistics.median(under), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# the GPU arm

class Arm:
    """One arm (E4M3 or fp16 KV) of the step, with rotating pool copies.

    A workload of several layers (the 24-layer verify and mixed batches)
    gives every layer its own seeded K/V, queries, calibrated scales and
    pools; the block tables, context lengths and top-k lists are shared, as
    every layer of one model attends the same sequences.  A step runs the
    append, attention and combine of every layer in turn."""

    def __init__(self, w, e4m3: bool, dev, seed_rank: int, l2_bytes: int):
        import torch
        from fp8_paged_kv_e4m3_gb300 import inputs, kvq
        self.torch, self.kvq, self.w, self.e4m3, self.dev = torch, kvq, w, e4m3, dev
        w = rank_workload(w, seed_rank)
        self.w = w
        self.layers = max(1, w.layers)
        lay = inputs.page_layout(w)
        self.lay = lay
        lens = lay.lens.astype(np.int64)
        total = int(lens.sum())
        offs = np.concatenate([[0], np.cumsum(lens)[:-1]])
        hs, hp = inputs.history_tokens(w, lay)
        ss, sp = inputs.step_tokens(w, lay)
        hist_slots = torch.from_numpy(inputs.slot_mapping(lay.block_tables, hs, hp)).to(dev)
        hist_rows = torch.from_numpy(offs[hs] + hp).to(dev)
        step_slots = torch.from_numpy(inputs.slot_mapping(lay.block_tables, ss, sp)).to(dev)
        step_rows = torch.from_numpy(offs[ss] + sp).to(dev)
        self.prefill = w.prefill_chunk > 0
        if self.prefill:
            # the step also appends a new sequence's prefill chunk (mixed
            # batches), in the same append call as the decode tokens
            pslots = torch.from_numpy(inputs.prefill_slots(lay)[: w.prefill_chunk]).to(dev)
            step_slots = torch.cat([step_slots, pslots]).contiguous()
        self.step_slots = step_slots
        ti, tl = inputs.topk_lists(w, lay.lens)
        self.topk_idx = None if ti is None else torch.from_numpy(ti).to(dev)
        self.topk_lens = None if tl is None else torch.from_numpy(tl).to(dev)
        self.topk_np = (ti, tl)
        self.bt = torch.from_numpy(lay.block_tables).to(dev)
        self.cl = torch.from_numpy(lay.lens).to(dev)
        shape = (lay.num_pages, w.num_kv_heads, 4, w.head_dim)
        dt = torch.uint8 if e4m3 else torch.float16
        pool_bytes = 2 * math.prod(shape) * (1 if e4m3 else 2)
        self.copies = max(1, math.ceil(2 * l2_bytes / (pool_bytes * self.layers)))
        # per layer: queries, the step's new K/V rows, scales; per (copy, layer): pools
        self.q, self.k_new, self.v_new, self.ks, self.vs = [], [], [], [], []
        self.pools = [[None] * self.layers for _ in range(self.copies)]
        self.beyond = [0, 0]   # E4M3 arm: K and V elements with |x| > 448 * scale (saturated by the quantiser)
        for l in range(self.layers):
            k = inputs.kv_tokens(w, l, total, "k", device=dev)
            v = inputs.kv_tokens(w, l, total, "v", device=dev)
            self.q.append(inputs.queries(w, l, device=dev))
            ks = vs = 1.0
            if e4m3:
                ks = kvq.calibrate_scale(inputs.calibration_draw(w, l, "k", device=dev))
                vs = kvq.calibrate_scale(inputs.calibration_draw(w, l, "v", device=dev))
            self.ks.append(ks)
            self.vs.append(vs)
            kn, vn = k[step_rows], v[step_rows]           # [B * q_len, Hkv, D], rows in (b, i) order
            if self.prefill:
                kn = torch.cat([kn, inputs.prefill_tokens(w, l, "k", device=dev)])
                vn = torch.cat([vn, inputs.prefill_tokens(w, l, "v", device=dev)])
            if e4m3:
                for j, (x, sc) in enumerate(((k, ks), (v, vs))):
                    self.beyond[j] += count_beyond(x, 448.0 * sc)
                    if self.prefill:
                        self.beyond[j] += count_beyond((kn, vn)[j][step_rows.numel():], 448.0 * sc)
            self.k_new.append(kn.contiguous())
            self.v_new.append(vn.contiguous())
            kh, vh = k[hist_rows].contiguous(), v[hist_rows].contiguous()
            del k, v
            for c in range(self.copies):
                kc = torch.zeros(shape, dtype=dt, device=dev)
                vc = torch.zeros(shape, dtype=dt, device=dev)
                self._append(l, kh, vh, hist_slots, kc, vc)
                self.pools[c][l] = (kc, vc)
            del kh, vh
        if e4m3:
            kvq.validate_scales(self.ks, self.vs)
        # batches of varied lengths: the split kernel takes the sequences longest first
        self.longest_first = not w.lens.startswith("fixed")
        self.p = kvq.attn_params(self.q[0], w.num_kv_heads, self.bt.shape[1], w.num_splits,
                                 0 if self.topk_idx is None else self.topk_idx.shape[2],
                                 split_pages=w.split_pages, longest_first=self.longest_first)
        self.S = kvq.num_splits(self.p)
        # one workspace serves every layer: each layer's combine reads it before the
        # next layer's attention writes it (stream order)
        self.ws = kvq.alloc_workspace(self.p, dev)
        self.out = [torch.empty_like(self.q[0]) for _ in range(self.layers)]
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.pool_bytes = pool_bytes
        per_layer = algorithmic_bytes(w, 1 if e4m3 else 2, lay.lens, self.topk_np)
        self.bytes = {"step": per_layer["step"] * self.layers, "attention_kernel": per_layer["attention_kernel"],
                      "layer": per_layer["step"]}
        self.bitcast = False  # E4M3 decoder: hardware conversion (default) or bitcast
        self.mma_sync = False  # many-row tiles: the tcgen05 kernel (default) or the mma.sync kernel
        self.fp8_qk = False    # tcgen05 kernel: fp16 scores (default) or the FP8 score variant
        self.uses_tc = w.head_dim == 128 and w.group * w.q_len > 8
        # dense batches: the fused step call (the append done by the attention launch);
        # with top-k lists or a prefill chunk, the append call and then the attention call
        self.fused = self.topk_idx is None and not self.prefill
        self.shape4 = (w.batch, w.q_len, w.num_kv_heads, w.head_dim)
        torch.cuda.synchronize(dev)

    @property
    def launches(self):
        """Kernels of one step: per layer, the attention call's (as the library
        reports them for these parameters: attention and combine, or one
        cluster-merging attention kernel, with the fused step's append on the
        tcgen05 shapes), plus the append call's unless fused."""
        p = self.kvq.attn_params(self.q[0], self.w.num_kv_heads, self.bt.shape[1], self.S,
                                 0 if self.topk_idx is None else self.topk_idx.shape[2],
                                 split_pages=self.w.split_pages, bitcast_decode=self.bitcast,
                                 mma_sync=self.mma_sync, fp8_qk=self.fp8_qk, longest_first=self.longest_first)
        per_layer = self.kvq.attn_launches(p, self.e4m3, self.fused) + (0 if self.fused else 1)
        return per_layer * self.layers

    def _append(self, l, k, v, slots, kc, vc):
        if self.e4m3:
            self.kvq.kv_append_e4m3(k, v, slots, kc, vc, self.ks[l], self.vs[l], None)
        else:
            self.kvq.kv_append_fp16(k, v, slots, kc, vc, None)

    def _attention(self, l, kc, vc, q=None, bt=None, cl=None, out=None):
        """The attention of layer l through the public calls: with `out`, the
        full call (split-K attention and the merge of its partials); without,
        the partial call alone (split-K attention into the workspace)."""
        kvq = self.kvq
        q = self.q[l] if q is None else q
        bt = self.bt if bt is None else bt
        cl = self.cl if cl is None else cl
        if out is not None:
            if self.e4m3:
                kvq.paged_decode_attn_e4m3(q, kc, vc, bt, cl, self.ks[l], self.vs[l], self.ws, out,
                                           self.topk_idx, self.topk_lens, num_splits=self.S,
                                           err_flag=self.err, split_pages=self.w.split_pages,
                                           bitcast_decode=self.bitcast, mma_sync=self.mma_sync,
                                           fp8_qk=self.fp8_qk, longest_first=self.longest_first)
            else:
                kvq.paged_decode_attn_fp16(q, kc, vc, bt, cl, self.ws, out, self.topk_idx, self.topk_lens,
                                           num_splits=self.S, err_flag=self.err, split_pages=self.w.split_pages,
                                           mma_sync=self.mma_sync, longest_first=self.longest_first)
            return
        if self.e4m3:
            kvq.paged_decode_attn_e4m3_partial(q, kc, vc, bt, cl, self.ks[l], self.vs[l], self.ws,
                                               self.topk_idx, self.topk_lens, num_splits=self.S,
                                               err_flag=self.err, split_pages=self.w.split_pages,
                                               bitcast_decode=self.bitcast, mma_sync=self.mma_sync,
                                               fp8_qk=self.fp8_qk, longest_first=self.longest_first)
        else:
            kvq.paged_decode_attn_fp16_partial(q, kc, vc, bt, cl, self.ws, self.topk_idx,
                                               self.topk_lens, num_splits=self.S, err_flag=self.err,
                                               split_pages=self.w.split_pages, mma_sync=self.mma_sync,
                                               longest_first=self.longest_first)

    def _layer_step(self, l, kc, vc, k, v, slots, q, bt, cl, out):
        """Layer l's share of a step: the append of the step's tokens and the
        attention over the updated cache -- the fused step call, or the append
        call and the attention call; chained with programmatic dependent
        launch.  The kernels each call launches are those the library reports
        (kvq_attn_launches)."""
        kvq = self.kvq
        if not self.fused:
            self._append(l, k, v, slots, kc, vc)
            self._attention(l, kc, vc, q, bt, cl, out=out)
            return
        k4, v4 = k.view(self.shape4), v.view(self.shape4)
        if self.e4m3:
            kvq.paged_decode_step_e4m3(q, k4, v4, kc, vc, bt, cl, self.ks[l], self.vs[l], self.ws, out,
                                       num_splits=self.S, err_flag=self.err, split_pages=self.w.split_pages,
                                       bitcast_decode=self.bitcast, mma_sync=self.mma_sync, fp8_qk=self.fp8_qk,
                                       longest_first=self.longest_first)
        else:
            kvq.paged_decode_step_fp16(q, k4, v4, kc, vc, bt, cl, self.ws, out, num_splits=self.S,
                                       err_flag=self.err, split_pages=self.w.split_pages, mma_sync=self.mma_sync,
                                       longest_first=self.longest_first)

    def step(self, i):
        """One step on pool copy i: every layer's append and attention."""
        for l in range(self.layers):
            kc, vc = self.pools[i % self.copies][l]
            self._layer_step(l, kc, vc, self.k_new[l], self.v_new[l], self.step_slots, self.q[l], self.bt,
                             self.cl, self.out[l])

    def capture(self):
        """CUDA graphs of the step: one per pool copy holding one step, and
        one holding GRAPH_STEPS consecutive steps (cycling the copies), as a
        serving loop captures many layers in one graph; replaying them
        removes host launch cost and most of the gap between graphs."""
        torch = self.torch
        for i in range(2):                       # warm up (sets kernel attributes) before capture
            self.step(i)
        torch.cuda.synchronize(self.dev)
        graphs = []
        for r in range(self.copies):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self.step(r)
            graphs.append(g)
        many = None
        if self.layers == 1:                     # a multi-layer step is already a long graph
            many = torch.cuda.CUDAGraph()
            with torch.cuda.graph(many):
                for r in range(GRAPH_STEPS):
                    self.step(r)
        torch.cuda.synchronize(self.dev)
        self.graphs, self.many = graphs, many

    def time(self, steps, warmup, barrier=None):
        """Exactly `steps` whole steps between two events: replays of the
        GRAPH_STEPS-step graph, then one-step graphs for the remainder.  The
        warm-up replays the one-step graphs `warmup` times and the multi-step
        graph once, so that no graph's first launch is timed."""
        torch = self.torch
        if not getattr(self, "graphs", None):
            self.capture()
        graphs, many = self.graphs, self.many
        for i in range(warmup):
            graphs[i % self.copies].replay()
        if many is not None and steps >= GRAPH_STEPS:
            many.replay()   # the multi-step graph's first launch (its upload) stays out of the timed region
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(self.dev)
        if barrier:
            barrier()
        torch.cuda.synchronize(self.dev)
        torch.cuda.nvtx.range_push("kvq_timed")
        start.record()
        n_many = steps // GRAPH_STEPS if many is not None else 0
        for _ in range(n_many):
            many.replay()
        for i in range(steps - n_many * GRAPH_STEPS):
            graphs[i % self.copies].replay()
        end.record()
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize(self.dev)
        if barrier:
            barrier()
        assert self.err.item() == 0, f"device error bits {self.err.item()}"
        return start.elapsed_time(end)

    def time_kernel(self, steps, warmup):
        """Average duration of one attention kernel (one layer; the partial
        call): `steps` back-to-back launches over the rotating pool copies and
        layers, between two events on the launching stream (the queue stays
        full, so host launch time is hidden)."""
        torch = self.torch
        n = self.copies * self.layers

        def run(j):
            c, l = divmod(j % n, self.layers)
            kc, vc = self.pools[c][l]
            self._attention(l, kc, vc)

        for i in range(warmup):
            run(i)
        torch.cuda.synchronize(self.dev)
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.nvtx.range_push("kvq_kernel_timed")
        start.record()
        for i in range(steps):
            run(warmup + i)
        end.record()
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize(self.dev)
        assert self.err.item() == 0, f"device error bits {self.err.item()}"
        return start.elapsed_time(end) / steps

    def step_percentiles(self, steps):
        """Per-step durations (ms) of graph replays, each between its own
        events: (p10, median, p90)."""
        torch = self.torch
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
        torch.cuda.synchronize(self.dev)
        evs[0].record()
        for i in range(steps):
            self.graphs[i % self.copies].replay()
            evs[i + 1].record()
        torch.cuda.synchronize(self.dev)
        d = np.array([evs[i].elapsed_time(evs[i + 1]) for i in range(steps)])
        return tuple(float(x) for x in np.percentile(d, [10, 50, 90]))

    def time_e2e(self, steps, warmup):
        """Every step: the H2D copy of the step's inputs (every layer's Q and
        new K/V, the slots, block tables and lengths; packed in one pinned
        host buffer, so one copy), the step through the public calls, and a
        D2H read of every layer's output.  Returns (pipelined ms, serial ms,
        H2D bytes, D2H bytes): pipelined = the copies on their own streams,
        overlapping the neighbouring steps' compute (two input and two output
        buffers); serial = copies and compute in one graph per step on one
        stream."""
        torch = self.torch
        src = ([] if self.fused else [("slots", self.step_slots)]) + [("bt", self.bt), ("cl", self.cl)]
        for l in range(self.layers):
            src += [(f"q{l}", self.q[l]), (f"k{l}", self.k_new[l]), (f"v{l}", self.v_new[l])]
        sets = [staged_buffers(torch, src, self.dev) for _ in range(2)]
        oshape = (self.layers,) + tuple(self.out[0].shape)
        outs = [torch.empty(oshape, dtype=self.out[0].dtype, device=self.dev) for _ in range(2)]
        out_host = [torch.empty(oshape, dtype=self.out[0].dtype).pin_memory() for _ in range(2)]
        h2d = sum(t.numel() * t.element_size() for _, t in src)
        d2h = out_host[0].numel() * out_host[0].element_size()

        def copy_in(p):
            sets[p][1]["_buf"].copy_(sets[p][0]["_buf"], non_blocking=True)

        def compute(i):
            dev = sets[i % 2][1]
            for l in range(self.layers):
                kc, vc = self.pools[i % self.copies][l]
                self._layer_step(l, kc, vc, dev[f"k{l}"], dev[f"v{l}"], dev.get("slots"), dev[f"q{l}"], dev["bt"],
                                 dev["cl"], outs[i % 2][l])

        def copy_out(p):
            out_host[p].copy_(outs[p], non_blocking=True)

        def one(i):
            copy_in(i % 2)
            compute(i)
            copy_out(i % 2)

        ncap = self.copies * 2 // math.gcd(self.copies, 2)   # pool copies and buffer sets both cycle
        piped = pipelined_timed(torch, self.dev, copy_in, compute, copy_out, ncap, steps, warmup)
        serial = replay_timed(torch, self.dev, one, ncap, steps, warmup)
        return piped, serial, h2d, d2h


def staged_buffers(torch, src, device):
    """One pinned host buffer and one device buffer holding the tensors of
    `src` (name, tensor) at 256-byte aligned offsets, filled with their
    values; returns (host views, device views), each with "_buf"."""
    offs, total = {}, 0
    for name, t in src:
        offs[name] = total
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    hbuf = torch.empty(total, dtype=torch.uint8).pin_memory()
    dbuf = torch.empty(total, dtype=torch.uint8, device=device)
    host, dev = {"_buf": hbuf}, {"_buf": dbuf}
    for name, t in src:
        n = t.numel() * t.element_size()
        hv = hbuf[offs[name]:offs[name] + n].view(t.dtype).view(t.shape)
        hv.copy_(t.cpu())
        host[name] = hv
        dev[name] = dbuf[offs[name]:offs[name] + n].view(t.dtype).view(t.shape)
    return host, dev


def pipelined_timed(torch, device, copy_in, compute, copy_out, period, steps, warmup, graph_steps=GRAPH_STEPS):
    """Steps with their copies on their own streams, as a serving loop
    overlaps them: copy_in(p) (H2D into input set p), compute(i) (input set
    and output buffer i % 2) and copy_out(p) (D2H of output buffer p).  Step
    i's inputs copy in while step i-1 computes and step i-2's output copies
    out; a buffer is reused only after the step two back has finished with
    it.  A run of n steps (n a multiple of `period`, about GRAPH_STEPS) is
    captured in one CUDA graph with the three streams forked from and joined
    to the capture stream, so the host issues one launch per n steps
    (n about graph_steps).
    Returns the average ms per step over the replays covering `steps`."""
    n = period * max(1, round(graph_steps / period))
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    for i in range(2):
        copy_in(i % 2)
        compute(i)
        copy_out(i % 2)
    torch.cuda.synchronize(device)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_c = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cap = torch.cuda.current_stream(device)
        s_in.wait_stream(cap)
        s_out.wait_stream(cap)
        for i in range(n):
            p = i % 2
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_c[p])      # the step two back has read input set p
                copy_in(p)
                ev_in[p].record(s_in)
            cap.wait_event(ev_in[p])
            if i >= 2:
                cap.wait_event(ev_out[p])         # the step two back's output has been read
            compute(i)
            ev_c[p].record(cap)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_c[p])
                copy_out(p)
                ev_out[p].record(s_out)
        cap.wait_stream(s_in)
        cap.wait_stream(s_out)
    for _ in range(max(1, warmup // n)):
        g.replay()
    torch.cuda.synchronize(device)
    reps = max(1, steps // n)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for _ in range(reps):
        g.replay()
    end.record()
    torch.cuda.synchronize(device)
    return start.elapsed_time(end) / (reps * n)


def replay_timed(torch, device, one, copies, steps, warmup):
    """Capture one(i) for i < copies in CUDA graphs, replay them in turn and
    return the average ms per step (events around exactly `steps` replays)."""
    for i in range(2):
        one(i)
    torch.cuda.synchronize(device)
    graphs = []
    for r in range(copies):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            one(r)
        graphs.append(g)
    for i in range(warmup):
        graphs[i % copies].replay()
    torch.cuda.synchronize(device)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for i in range(steps):
        graphs[i % copies].replay()
    end.record()
    torch.cuda.synchronize(device)
    return start.elapsed_time(end) / steps


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline leg and the reference arm)

def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), or "unknown"."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def step_units(w):
    """Every (sequence, kv head) unit of one layer of the workload's step."""
    return [(b, g) for b in range(w.batch) for g in range(w.num_kv_heads)]


_ORACLE_DATA = {}
_ORACLE_BARRIER = None


def _oracle_data(w):
    """The workload's CPU-drawn K/V rows, layout and calibrated scales (layer
    0), drawn once per process."""
    from fp8_paged_kv_e4m3_gb300 import inputs
    import oracle
    if w not in _ORACLE_DATA:
        lay = inputs.page_layout(w)
        lens = lay.lens.astype(np.int64)
        total = int(lens.sum())
        k = inputs.kv_tokens(w, 0, total, "k").numpy()
        v = inputs.kv_tokens(w, 0, total, "v").numpy()
        ks = oracle.calibrate_scale(inputs.calibration_draw(w, 0, "k").numpy())
        vs = oracle.calibrate_scale(inputs.calibration_draw(w, 0, "v").numpy())
        _ORACLE_DATA[w] = (lay, np.concatenate([[0], np.cumsum(lens)[:-1]]), k, v,
                           inputs.queries(w, 0).numpy(), ks, vs)
    return _ORACLE_DATA[w]


def _oracle_units(w, picks, barrier_timeout=None):
    """The oracle on (sequence, kv head) units of the step: untimed, each
    unit's cached history appended into a pool of its own; then, timed, the
    append of the step's tokens and the binary64 attention of the unit's
    query heads.  With a barrier (the all-cores run) every worker starts its
    timed part together.  Returns (t0, t1, algorithmic bytes)."""
    import oracle
    lay, offs, k, v, q, ks, vs = _oracle_data(w)
    G, ql = w.group, w.q_len
    prepared = []
    nbytes = 0
    for b, g in picks:
        L = int(lay.lens[b])
        ku = np.ascontiguousarray(k[offs[b]:offs[b] + L, g:g + 1])
        vu = np.ascontiguousarray(v[offs[b]:offs[b] + L, g:g + 1])
        pages = (L + 3) // 4
        kc = np.zeros((pages, 1, 4, w.head_dim), np.uint8)
        vc = np.zeros_like(kc)
        slots = np.arange(L, dtype=np.int32)
        oracle.append_e4m3(ku[: L - ql], vu[: L - ql], slots[: L - ql], kc, vc, ks, vs)
        qu = np.ascontiguousarray(q[b:b + 1, :, g * G:(g + 1) * G])
        prepared.append((L, ku, vu, slots, kc, vc, qu, np.arange(pages, dtype=np.int32)[None]))
        nbytes += 2 * L * w.head_dim + 2 * qu.nbytes + pages * 4 + ql * w.head_dim * 6
    if _ORACLE_BARRIER is not None and barrier_timeout:
        _ORACLE_BARRIER.wait(barrier_timeout)
    t0 = time.perf_counter()
    for L, ku, vu, slots, kc, vc, qu, bt in prepared:
        oracle.append_e4m3(ku[L - ql:], vu[L - ql:], slots[L - ql:], kc, vc, ks, vs)
        oracle.attention(qu, kc, vc, bt, np.array([L], np.int32), ks, vs)
    t1 = time.perf_counter()
    return t0, t1, nbytes


def _oracle_pool_init(barrier):
    """Worker set-up: one thread per worker process (the oracle is single-
    threaded; idle library threads spinning after the input draw would take
    cores from the other workers' timed parts)."""
    global _ORACLE_BARRIER
    _ORACLE_BARRIER = barrier
    os.environ["OMP_NUM_THREADS"] = "1"
    import torch
    torch.set_num_threads(1)


class OracleTimer:
    """The oracle timed on this host: one process per core (spawned, so no
    worker inherits a CUDA context), each taking an equal share of the
    units; their timed parts start together at a barrier, and the wall time
    runs from the first start to the last end."""

    def __init__(self, workers=None):
        import concurrent.futures as cf
        import multiprocessing as mp
        self.workers = workers or host_cores()
        ctx = mp.get_context("spawn")
        self.barrier = ctx.Barrier(self.workers)
        self.ex = cf.ProcessPoolExecutor(max_workers=self.workers, mp_context=ctx,
                                         initializer=_oracle_pool_init, initargs=(self.barrier,))

    def run(self, w, picks):
        """(seconds, bytes) of the timed part over `picks`, on all workers."""
        shares = [picks[i::self.workers] for i in range(self.workers)]
        futs = [self.ex.submit(_oracle_units, w, sh, 600.0) for sh in shares]
        res = [f.result() for f in futs]
        return max(r[1] for r in res) - min(r[0] for r in res), sum(r[2] for r in res)

    def close(self):
        self.ex.shutdown(cancel_futures=True)


def oracle_one_core(w, picks):
    """(seconds, bytes) of the timed part over `picks` in this process."""
    t0, t1, nb = _oracle_units(w, picks)
    return t1 - t0, nb


def cpu_baseline_decode(w):
    """The oracle on every (sequence, kv head) unit of one layer of the step,
    over all host cores and on one core."""
    picks = step_units(w)
    cores = host_cores()
    timer = OracleTimer(cores)
    try:
        timer.run(w, picks[: timer.workers])              # start-up: spawn, import, draw the inputs
        t_all, nb = timer.run(w, picks)
    finally:
        timer.close()
    t_one, nb1 = oracle_one_core(w, picks)
    return {"value": nb / t_all / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "cpu_model": cpu_model(), "nproc": os.cpu_count(),
            "value_1core": nb1 / t_one / 1e9, "seconds_all_cores": t_all, "seconds_1core": t_one,
            "sample": f"all {len(picks)} (sequence, kv head) units of one layer of the {w.name} step "
                      f"({w.group} query heads each): append of the step's tokens + binary64 attention; "
                      f"{cores} spawned processes, timed parts started together; and the same on 1 core"}


def library_splits(w, max_pages: int, sm_count: int, longest_first: bool = False) -> int:
    """The split count the library picks for this workload (the rule of
    kvq_attn_num_splits, restated so that the reference arm can label its
    config like ours without loading the CUDA library)."""
    max_topk = w.topk if w.topk > 0 else 0
    if w.num_splits > 0:
        return w.num_splits
    if w.split_pages > 0:
        sp = w.split_pages
        return max(1, -(-max_pages // sp), -(-max_topk // (4 * sp)))
    pairs = max(w.batch, 1) * w.num_kv_heads
    rows = w.group * w.q_len
    if w.head_dim == 128 and 8 < rows <= 64:          # the tcgen05 kernel
        s = -(-(sm_count * 6) // pairs)
        cap = -(-max_pages // 16)
        if max_topk > 0:
            cap = max(cap, -(-max_topk // 32))
    else:                                              # the split kernel
        slots = sm_count * 4
        s = (slots * 5 // 2) // pairs if longest_first else (slots * 2) // pairs
        cap = -(-max_pages // 256)
        if max_topk > 0:
            cap = max(cap, -(-max_topk // 1024))
    return max(1, min(s, cap, 1024))


def reference_config(w, world: int, sample: str) -> dict:
    """The config of our arm's line for workload w, for the reference arm."""
    from fp8_paged_kv_e4m3_gb300 import inputs
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count if torch.cuda.is_available() else 152
    lay = inputs.page_layout(w)
    return {"workload": describe(w, library_splits(w, lay.block_tables.shape[1], sms,
                                                   longest_first=not w.lens.startswith("fixed"))),
            "global_batch": world * w.batch, "kv_dtype": "e4m3 (fp16 MMA, fp32 accumulate)",
            "l2": "host oracle: no GPU cache to defeat", "parallelism": f"replicas x{world}",
            "sample": sample}


def run_reference(args, w):
    """The reference arm: the CPU oracle over all host cores, each step the
    (sequence, kv head) units of one layer of the step -- all of them, or,
    where that would take too long, a seeded sample sized so that the whole
    run stays within about three minutes."""
    if w.name == "prefill":
        return run_reference_prefill(args, w)
    picks = step_units(w)
    timer = OracleTimer()
    try:
        t_cal, _ = timer.run(w, picks[: timer.workers])       # start-up, and one unit per worker
        per_step_budget = 150.0 / max(1, args.steps + args.warmup)
        n = len(picks)
        if t_cal * len(picks) / timer.workers > per_step_budget:
            n = max(timer.workers, int(per_step_budget / max(t_cal, 1e-3) * timer.workers))
        rng = np.random.default_rng(1234)
        sample = picks if n >= len(picks) else [picks[i] for i in np.sort(rng.choice(len(picks), n, False))]
        for _ in range(args.warmup):
            timer.run(w, sample)
        t = nb = 0.0
        for _ in range(args.steps):
            dt, b = timer.run(w, sample)
            t += dt
            nb += b
    finally:
        timer.close()
    gbs = nb / t / 1e9
    what = "all" if len(sample) == len(picks) else f"a seeded sample of {len(sample)} of the"
    sample_txt = (f"{what} {len(picks)} (sequence, kv head) units of one layer of the {w.name} step per step "
                  f"(append of the step's tokens + binary64 attention of {w.group} query heads), "
                  f"{timer.workers} processes")
    line = {"impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * t / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": reference_config(w, args.gpus, sample_txt),
            "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": timer.workers, "kind": "oracle",
                             "cpu_model": cpu_model(), "sample": sample_txt},
            "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# chunked prefill (the mixed batch's 8192-token chunk attended)

PREFILL_METRIC = "E4M3 paged chunked-prefill attention TFLOP/s (causal, fp16 MMA) vs FP16 KV"


def prefill_flops(n: int, base: int, Hq: int, D: int) -> float:
    """QK and PV multiply-adds (2 flops each) of a causal chunk of n query
    tokens after `base` earlier keys: row i attends base + i + 1 keys."""
    keys = n * base + n * (n + 1) / 2
    return 4.0 * D * Hq * keys


class PrefillArm:
    """One arm of the prefill step: append of the chunk (quantise-on-write
    for E4M3), then the prefill call (tile gather + attention)."""

    def __init__(self, w, e4m3: bool, dev, seed_rank: int, l2_bytes: int):
        import torch
        from fp8_paged_kv_e4m3_gb300 import inputs, kvq
        self.torch, self.kvq, self.e4m3, self.dev = torch, kvq, e4m3, dev
        w = rank_workload(w, seed_rank)
        self.w = w
        lay = inputs.page_layout(w)
        n, B = w.q_len, w.batch
        lens = lay.lens.astype(np.int64)
        ss, sp = inputs.step_tokens(w, lay)                  # the chunk: the last n positions
        self.slots = torch.from_numpy(inputs.slot_mapping(lay.block_tables, ss, sp)).to(dev)
        offs = np.concatenate([[0], np.cumsum(lens)[:-1]])
        rows = torch.from_numpy(offs[ss] + sp).to(dev)
        total = int(lens.sum())
        self.bt = torch.from_numpy(lay.block_tables).to(dev)
        self.cl = torch.from_numpy(lay.lens).to(dev)
        self.q_start = torch.arange(0, (B + 1) * n, n, dtype=torch.int32, device=dev)
        shape = (lay.num_pages, w.num_kv_heads, 4, w.head_dim)
        dt = torch.uint8 if e4m3 else torch.float16
        # copies of (chunk K/V, Q, pools, out) rotated so that one step's data is not in L2
        per_copy = (2 * n * B * w.num_kv_heads * w.head_dim * 2 + 2 * n * B * w.num_q_heads * w.head_dim * 2
                    + 2 * math.prod(shape) * (1 if e4m3 else 2))
        self.copies = max(2, math.ceil(2 * l2_bytes / per_copy))
        self.sets = []
        for c in range(self.copies):
            layer = c % max(1, w.layers)
            k = inputs.kv_tokens(w, layer, total, "k", device=dev)[rows].contiguous()
            v = inputs.kv_tokens(w, layer, total, "v", device=dev)[rows].contiguous()
            q = inputs.queries(w, layer, device=dev).reshape(B * n, w.num_q_heads, w.head_dim).contiguous()
            ks = vs = 1.0
            if e4m3:
                ks = kvq.calibrate_scale(inputs.calibration_draw(w, layer, "k", device=dev))
                vs = kvq.calibrate_scale(inputs.calibration_draw(w, layer, "v", device=dev))
            if e4m3 and c == 0:   # the copy whose output is compared with the fp16 arm's
                self.beyond = [count_beyond(k, 448.0 * ks), count_beyond(v, 448.0 * vs)]
            kc = torch.zeros(shape, dtype=dt, device=dev)
            vc = torch.zeros(shape, dtype=dt, device=dev)
            self.sets.append((k, v, q, kc, vc, torch.empty_like(q), ks, vs))
        self.p = kvq.PrefillParams(B, w.num_q_heads, w.num_kv_heads, w.head_dim, self.bt.shape[1], n,
                                   B * n, 0.0, 0)
        self.ws = kvq.alloc_prefill_workspace(self.p, dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.flops = sum(prefill_flops(n, int(L) - n, w.num_q_heads, w.head_dim) for L in lens)
        self.launches = 3   # append, tile gather, attention
        for i in range(self.copies):
            self._append(i)

    def _append(self, i):
        k, v, q, kc, vc, out, ks, vs = self.sets[i]
        if self.e4m3:
            self.kvq.kv_append_e4m3(k, v, self.slots, kc, vc, ks, vs, self.err)
        else:
            self.kvq.kv_append_fp16(k, v, self.slots, kc, vc, self.err)

    def attention(self, i, q=None, out=None):
        k, v, q0, kc, vc, out0, ks, vs = self.sets[i]
        q = q0 if q is None else q
        out = out0 if out is None else out
        kvq = self.kvq
        if self.e4m3:
            kvq.paged_prefill_attn_e4m3(q, kc, vc, self.bt, self.cl, self.q_start, ks, vs, self.ws, out=out,
                                        max_q_len=self.w.q_len, err_flag=self.err)
        else:
            kvq.paged_prefill_attn_fp16(q, kc, vc, self.bt, self.cl, self.q_start, self.ws, out=out,
                                        max_q_len=self.w.q_len, err_flag=self.err)

    def step(self, i):
        self._append(i % self.copies)
        self.attention(i % self.copies)

    def _events(self, fn, steps, warmup):
        torch = self.torch
        for i in range(warmup):
            fn(i)
        torch.cuda.synchronize(self.dev)
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for i in range(steps):
            fn(i)
        e.record()
        torch.cuda.synchronize(self.dev)
        assert self.err.item() == 0, f"device error bits {self.err.item()}"
        return s.elapsed_time(e)

    def time(self, steps, warmup):
        return self._events(self.step, steps, warmup)

    def time_kernel(self, steps, warmup):
        """The prefill call alone (tile gather + attention), back to back."""
        return self._events(lambda i: self.attention(i % self.copies), steps, warmup) / steps

    def time_e2e(self, steps, warmup):
        """Through the public calls with the chunk's Q and K/V copied in from
        pinned host memory (one packed buffer, one copy) and the output read
        back, every step.  Returns (pipelined ms, serial ms, H2D bytes, D2H
        bytes), as the decode arm's time_e2e."""
        torch = self.torch
        k, v, q, kc, vc, out, ks, vs = self.sets[0]
        sets = [staged_buffers(torch, [("k", k), ("v", v), ("q", q)], self.dev) for _ in range(2)]
        outs = [out, torch.empty_like(out)]
        ho = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]

        def copy_in(p):
            sets[p][1]["_buf"].copy_(sets[p][0]["_buf"], non_blocking=True)

        def compute(i):
            dev = sets[i % 2][1]
            if self.e4m3:
                self.kvq.kv_append_e4m3(dev["k"], dev["v"], self.slots, kc, vc, ks, vs, self.err)
            else:
                self.kvq.kv_append_fp16(dev["k"], dev["v"], self.slots, kc, vc, self.err)
            self.attention(0, q=dev["q"], out=outs[i % 2])

        def copy_out(p):
            ho[p].copy_(outs[p], non_blocking=True)

        def one(i):
            copy_in(i % 2)
            compute(i)
            copy_out(i % 2)

        piped = pipelined_timed(torch, self.dev, copy_in, compute, copy_out, 2, steps, warmup)
        serial = replay_timed(torch, self.dev, one, 2, steps, warmup)
        assert self.err.item() == 0, f"device error bits {self.err.item()}"
        return piped, serial, sum(t.numel() * t.element_size() for t in (k, v, q)), ho[0].numel() * ho[0].element_size()


def prefill_oracle_sample(w, rows=(0, 4095, 8191)):
    """The oracle on a few rows of the chunk (each row one decode-sized
    problem: row i attends keys 0 .. L - n + i).  Returns (seconds, flops)."""
    import oracle
    from fp8_paged_kv_e4m3_gb300 import inputs
    lay = inputs.page_layout(w)
    n = w.q_len
    L = int(lay.lens[0])
    k = inputs.kv_tokens(w, 0, L, "k").numpy()
    v = inputs.kv_tokens(w, 0, L, "v").numpy()
    q = inputs.queries(w, 0).numpy()
    ks = oracle.calibrate_scale(inputs.calibration_draw(w, 0, "k").numpy())
    vs = oracle.calibrate_scale(inputs.calibration_draw(w, 0, "v").numpy())
    shape = (lay.num_pages, w.num_kv_heads, 4, w.head_dim)
    kc = np.zeros(shape, np.uint8)
    vc = np.zeros(shape, np.uint8)
    pos = np.arange(L)
    slots = inputs.slot_mapping(lay.block_tables[:1], np.zeros(L, np.int64), pos)
    oracle.append_e4m3(k, v, slots, kc, vc, ks, vs)
    t0 = time.perf_counter()
    fl = 0.0
    for i in rows:
        Li = L - n + i + 1
        oracle.attention(q[:1, i:i + 1], kc, vc, lay.block_tables[:1], np.array([Li], np.int32), ks, vs)
        fl += 4.0 * w.head_dim * w.num_q_heads * Li
    return time.perf_counter() - t0, fl


def describe_prefill(w) -> str:
    return (f"prefill: {w.batch} x {w.q_len}-token chunk over its own context (causal), {w.num_q_heads} q / "
            f"{w.num_kv_heads} kv heads, head_dim {w.head_dim}, page 4; one layer")


def measure_prefill(args, w, dev, l2, rank, world, reduce_max, barrier, with_cpu=True):
    """The prefill step (append of the chunk, then the prefill call) of both
    arms; returns the JSON fields of its line (rank 0) without the clocks."""
    import torch
    tpeak, tkind = _tensor_peak()
    arm = PrefillArm(w, True, dev, rank, l2)
    if barrier:
        barrier()
    total_ms = reduce_max(arm.time(args.steps, args.warmup))
    kern_ms = reduce_max(arm.time_kernel(args.steps, args.warmup))
    ms = total_ms / args.steps
    tflops = world * arm.flops / (ms * 1e-3) / 1e12
    achieved = arm.flops / (kern_ms * 1e-3) / 1e12
    e2e_ms, e2e_serial_ms, h2d, d2h = arm.time_e2e(max(3, args.steps // 4), 2)
    e2e_ms, e2e_serial_ms = reduce_max(e2e_ms), reduce_max(e2e_serial_ms)
    copies, flops, launches = arm.copies, arm.flops, arm.launches
    fp16 = out_err = None
    if not args.no_fp16:
        out8 = arm.sets[0][5].clone()                   # copy 0's output
        del arm.sets
        torch.cuda.empty_cache()
        a16 = PrefillArm(w, False, dev, rank, l2)
        ms16 = reduce_max(a16.time(args.steps, args.warmup)) / args.steps
        k16 = reduce_max(a16.time_kernel(args.steps, args.warmup))
        fp16 = {"ms_per_step": ms16, "value": world * a16.flops / (ms16 * 1e-3) / 1e12,
                "prefill_call_ms": k16}
        out_err = output_error([out8], [a16.sets[0][5]])
        out_err["k_elements_beyond_448_scale"], out_err["v_elements_beyond_448_scale"] = arm.beyond
        del a16
    del arm
    torch.cuda.empty_cache()
    cpu = None
    if rank == 0 and with_cpu and not args.no_cpu_baseline:
        t, fl = prefill_oracle_sample(w)
        cpu = {"value": fl / t / 1e12, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
               "sample": f"3 rows (tokens 0, 4095, 8191) of the chunk, all {w.num_q_heads} query heads, "
                         f"binary64 attention, {t:.1f} s"}
    return {
        "metric": PREFILL_METRIC, "value": tflops, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 (fp16 MMA, fp32 accumulate)",
        "data": "synthetic",
        "config": {"workload": describe_prefill(w),
                   "l2": f"rotating {copies} copies of chunk K/V, Q, pools and output (> 2 x L2)",
                   "parallelism": f"replicas x{world}"},
        "flops_per_step": world * flops,
        "fp16_arm": fp16,
        "e4m3_speedup_vs_fp16": (fp16["ms_per_step"] / ms) if fp16 else None,
        "e4m3_vs_fp16_output": out_err,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": tpeak, "unit": "TFLOP/s",
                     "frac": achieved / tpeak, "traffic": profiled_traffic("prefill_attn_kernel", w.name),
                     "kernel": "kv_tile_kernel + prefill_attn_kernel (E4M3, tcgen05), one call",
                     "peak_kind": tkind, "prefill_call_ms": kern_ms},
        "cpu_baseline": cpu,
        "e2e": {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "copies": "own streams, overlapping the neighbouring steps' compute",
                "serial_ms_per_step": e2e_serial_ms},
        "gpu_launches": launches * args.steps,
        "launch": "append, tile gather, attention per step (programmatic dependent launch); "
                  "e2e: the compute of each step in a CUDA graph, H2D and D2H copies on their own streams",
    }


def run_prefill_bench(args, w, dev, l2, rank, world, reduce_max, barrier):
    import torch
    with ClockSampler(torch.cuda.current_device()) as clk:
        line = measure_prefill(args, w, dev, l2, rank, world, reduce_max, barrier)
    if rank == 0:
        line["clocks"] = clk.summary()
        print(json.dumps(line), flush=True)


def run_reference_prefill(args, w):
    """The reference arm on the prefill workload: the oracle on a few rows of
    the chunk per step."""
    for _ in range(min(args.warmup, 1)):
        prefill_oracle_sample(w, rows=(8191,))
    t = fl = 0.0
    for _ in range(args.steps):
        dt, f = prefill_oracle_sample(w, rows=(8191,))
        t += dt
        fl += f
    v = fl / t / 1e12
    sample = f"row 8191 of the {w.q_len}-token chunk (all {w.num_q_heads} query heads) per step, binary64"
    print(json.dumps({"impl": "reference", "metric": PREFILL_METRIC, "value": v, "unit": "TFLOP/s",
                      "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                      "ms_per_step": 1e3 * t / args.steps, "higher_is_better": True, "scaling": "weak",
                      "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                      "config": {"workload": describe_prefill(w), "l2": "host oracle: no GPU cache to defeat",
                                 "parallelism": f"replicas x{args.gpus}", "sample": sample},
                      "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": 1, "kind": "oracle", "sample": sample},
                      "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
                      "gpu_launches": 0}), flush=True)


# ---------------------------------------------------------------------------
# multi-rank helpers (replicas: no data-path exchange, only the timing reduction)

def max_over_ranks(x: float, device, world: int) -> float:
    """The slowest rank's value (timing is max over ranks)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(step_bytes_per_rank: int, batch_per_rank: int, world: int, ms_max: float):
    """Whole-job GB/s and sequence-steps/s from the slowest rank's step time:
    every rank processes its own batch of the same shape (weak scaling)."""
    return (world * step_bytes_per_rank / (ms_max * 1e-3) / 1e9,
            world * batch_per_rank / (ms_max * 1e-3))


def rank_workload(w, rank: int):
    """Rank r's replica: same shapes, its own seeded data."""
    import dataclasses
    return dataclasses.replace(w, seed=rank) if rank else w


# ---------------------------------------------------------------------------

EXTRA_WORKLOADS = ("decode32k", "long", "verify", "mixed", "prefill")


def count_beyond(x, limit: float) -> int:
    """Elements of x with |x| > limit (compared in binary32, in chunks)."""
    flat = x.reshape(-1)
    return sum(int((c.float().abs() > limit).sum()) for c in flat.split(1 << 26))


def output_error(e4m3_outs, fp16_outs):
    """The E4M3 arm's outputs against the fp16-KV arm's on the same inputs
    (reported, not gated): the largest |difference|, the RMS of the
    differences, that RMS over the RMS of the fp16 outputs, and the smallest
    cosine similarity of one output row (one query row of one head, D values)."""
    import torch
    a = torch.cat([o.reshape(-1, o.shape[-1]).float() for o in e4m3_outs])
    b = torch.cat([o.reshape(-1, o.shape[-1]).float() for o in fp16_outs])
    d = a - b
    rms = d.square().mean().sqrt().item()
    ref = b.square().mean().sqrt().item()
    cos = torch.nn.functional.cosine_similarity(a, b, dim=1)
    return {"max_abs": d.abs().max().item(), "rms": rms, "rel_rms": rms / ref if ref > 0 else None,
            "min_row_cosine": cos.min().item(), "rows": int(a.shape[0]),
            "rows_below_0_99_cosine": int((cos < 0.99).sum()),
            "note": "E4M3 arm vs fp16-KV arm, same inputs; reported, not gated"}


def measure(args, w, dev, l2, rank, world, reduce_max, barrier, peak, peak_kind, headline=False):
    """The step of a decode / verify workload, both arms; returns the JSON
    fields of its line (rank 0) without the clocks and the CPU baseline."""
    import torch
    arm = Arm(w, True, dev, rank, l2)
    arm.capture()
    total_ms = reduce_max(arm.time(args.steps, args.warmup, barrier))
    ms = total_ms / args.steps
    kern_steps = max(args.steps, arm.layers)
    kern_avg = reduce_max(arm.time_kernel(kern_steps, args.warmup))
    step_bytes = arm.bytes["step"]
    gbs, seq_steps = aggregate(step_bytes, w.batch, world, ms)
    achieved = arm.bytes["attention_kernel"] / (kern_avg * 1e-3) / 1e9
    pct = arm.step_percentiles(max(20, args.steps)) if headline else None   # context: per-step spread
    separate_ms = None
    if arm.fused:                                       # context: the append call, then the attention call
        arm.fused, arm.graphs, arm.many = False, None, None
        separate_ms = reduce_max(arm.time(args.steps, args.warmup, barrier)) / args.steps
        arm.fused, arm.graphs, arm.many = True, None, None
    arm.bitcast = True                                  # context: the pages' bitcast decoder
    bitcast_ms = reduce_max(arm.time_kernel(kern_steps, args.warmup))
    arm.bitcast = False
    mma_sync_ms = fp8_qk_ms = None
    if arm.uses_tc:                                     # context: the same shape on the mma.sync kernel
        arm.mma_sync = True
        mma_sync_ms = reduce_max(arm.time_kernel(kern_steps, args.warmup))
        arm.mma_sync = False
        arm.fp8_qk = True                               # context: the FP8 score variant (other numerics)
        fp8_qk_ms = reduce_max(arm.time_kernel(kern_steps, args.warmup))
        arm.fp8_qk = False
    arm.graphs = arm.many = None
    e2e_steps = max(5, args.steps // 2) if arm.layers == 1 else max(3, args.steps // 4)
    e2e_ms, e2e_serial_ms, h2d, d2h = arm.time_e2e(e2e_steps, args.warmup if arm.layers == 1 else 2)
    e2e_ms, e2e_serial_ms = reduce_max(e2e_ms), reduce_max(e2e_serial_ms)
    info = dict(S=arm.S, copies=arm.copies, pool_bytes=arm.pool_bytes, layers=arm.layers,
                launches=arm.launches, uses_tc=arm.uses_tc, kernel_bytes=arm.bytes["attention_kernel"],
                fused=arm.fused)
    outs8 = [o.clone() for o in arm.out]               # every layer's output of the last step
    beyond = arm.beyond
    del arm
    torch.cuda.empty_cache()

    fp16 = out_err = None
    if not args.no_fp16:
        arm16 = Arm(w, False, dev, rank, l2)
        arm16.capture()
        ms16 = reduce_max(arm16.time(args.steps, args.warmup, barrier)) / args.steps
        a16avg = reduce_max(arm16.time_kernel(kern_steps, args.warmup))
        fp16 = {"ms_per_step": ms16,
                "value": world * arm16.bytes["step"] / (ms16 * 1e-3) / 1e9,
                "seq_steps_per_s": world * w.batch / (ms16 * 1e-3),
                "attention_kernel_ms": a16avg,
                "attention_kernel_gbs": arm16.bytes["attention_kernel"] / (a16avg * 1e-3) / 1e9,
                "pool_copies": arm16.copies}
        out_err = output_error(outs8, arm16.out)
        out_err["k_elements_beyond_448_scale"], out_err["v_elements_beyond_448_scale"] = beyond
        del arm16
        torch.cuda.empty_cache()

    kname = "attn_tc_kernel" if info["uses_tc"] else "attn_split_kernel"
    layers = info["layers"]
    return {
        "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3", "data": "synthetic",
        "config": {"workload": describe(w, info["S"]),
                   "global_batch": world * w.batch, "kv_dtype": "e4m3 (fp16 MMA, fp32 accumulate)",
                   "l2": (f"rotating {info['copies']} KV pool copies of {info['pool_bytes'] / 1e6:.0f} MB "
                          f"(> 2 x L2 {l2 / 1e6:.0f} MB)") if layers == 1 else
                         (f"{layers} layers' own pools of {info['pool_bytes'] / 1e6:.0f} MB each per step "
                          f"(> 2 x L2 {l2 / 1e6:.0f} MB)"),
                   "parallelism": f"replicas x{world}"},
        "pct_of_peak": 100.0 * gbs / world / peak,
        "seq_steps_per_s": seq_steps,
        "layers_per_step": layers,
        "step_bytes": step_bytes,
        "fp16_arm": fp16,
        "e4m3_speedup_vs_fp16": (fp16["ms_per_step"] / ms) if fp16 else None,
        "e4m3_vs_fp16_output": out_err,
        "step_ms_p10_p50_p90_one_graph_each": pct,
        "step_calls": ("paged_decode_step_e4m3 per layer (the append inside the attention launch, then the "
                       "merge of the partials)") if info["fused"] else
                      "kv_append_e4m3, then paged_decode_attn_e4m3, per layer",
        "launches_per_step": info["launches"],
        "separate_append_ms_per_step": separate_ms,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak,
                     "traffic": profiled_traffic(kname, w.name),
                     "kernel": kname + (" (E4M3, tcgen05)" if info["uses_tc"] else " (E4M3)"),
                     "peak_kind": peak_kind,
                     "attention_kernel_ms": kern_avg,
                     "bytes_per_launch": info["kernel_bytes"],
                     "launches_timed": kern_steps,
                     "decoder": "hardware E4M3 conversion",
                     "bitcast_decoder_ms": bitcast_ms,
                     "bitcast_decoder_kernel": kname,
                     "bitcast_decoder_gbs": info["kernel_bytes"] / (bitcast_ms * 1e-3) / 1e9,
                     "mma_sync_kernel_ms": mma_sync_ms,
                     "fp8_scores_kernel_ms": fp8_qk_ms},
        "e2e": {"value": world * step_bytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms,
                "copies": "own streams, overlapping the neighbouring steps' compute",
                "serial_ms_per_step": e2e_serial_ms},
        "gpu_launches": info["launches"] * args.steps,
        "launch": (f"CUDA graphs of {GRAPH_STEPS} steps" if layers == 1 else "a CUDA graph per step") +
                  (f" (per layer: the fused step call, {info['launches'] // layers} kernel(s)" if info["fused"]
                   else f" (per layer: the append, then the attention call, {info['launches'] // layers} kernels") +
                  "; programmatic dependent launch); e2e: the compute of each step in a CUDA graph, H2D and D2H "
                  "copies on their own streams",
    }


def _entry(line):
    """A workloads entry: the line's figures without the keys it shares with the headline."""
    drop = {"metric", "n_gpus", "steps", "warmup", "higher_is_better", "scaling", "vs_baseline", "data",
            "cpu_baseline"}
    return {k: v for k, v in line.items() if k not in drop}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=None,
                    help="time this workload alone (default: decode, plus the workloads object)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-fp16", action="store_true")
    ap.add_argument("--no-workloads", action="store_true", help="the headline workload only")
    ap.add_argument("--layers", type=int, default=None,
                    help="layers per step of --workload (default: the workload's own; 1 keeps a profiled case small)")
    ap.add_argument("--kernel-hash", choices=sorted(KERNEL_SOURCES),
                    help="print the source hash an ncu summary of that kernel records, and exit")
    args = ap.parse_args()
    if args.kernel_hash:
        print(kernel_source_hash(args.kernel_hash))
        return
    args.warmup = max(3, args.warmup)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    from fp8_paged_kv_e4m3_gb300 import inputs
    w = inputs.get(args.workload or "decode")
    if args.layers is not None:
        w = inputs.get(w.name, layers=max(1, args.layers))
    extras = [] if (args.workload or args.no_workloads) else list(EXTRA_WORKLOADS)

    if args.impl == "reference":
        if rank == 0:
            run_reference(args, w)
        return

    import torch
    import torch.distributed as dist
    from fp8_paged_kv_e4m3_gb300 import build as kbuild, kvq
    kbuild.build()
    kvq.load()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
        barrier = lambda: dist.barrier(device_ids=[local_rank])
    else:
        barrier = None
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size or L2_BYTES_DEFAULT
    peak, peak_kind = _peaks()
    reduce_max = lambda x: max_over_ranks(x, dev, world)

    if w.name == "prefill":
        run_prefill_bench(args, w, dev, l2, rank, world, reduce_max, barrier)
        if world > 1:
            dist.destroy_process_group()
        return

    # the CPU baseline first: its worker processes are spawned, and none of
    # them starts while this process holds busy GPU streams
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline_decode(w)

    with ClockSampler(torch.cuda.current_device()) as clk:
        line = measure(args, w, dev, l2, rank, world, reduce_max, barrier, peak, peak_kind, headline=True)
        workloads = {}
        for name in extras:
            wx = inputs.get(name)
            if wx.name == "prefill":
                workloads[name] = _entry(measure_prefill(args, wx, dev, l2, rank, world, reduce_max, barrier,
                                                         with_cpu=False))
            else:
                workloads[name] = _entry(measure(args, wx, dev, l2, rank, world, reduce_max, barrier, peak,
                                                 peak_kind))
    if rank == 0:
        line["cpu_baseline"] = cpu
        if workloads:
            line["workloads"] = workloads
            line["gpu_launches"] += sum(e["gpu_launches"] for e in workloads.values())
        line["clocks"] = clk.summary()
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
