"""Throughput of one continuous-batching attention step on the GPU.

A step is the whole hot path over one batch: copy-on-write block copies (when
the workload has any), the KV scatter, and ragged causal paged attention
(split-KV decode + combine for single-token rows, the prefill kernel for the
rest).  The headline workload is the pure-decode batch: 256 sequences x 1 new
token, history uniform in [512, 4096], 32/32 heads of 128 dims, block size
16, a 70,000-block pool; its metric is the KV bytes the step must read per
second.  Prefill (16 ragged prompts, 8192 tokens, 32/8 heads) and the mixed
step (240 decodes + two 3976-token chunks) are reported as secondary
measurements.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun every rank runs an independent replica (the path has no
collective); rank 0 prints one JSON line.  ``--impl reference`` times the CPU
oracle on a bounded sample of the same workload.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "decode KV-read GB/s"
BASELINE_METRIC = "decode KV-read GB/s, prefill TFLOP/s, mixed-batch attn tokens/s (1×GB300)"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# ---------------------------------------------------------------------------
# algorithmic work

def kv_bytes(seq_lens, num_kv_heads, head_dim, itemsize=2):
    """K and V bytes a step must read: every live key of every sequence, once."""
    return int(np.sum(np.asarray(seq_lens, dtype=np.int64))) * 2 * num_kv_heads * head_dim * itemsize


def decode_kernel_bytes(lay, rows):
    """Algorithmic bytes of the decode kernel for sequences ``rows``: K/V of every
    live key, the query and output rows, and the block-table entries it reads."""
    seq = lay.seq_lens[rows].astype(np.int64)
    kv = kv_bytes(seq, lay.num_kv_heads, lay.head_dim)
    qo = 2 * len(rows) * lay.num_q_heads * lay.head_dim * 2
    tables = int(np.sum(-(-seq // lay.block_size))) * 4
    return kv + qo + tables


def attention_flops(lay, rows):
    """4 * D FLOPs per visible (query head, key) pair (q.k and p.v)."""
    q = lay.query_lens[rows].astype(np.int64)
    c = (lay.seq_lens[rows] - lay.query_lens[rows]).astype(np.int64)
    pairs = int(np.sum(q * c + q * (q + 1) // 2))
    return 4 * lay.head_dim * lay.num_q_heads * pairs


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm": float(d["hbm_gbs"]), "bf16": float(d["bf16_tflops"]),
                "bf16_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "src": "measured"}
    return {"hbm": FALLBACK_HBM_GBS, "bf16": FALLBACK_BF16_TFLOPS,
            "bf16_sustained": FALLBACK_BF16_TFLOPS, "src": "fallback"}


def source_digest(*names):
    h = hashlib.sha256()
    for n in names:
        h.update(open(os.path.join(ROOT, "paged_kv_cache_133_gb300", "csrc", n), "rb").read())
    return h.hexdigest()[:16]


def measured_traffic(kernel, workload, digest):
    """DRAM bytes per launch from a committed ncu summary, if it matches the current source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    for e in json.load(open(p)):
        if e.get("kernel") == kernel and e.get("workload") == workload and e.get("source") == digest:
            return float(e["dram_bytes_per_launch"])
    return None


# ---------------------------------------------------------------------------
# clocks during the timed region

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    def summary(self):
        if not self.lines:
            return None
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        loaded = [x for x in sm if x > 0.5 * mx] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# GPU side

class Step:
    """Device-resident inputs of one workload and the calls of one step."""

    def __init__(self, lay, dev, seed=0, fused=False, prefix_blocks=0):
        import torch
        import paged_kv_cache_133_gb300 as pa
        self.pa, self.torch, self.lay, self.dev = pa, torch, lay, dev
        self.fused = fused  # one pa_write_kv_attention call instead of pa_write_kv + pa_attention
        self.prefix_blocks = prefix_blocks  # > 0: pa_attention_cascade over a shared prefix
        self.g = workloads.make_tensors(lay, seed=seed, device=dev)
        self.md = {
            "qsl": torch.from_numpy(lay.query_start_loc).to(dev),
            "seq_lens": torch.from_numpy(lay.seq_lens).to(dev),
            "bt": torch.from_numpy(lay.block_tables).to(dev),
            "slots": torch.from_numpy(lay.slot_mapping).to(dev),
            "pairs": torch.from_numpy(np.ascontiguousarray(lay.cow_pairs, np.int32)).to(dev),
        }
        self.out = torch.empty_like(self.g["q"])
        need = pa.workspace_size(lay.num_decode_seqs, lay.num_q_heads, lay.num_kv_heads,
                                 lay.head_dim, lay.max_seq_len)
        if prefix_blocks:
            need = pa.cascade_workspace_size(lay.num_seqs, lay.num_q_heads, lay.num_kv_heads,
                                             lay.head_dim, lay.max_seq_len, prefix_blocks,
                                             lay.block_size)
        self.ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)

    def run(self, attn_events=None, g=None, md=None, out=None):
        pa, lay = self.pa, self.lay
        g = g or self.g
        md = md or self.md
        out = self.out if out is None else out
        if len(lay.cow_pairs):
            pa.copy_blocks(g["k_cache"], g["v_cache"], md["pairs"], err=self.err)
        if self.fused:
            if attn_events is not None:
                attn_events[0].record()
            pa.write_kv_attention(g["q"], g["k"], g["v"], g["k_cache"], g["v_cache"], md["slots"],
                                  md["qsl"], md["seq_lens"], md["bt"],
                                  num_decode_seqs=lay.num_decode_seqs,
                                  max_query_len=lay.max_query_len, max_seq_len=lay.max_seq_len,
                                  scale=lay.scale, out=out, workspace=self.ws, err=self.err)
            if attn_events is not None:
                attn_events[1].record()
            return
        pa.write_kv(g["k"], g["v"], g["k_cache"], g["v_cache"], md["slots"], err=self.err)
        if attn_events is not None:
            attn_events[0].record()
        if self.prefix_blocks:
            pa.attention_cascade(g["q"], g["k_cache"], g["v_cache"], md["qsl"], md["seq_lens"],
                                 md["bt"], prefix_blocks=self.prefix_blocks,
                                 max_seq_len=lay.max_seq_len, scale=lay.scale, out=out,
                                 workspace=self.ws, err=self.err)
            if attn_events is not None:
                attn_events[1].record()
            return
        pa.attention(g["q"], g["k_cache"], g["v_cache"], md["qsl"], md["seq_lens"], md["bt"],
                     num_decode_seqs=lay.num_decode_seqs, max_query_len=lay.max_query_len,
                     max_seq_len=lay.max_seq_len, scale=lay.scale, out=out,
                     workspace=self.ws, err=self.err)
        if attn_events is not None:
            attn_events[1].record()

    def attention(self):
        """The step's attention call alone (the cache already holds the new
        tokens' K/V)."""
        pa, lay, g, md = self.pa, self.lay, self.g, self.md
        pa.attention(g["q"], g["k_cache"], g["v_cache"], md["qsl"], md["seq_lens"], md["bt"],
                     num_decode_seqs=lay.num_decode_seqs, max_query_len=lay.max_query_len,
                     max_seq_len=lay.max_seq_len, scale=lay.scale, out=self.out,
                     workspace=self.ws, err=self.err)


def _barrier(dist_on):
    if dist_on:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(x, dist_on, dev):
    if not dist_on:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def time_device(step, steps, warmup, dist_on, clocks=None):
    """Device time per step (ms) and mean attention-call time (ms) over the timed steps."""
    torch = step.torch
    for _ in range(warmup):
        step.run()
    _barrier(dist_on)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    launches0 = step.pa.kernel_launches()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ctx = clocks if clocks is not None else _Null()
    with ctx:
        start.record()
        for i in range(steps):
            step.run(attn_events=ev[i])
        end.record()
        torch.cuda.synchronize()
    launches = step.pa.kernel_launches() - launches0
    _barrier(dist_on)
    total = start.elapsed_time(end)
    attn = sum(a.elapsed_time(b) for a, b in ev) / steps
    return total / steps, attn, launches


def time_graph(step, calls=10, replays=5):
    """Device time per step (ms) with `calls` steps captured in one CUDA graph
    and replayed (no host launch gaps); best of `replays` replays."""
    torch = step.torch
    for _ in range(3):
        step.run()
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        for _ in range(calls):
            step.run()
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    best = float("inf")
    for _ in range(replays):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        graph.replay()
        b.record()
        torch.cuda.synchronize()
        best = min(best, a.elapsed_time(b) / calls)
    del graph
    return best


class _Null:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False


E2E_COPIES = ("pinned host -> device inputs and device -> pinned host output every step, "
              "double-buffered on copy streams so that they overlap the neighbouring steps")


def time_e2e(step, steps, warmup, dist_on):
    """Per-step time with the step's inputs copied in from pinned host memory
    and the output read back, all inside the timed region.

    The copies are pipelined as a serving loop would: inputs and outputs are
    double-buffered on the device, the next step's inputs go up on a copy
    stream while the current step computes, and the result comes back on a
    second copy stream while the next step computes.  Returns (pipelined ms
    per step, host-to-device bytes, device-to-host bytes, serial ms per step),
    where the serial loop runs copy, step and read-back back to back."""
    torch = step.torch
    host = {k: step.g[k].cpu().pin_memory() for k in ("q", "k", "v")}
    for k in ("qsl", "seq_lens", "bt", "slots", "pairs"):
        host[k] = step.md[k].cpu().pin_memory()
    bufs = []
    for _ in range(2):
        bufs.append({"in": {k: torch.empty_like(step.g[k]) for k in ("q", "k", "v")},
                     "md": {k: torch.empty_like(step.md[k]) for k in step.md},
                     "out": torch.empty_like(step.out),
                     "out_host": torch.empty(step.out.shape, dtype=step.out.dtype).pin_memory()})
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = bufs[0]["out_host"].numel() * bufs[0]["out_host"].element_size()
    comp = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()

    def upload(b):
        for k in ("q", "k", "v"):
            b["in"][k].copy_(host[k], non_blocking=True)
        for k in b["md"]:
            b["md"][k].copy_(host[k], non_blocking=True)

    def compute(b):
        g = {"q": b["in"]["q"], "k": b["in"]["k"], "v": b["in"]["v"],
             "k_cache": step.g["k_cache"], "v_cache": step.g["v_cache"]}
        step.run(g=g, md=b["md"], out=b["out"])

    def serial_step():
        b = bufs[0]
        upload(b)
        compute(b)
        b["out_host"].copy_(b["out"], non_blocking=True)

    def pipelined(n):
        """n steps; returns after queueing everything (the caller syncs)."""
        in_ready, in_free, out_ready, out_free = ([ev(), ev()] for _ in range(4))
        for i in range(2):  # buffers start free
            in_free[i].record(comp)
            out_free[i].record(comp)
        with torch.cuda.stream(up):
            up.wait_stream(comp)
            upload(bufs[0])
            in_ready[0].record(up)
        for i in range(n):
            b, nb = i % 2, (i + 1) % 2
            if i + 1 < n:  # next step's inputs, once its buffer's last reader is done
                with torch.cuda.stream(up):
                    up.wait_event(in_free[nb])
                    upload(bufs[nb])
                    in_ready[nb].record(up)
            comp.wait_event(in_ready[b])
            comp.wait_event(out_free[b])
            compute(bufs[b])
            in_free[b].record(comp)
            with torch.cuda.stream(down):
                down.wait_stream(comp)
                bufs[b]["out_host"].copy_(bufs[b]["out"], non_blocking=True)
                out_free[b].record(down)
        comp.wait_stream(down)
        comp.wait_stream(up)

    for _ in range(warmup):
        serial_step()
    pipelined(max(warmup, 2))
    _barrier(dist_on)
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(steps):
        serial_step()
    e.record()
    torch.cuda.synchronize()
    serial_ms = s.elapsed_time(e) / steps
    _barrier(dist_on)
    torch.cuda.synchronize()
    s.record()
    pipelined(steps)
    e.record()
    torch.cuda.synchronize()
    _barrier(dist_on)
    return s.elapsed_time(e) / steps, h2d, d2h, serial_ms


# ---------------------------------------------------------------------------
# CPU oracle (baseline and reference arm)

def sample_layout(lay, seqs):
    """A layout holding only sequences ``seqs`` of ``lay`` (same lengths and heads),
    with a pool sized exactly for them."""
    cached = lay.cached_lens[seqs]
    queries = lay.query_lens[seqs]
    nb = int(np.sum(-(-lay.seq_lens[seqs].astype(np.int64) // lay.block_size)))
    return workloads.custom_layout(lay.name + "-sample", cached, queries, lay.num_q_heads,
                                   lay.num_kv_heads, lay.head_dim, lay.block_size, nb, 77)


def oracle_step_seconds(sub, seed=0):
    """Wall time of the oracle's scatter + attention on a sample layout (CPU)."""
    import torch
    from oracle import attention as ref
    ts = workloads.make_tensors(sub, seed=seed)
    f = {k: v.to(torch.float64).numpy() for k, v in ts.items()}
    t0 = time.perf_counter()
    kc, vc = ref.write_kv(f["k_cache"], f["v_cache"], f["k"], f["v"], sub.slot_mapping,
                          sub.block_size)
    ref.attention(f["q"], kc, vc, sub.query_start_loc, sub.seq_lens, sub.block_tables,
                  sub.block_size, sub.scale, sub.num_kv_heads)
    return time.perf_counter() - t0


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(lay, budget_s=12.0):
    """Oracle GB/s on a bounded sample of the decode workload (first sequences)."""
    seqs, elapsed, nbytes = [], 0.0, 0
    i = 0
    while elapsed < budget_s and i < lay.num_seqs:
        batch = list(range(i, min(lay.num_seqs, i + 4)))
        sub = sample_layout(lay, np.array(batch))
        elapsed += oracle_step_seconds(sub, seed=i)
        nbytes += kv_bytes(sub.seq_lens, sub.num_kv_heads, sub.head_dim)
        seqs += batch
        i += 4
    return {"value": nbytes / elapsed / 1e9, "unit": "GB/s", "cores": cpu_cores(),
            "kind": "oracle",
            "sample": f"fp64 numpy oracle (scatter + attention) on the first {len(seqs)} of "
                      f"{lay.num_seqs} decode sequences, {elapsed:.1f} s; BLAS threads default"}


def run_reference(args, rank):
    if rank != 0:
        return
    lay = workloads.config_layout(2, args.seed)
    per = 2
    rng = np.random.default_rng(args.seed)
    times, nbytes = [], []
    for it in range(args.warmup + args.steps):
        seqs = np.sort(rng.choice(lay.num_seqs, size=per, replace=False))
        sub = sample_layout(lay, seqs)
        dt = oracle_step_seconds(sub, seed=it)
        if it >= args.warmup:
            times.append(dt)
            nbytes.append(kv_bytes(sub.seq_lens, sub.num_kv_heads, sub.head_dim))
    value = sum(nbytes) / sum(times) / 1e9
    ms = 1e3 * sum(times) / len(times)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": "decode: 256 seqs x 1 token, history U[512,4096], 32q/32kv, "
                               "head_dim 128, block_size 16, 70000-block pool",
                   "sample_per_step": f"{per} random sequences of the 256",
                   "parallelism": "replicas"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": f"{per} sequences per step, fp64 numpy"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------

def shared_prefix_blocks(lay):
    """Leading block-table entries that every sequence shares."""
    tabs = [list(t) for t in lay.tables]
    n = 0
    while all(len(t) > n for t in tabs) and len({t[n] for t in tabs}) == 1:
        n += 1
    return n


def secondary(dev, steps, warmup, peaks):
    """Prefill and mixed-step measurements (device time only)."""
    res = {}
    lay = workloads.config_layout(3, 0)
    st = Step(lay, dev)
    ms, attn_eager, _ = time_device(st, steps, warmup, False)
    msg = time_graph(st)
    attn_flushed = time_call_graph(st.attention, dev)
    # three input sets (168 MB touched per launch, 504 MB in all) in turn
    rot = [st] + [Step(lay, dev, seed=s) for s in (1, 2)]
    attn_ms = _graph_us([x.attention for x in rot], 12) * 1e-3
    fl = attention_flops(lay, np.arange(lay.num_seqs))
    tf = fl / (attn_ms * 1e-3) / 1e12
    del st, rot
    st = Step(lay, dev, fused=True)
    msf, _, _ = time_device(st, steps, warmup, False)
    res["prefill"] = {"workload": "16 prompts (log-uniform 16..2048, sum 8192), 32q/8kv, D 128, bs 16",
                      "fused_ms_per_step": msf, "fused_TFLOP/s_per_step": fl / (msf * 1e-3) / 1e12,
                      "metric": "prefill TFLOP/s", "value": tf, "ms_attention": attn_ms,
                      "ms_attention_eager": attn_eager, "ms_attention_flushed": attn_flushed,
                      "timing": "ms_attention: the attention launch alone, 12 launches in one CUDA "
                                "graph cycling through three input sets (168 MB touched per "
                                "launch, 504 MB in all, so no launch finds its inputs in L2); "
                                "ms_attention_flushed: 8 launches each after a 256 MB write that "
                                "flushes L2 (leaving it full of dirty lines), minus the writes "
                                "alone; ms_attention_eager: events around eager calls, which "
                                "include host launch gaps",
                      "ms_per_step": ms, "graph_ms_per_step": msg, "flops": fl,
                      "roofline": {"bound": "tensor", "achieved": tf, "peak": peaks["bf16"],
                                   "unit": "TFLOP/s", "frac": tf / peaks["bf16"]}}
    del st
    lay = workloads.config_layout(6, 0)
    st = Step(lay, dev)
    ms6, attn6_eager, _ = time_device(st, steps, warmup, False)
    attn6 = _graph_us([st.attention], 8) * 1e-3  # 579 MB of K/V per launch: larger than L2
    fl6 = attention_flops(lay, np.arange(lay.num_seqs))
    tf6 = fl6 / (attn6 * 1e-3) / 1e12
    del st
    st = Step(lay, dev, fused=True)
    msf6, _, _ = time_device(st, steps, warmup, False)
    res["prefix"] = {"workload": "32 prefix-cache hits: cached U[1024,8192], new chunks U[64,512], 32q/8kv, D 128, bs 16",
                     "fused_ms_per_step": msf6, "fused_TFLOP/s_per_step": fl6 / (msf6 * 1e-3) / 1e12,
                     "metric": "prefix-cached prefill TFLOP/s", "value": tf6, "ms_attention": attn6,
                     "ms_attention_eager": attn6_eager,
                     "ms_per_step": ms6, "flops": fl6,
                     "roofline": {"bound": "tensor", "achieved": tf6, "peak": peaks["bf16"],
                                  "unit": "TFLOP/s", "frac": tf6 / peaks["bf16"]}}
    del st
    lay = workloads.config_layout(4, 0)
    st = Step(lay, dev)
    ms, attn_ms, _ = time_device(st, steps, warmup, False)
    attn4g = _graph_us([st.attention], 8) * 1e-3  # 4 GB of K/V per launch: larger than L2
    dec = np.arange(lay.num_decode_seqs)
    pre = np.arange(lay.num_decode_seqs, lay.num_seqs)
    t_dec = decode_kernel_bytes(lay, dec) / (peaks["hbm"] * 1e9)
    t_pre = attention_flops(lay, pre) / (peaks["bf16"] * 1e12)
    t_star = t_dec + t_pre
    t_over = max(t_dec, t_pre)
    ms4g = time_graph(st)
    del st
    st = Step(lay, dev, fused=True)
    ms4f, _, _ = time_device(st, steps, warmup, False)
    del st
    lay5 = workloads.config_layout(5, 0)
    st = Step(lay5, dev)
    ms5, attn5, _ = time_device(st, steps, warmup, False)
    del st
    pb5 = shared_prefix_blocks(lay5)
    st = Step(lay5, dev, prefix_blocks=pb5)
    ms5c, attn5c, _ = time_device(st, steps, warmup, False)
    kvb5 = kv_bytes(lay5.seq_lens, lay5.num_kv_heads, lay5.head_dim)
    res["shared"] = {"workload": "64 seqs sharing a 16384-token prompt (63 copy-on-write pairs), tails U[1,256], 64q/8kv",
                     "metric": "logical KV-read GB/s", "value": kvb5 / (ms5 * 1e-3) / 1e9,
                     "ms_per_step": ms5, "ms_attention": attn5,
                     "cascade": {"prefix_blocks": pb5, "ms_per_step": ms5c, "ms_attention": attn5c,
                                 "value": kvb5 / (ms5c * 1e-3) / 1e9,
                                 "call": "pa_attention_cascade: the shared prefix read once per 128 "
                                         "query rows of a kv head, merged with each sequence's own keys"},
                     "note": "the shared prefix (67 MB of K+V) stays in L2; logical bytes count it once per sequence"}
    res["mixed"] = {"workload": "240 decodes (history U[128,8192]) + 2 chunks of 3976 on 1024/3000 cached, 32q/8kv",
                    "metric": "mixed-batch attn tokens/s", "value": lay.num_tokens / (ms * 1e-3),
                    "ms_per_step": ms, "ms_attention": attn_ms, "fused_ms_per_step": ms4f,
                    "graph_ms_per_step": ms4g,
                    "additive_roofline_ms": t_star * 1e3, "frac": t_star * 1e3 / ms,
                    "overlap_roofline_ms": t_over * 1e3, "overlap_frac": t_over * 1e3 / ms,
                    "ms_attention_graph": attn4g,
                    "attention_overlap_frac": t_over * 1e3 / attn4g,
                    "note": "the decode and prefill kernels run side by side on split SMs, so "
                            "max(decode bytes / HBM peak, prefill FLOPs / bf16 peak) bounds the "
                            "step from below; the additive bound is the serial one"}
    del st
    res["swap"] = swap_leg(dev)
    res["kv_copy"] = kv_copy_leg(dev, peaks)
    res["worked"] = worked_leg(dev)
    return res


def time_call_graph(fn, dev, calls=8, replays=5):
    """Device time (ms) of one `fn` launch with no host gaps and a cold L2.
    Two CUDA graphs are captured: `calls` times (write a 256 MB buffer, twice
    the L2; call fn), and the same writes alone.  Each is replayed between
    events; the launch time is the difference per call (best replay of each)."""
    import torch
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for _ in range(3):
        fn()
    torch.cuda.synchronize()

    def capture(with_fn):
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            for i in range(calls):
                flush.fill_(i & 255)
                if with_fn:
                    fn()
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        return graph

    def best_ms(graph):
        best = float("inf")
        for _ in range(replays):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            graph.replay()
            b.record()
            torch.cuda.synchronize()
            best = min(best, a.elapsed_time(b))
        return best

    g_both, g_flush = capture(True), capture(False)
    t = (best_ms(g_both) - best_ms(g_flush)) / calls
    del g_both, g_flush, flush
    return t


def _graph_us(fns, launches):
    """Microseconds per launch of `launches` calls cycling through `fns`,
    captured in one CUDA graph (no host launch gaps); best of 5 replays."""
    import torch
    for f in fns:
        f()
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        for i in range(launches):
            fns[i % len(fns)]()
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    best = float("inf")
    for _ in range(5):
        a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        graph.replay()
        e.record()
        torch.cuda.synchronize()
        best = min(best, a.elapsed_time(e) * 1e3 / launches)
    del graph
    return best


def kv_copy_leg(dev, peaks, launches=200, sets=8):
    """The scatter and the copy-on-write block copy alone, two ways.

    hbm: every launch works on a different set of inputs and destination
    blocks, 8 sets in rotation whose total (512 MB for the scatter, 1 GB for
    the copy) is several times L2, so each launch streams from and to HBM.
    GB/s count bytes read plus written, against the measured copy peak.  The
    scatter set is the prefill batch's 8192 new tokens (8 kv heads x 128 dims)
    into blocks of 16; the copy set is 1024 block pairs of the same geometry.

    workload: the workloads' own calls (the prefill batch's scatter, the
    shared-prefix batch's 63 copy pairs) replayed back to back: latencies,
    with working sets that stay in L2."""
    import torch
    import paged_kv_cache_133_gb300 as pa
    out = {}
    gen = torch.Generator(device="cpu").manual_seed(77)
    hkv, d, bs, T = 8, 128, 16, 8192
    err = torch.zeros(1, dtype=torch.int32, device=dev)

    # ---- scatter at HBM rate
    nb = sets * T // bs
    kc = torch.zeros((nb, bs, hkv, d), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    perm = torch.randperm(nb, generator=gen)
    tok = torch.arange(T)
    kv_sets = []
    for r in range(sets):
        blocks = perm[r * (T // bs):(r + 1) * (T // bs)]
        slots = (blocks[tok // bs] * bs + tok % bs).to(torch.int32).to(dev)
        k = torch.randn((T, hkv, d), generator=gen).to(torch.bfloat16).to(dev)
        v = torch.randn((T, hkv, d), generator=gen).to(torch.bfloat16).to(dev)
        kv_sets.append((k, v, slots))
    sbytes = 2 * 2 * T * hkv * d * 2  # K and V, read + written
    fns = [lambda k=k, v=v, sl=sl: pa.write_kv(k, v, kc, vc, sl, err=err) for k, v, sl in kv_sets]
    us = _graph_us(fns, launches)
    gbs = sbytes / (us * 1e-6) / 1e9
    out["scatter_hbm"] = {"what": f"{T} tokens x {hkv * d * 2} B of K and of V, {sets} rotating sets "
                                  f"({(sbytes // 2 * sets + kc.numel() * 4) >> 20} MB in all)",
                          "bytes_read_plus_written": sbytes, "us_per_launch": us, "GB/s": gbs,
                          "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm"],
                                       "unit": "GB/s", "frac": gbs / peaks["hbm"]}}
    del kc, vc, kv_sets, fns

    # ---- copy-on-write copy at HBM rate
    npairs = 1024
    nb = sets * 2 * npairs
    kc = torch.zeros((nb, bs, hkv, d), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    perm = torch.randperm(nb, generator=gen)
    pair_sets = []
    for r in range(sets):
        b = perm[r * 2 * npairs:(r + 1) * 2 * npairs]
        pair_sets.append(torch.stack([b[:npairs], b[npairs:]], 1).to(torch.int32).to(dev))
    pair_bytes = 2 * 2 * bs * hkv * d * 2  # K and V block, read + written
    cbytes = npairs * pair_bytes
    fns = [lambda p=p: pa.copy_blocks(kc, vc, p, err=err) for p in pair_sets]
    us = _graph_us(fns, 10 * sets)
    gbs = cbytes / (us * 1e-6) / 1e9
    out["copy_blocks_hbm"] = {"what": f"{npairs} pairs x {pair_bytes // 2 >> 10} KB of K+V, {sets} rotating "
                                      f"sets over {nb} blocks ({(kc.numel() * 4) >> 20} MB)",
                              "bytes_read_plus_written": cbytes, "us_per_launch": us, "GB/s": gbs,
                              "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm"],
                                           "unit": "GB/s", "frac": gbs / peaks["hbm"]}}
    del kc, vc, pair_sets, fns
    torch.cuda.synchronize()
    assert int(err.item()) == 0

    # ---- the workloads' own calls: latency, L2-resident
    lay = workloads.config_layout(3, 0)
    st = Step(lay, dev)
    g, md = st.g, st.md
    us = _graph_us([lambda: pa.write_kv(g["k"], g["v"], g["k_cache"], g["v_cache"], md["slots"],
                                        err=st.err)], launches)
    out["scatter_workload"] = {"what": "the prefill batch's scatter: 8192 tokens x 2 KB of K and of V",
                               "us_per_launch": us,
                               "note": "replayed back to back from a CUDA graph; the 67 MB set stays in L2"}
    lay5 = workloads.config_layout(5, 0)
    st5 = Step(lay5, dev)
    g5, md5 = st5.g, st5.md
    us = _graph_us([lambda: pa.copy_blocks(g5["k_cache"], g5["v_cache"], md5["pairs"], err=st5.err)],
                   launches)
    out["copy_blocks_workload"] = {"what": "the shared-prefix batch's 63 copy-on-write pairs x 64 KB of K+V",
                                   "us_per_launch": us,
                                   "note": "8 MB moved: launch latency, not bandwidth, sets the time"}
    del st, st5
    return out


def worked_leg(dev, launches=100):
    """Latency of the worked B/C/A step (2 decodes + a 5-token prompt, 4/4
    heads, D 64, block size 4): scatter + attention, from a CUDA graph."""
    lay = workloads.config_layout(1, 0)
    st = Step(lay, dev)
    us = time_graph(st, calls=launches) * 1e3
    ms, _, _ = time_device(st, 50, 5, False)
    return {"workload": "worked B/C/A step: T=7, query_start_loc [0,1,2,7], 4/4 heads, D 64, bs 4",
            "us_per_step_graph": us, "us_per_step_eager": ms * 1e3,
            "note": "pa_write_kv + pa_attention (decode and prefill kernels side by side); "
                    "graph replay removes host launch gaps"}


class Fp8Step:
    """The decode workload with an 8-bit (E4M3) pool: pa_write_kv_fp8 + pa_attention_fp8."""

    K_SCALE, V_SCALE = 0.03, 0.05

    def __init__(self, lay, dev, seed=0):
        import torch
        import paged_kv_cache_133_gb300 as pa
        self.pa, self.torch, self.lay = pa, torch, lay
        g = workloads.make_tensors(lay, seed=seed, device=dev)
        n_slots = lay.num_blocks * lay.block_size
        rows = lambda c: c.view(n_slots, lay.num_kv_heads, lay.head_dim)
        self.kc = torch.empty(g["k_cache"].shape, dtype=torch.uint8, device=dev)
        self.vc = torch.empty_like(self.kc)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        all_slots = torch.arange(n_slots, dtype=torch.int32, device=dev)
        pa.write_kv_fp8(rows(g["k_cache"]), rows(g["v_cache"]), self.kc, self.vc, all_slots,
                        self.K_SCALE, self.V_SCALE, err=self.err)
        self.q, self.k, self.v = g["q"], g["k"], g["v"]
        del g
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        self.md = {
            "qsl": torch.from_numpy(lay.query_start_loc).to(dev),
            "seq_lens": torch.from_numpy(lay.seq_lens).to(dev),
            "bt": torch.from_numpy(lay.block_tables).to(dev),
            "slots": torch.from_numpy(lay.slot_mapping).to(dev),
        }
        self.out = torch.empty_like(self.q)
        need = pa.workspace_size(lay.num_seqs, lay.num_q_heads, lay.num_kv_heads, lay.head_dim,
                                 lay.max_seq_len)
        self.ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)

    def run(self, attn_events=None):
        pa, md = self.pa, self.md
        pa.write_kv_fp8(self.k, self.v, self.kc, self.vc, md["slots"], self.K_SCALE, self.V_SCALE,
                        err=self.err)
        if attn_events is not None:
            attn_events[0].record()
        pa.attention_fp8(self.q, self.kc, self.vc, md["qsl"], md["seq_lens"], md["bt"],
                         k_scale=self.K_SCALE, v_scale=self.V_SCALE,
                         max_seq_len=self.lay.max_seq_len, scale=self.lay.scale, out=self.out,
                         workspace=self.ws, err=self.err)
        if attn_events is not None:
            attn_events[1].record()


def fp8_leg(dev, steps, warmup, peaks, bf16_ms):
    """Decode over an 8-bit pool: KV-read GB/s of the codes and tokens/s against bf16."""
    lay = workloads.config_layout(2, 0)
    st = Fp8Step(lay, dev)
    ms, attn_ms, _ = time_device(st, steps, warmup, False)
    kvb = kv_bytes(lay.seq_lens, lay.num_kv_heads, lay.head_dim, itemsize=1)
    algo = kvb + 2 * lay.num_seqs * lay.num_q_heads * lay.head_dim * 2 + \
        int(np.sum(-(-lay.seq_lens.astype(np.int64) // lay.block_size))) * 4
    ach = algo / (attn_ms * 1e-3) / 1e9
    res = {"workload": "decode batch (256 seqs, history U[512,4096], 32q/32kv, D 128, bs 16) on an E4M3 pool",
           "metric": "decode KV-read GB/s (8-bit cache)", "value": kvb / (ms * 1e-3) / 1e9,
           "ms_per_step": ms, "ms_attention": attn_ms, "kv_bytes_per_step": kvb,
           "tokens_per_s": lay.num_tokens / (ms * 1e-3),
           "speedup_vs_bf16_step": bf16_ms / ms,
           "roofline": {"bound": "hbm", "achieved": ach, "peak": peaks["hbm"], "unit": "GB/s",
                        "frac": ach / peaks["hbm"]}}
    del st
    return res


def swap_leg(dev, iters=20, warmup=3, pairs=4096, seed=0):
    """Block swap between the device pool and a pool in page-locked host memory.

    ``pairs`` random blocks of the decode pool's shape (bs 16, 8 KV heads, D 128:
    64 KiB of K+V per block) go device -> host, then host -> device into other
    blocks.  The link's own ceiling is one contiguous DMA copy of the same bytes
    (cudaMemcpyAsync through ``copy_``), timed the same way in each direction.
    """
    import torch
    import paged_kv_cache_133_gb300 as pa
    rng = np.random.default_rng(seed)
    bs, hkv, d = 16, 8, 128
    n_dev, n_host = 3 * pairs, 2 * pairs
    shape = (bs, hkv, d)
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    dk = torch.randn((n_dev,) + shape, generator=g, device=dev, dtype=torch.bfloat16)
    dv = torch.randn((n_dev,) + shape, generator=g, device=dev, dtype=torch.bfloat16)
    hk = torch.empty((n_host,) + shape, dtype=torch.bfloat16, pin_memory=True)
    hv = torch.empty((n_host,) + shape, dtype=torch.bfloat16, pin_memory=True)
    src = rng.permutation(n_dev)[:pairs]
    host = rng.permutation(n_host)[:pairs]
    back = rng.permutation(n_dev)[:pairs]
    p_out = torch.from_numpy(np.stack([src, host], 1).astype(np.int32)).to(dev)
    p_in = torch.from_numpy(np.stack([host, back], 1).astype(np.int32)).to(dev)
    nbytes = 2 * pairs * bs * hkv * d * 2
    st = torch.cuda.current_stream()

    def timed(fn):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        for _ in range(iters):
            fn()
        b.record(st)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / iters

    ms_out = timed(lambda: pa.swap_blocks(dk, dv, hk, hv, p_out))
    ms_in = timed(lambda: pa.swap_blocks(hk, hv, dk, dv, p_in))
    flat_d = dk[:2 * pairs].view(-1)
    flat_h = hk.view(-1)
    ms_d2h = timed(lambda: flat_h.copy_(flat_d, non_blocking=True))
    ms_h2d = timed(lambda: flat_d.copy_(flat_h, non_blocking=True))
    gbs = lambda ms: nbytes / (ms * 1e-3) / 1e9
    res = {"workload": f"{pairs} random blocks of 16 x 8 x 128 bf16 (K+V {nbytes >> 20} MiB) between HBM and pinned host memory",
           "metric": "swap GB/s (K+V bytes moved)",
           "swap_out": {"ms": ms_out, "GB/s": gbs(ms_out), "dma_contiguous_GB/s": gbs(ms_d2h),
                        "frac_of_dma": ms_d2h / ms_out},
           "swap_in": {"ms": ms_in, "GB/s": gbs(ms_in), "dma_contiguous_GB/s": gbs(ms_h2d),
                       "frac_of_dma": ms_h2d / ms_in}}
    del dk, dv, hk, hv
    return res


def run_other(args, dev, peaks, rank, world, dist_on):
    """One JSON line for the prefill, mixed, shared-prefix or 8-bit decode workload."""
    if args.workload == "decode_fp8":
        run_fp8(args, dev, peaks, rank, world, dist_on)
        return
    cfg = {"prefill": 3, "mixed": 4, "shared": 5, "prefix": 6}[args.workload]
    lay = workloads.config_layout(cfg, args.seed)
    pb = shared_prefix_blocks(lay) if args.cascade and args.workload == "shared" else 0
    step = Step(lay, dev, seed=args.seed + rank, fused=args.fused, prefix_blocks=pb)
    clocks = ClockSampler(int(os.environ.get("LOCAL_RANK", "0")))
    ms, attn_ms, launches = time_device(step, args.steps, args.warmup, dist_on, clocks)
    ms = _max_over_ranks(ms, dist_on, dev)
    attn_ms = _max_over_ranks(attn_ms, dist_on, dev)
    e2e_ms, h2d, d2h, e2e_serial_ms = time_e2e(step, args.steps, args.warmup, dist_on)
    e2e_serial_ms = _max_over_ranks(e2e_serial_ms, dist_on, dev)
    e2e_ms = _max_over_ranks(e2e_ms, dist_on, dev)
    # the attention launch alone, from a CUDA graph with L2 flushed before each
    attn_graph = None
    if not pb and not args.fused and args.workload in ("prefill", "prefix", "mixed"):
        calls = [step.attention]
        if args.workload == "prefill":  # 168 MB per launch: three input sets in turn
            calls += [Step(lay, dev, seed=args.seed + rank + 100 * s).attention for s in (1, 2)]
        attn_graph = _max_over_ranks(_graph_us(calls, 12) * 1e-3, dist_on, dev)
    if rank != 0:
        return
    dec = np.arange(lay.num_decode_seqs)
    pre = np.arange(lay.num_decode_seqs, lay.num_seqs)
    if args.workload in ("prefill", "prefix"):
        fl = attention_flops(lay, pre)
        value, unit = world * fl / (ms * 1e-3) / 1e12, "TFLOP/s"
        metric = "prefill TFLOP/s" if args.workload == "prefill" else "prefix-cached prefill TFLOP/s"
        ach = fl / ((attn_graph or attn_ms) * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": ach, "peak": peaks["bf16"], "unit": "TFLOP/s",
                "frac": ach / peaks["bf16"], "ms_per_launch": attn_graph or attn_ms,
                "launch_timing": ("CUDA graph of back-to-back launches, inputs larger than L2"
                                  + (" (three input sets in turn)" if args.workload == "prefill"
                                     else "") if attn_graph else "eager events")}
        e2e_v = world * fl / (e2e_ms * 1e-3) / 1e12
    elif args.workload == "mixed":
        value, unit, metric = world * lay.num_tokens / (ms * 1e-3), "tokens/s", "mixed-batch attn tokens/s"
        t_star = decode_kernel_bytes(lay, dec) / (peaks["hbm"] * 1e9) + \
            attention_flops(lay, pre) / (peaks["bf16"] * 1e12)
        t_over = max(decode_kernel_bytes(lay, dec) / (peaks["hbm"] * 1e9),
                     attention_flops(lay, pre) / (peaks["bf16"] * 1e12))
        roof = {"bound": "hbm+tensor (additive)", "achieved_ms": attn_ms, "ideal_ms": t_star * 1e3,
                "frac": t_star * 1e3 / attn_ms, "attention_graph_ms": attn_graph,
                "overlap_bound_ms": t_over * 1e3,
                "overlap_frac": t_over * 1e3 / (attn_graph or attn_ms)}
        e2e_v = world * lay.num_tokens / (e2e_ms * 1e-3)
    else:
        kvb = kv_bytes(lay.seq_lens, lay.num_kv_heads, lay.head_dim)
        value, unit, metric = world * kvb / (ms * 1e-3) / 1e9, "GB/s", "logical KV-read GB/s"
        ach = decode_kernel_bytes(lay, dec) / (attn_ms * 1e-3) / 1e9
        roof = {"bound": "hbm (logical bytes; the shared prefix is L2-resident)", "achieved": ach,
                "peak": peaks["hbm"], "unit": "GB/s", "frac": ach / peaks["hbm"]}
        e2e_v = world * kvb / (e2e_ms * 1e-3) / 1e9
    line = {"metric": metric, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": lay.name, "ms_attention": attn_ms, "fused": bool(args.fused),
                       "cascade_prefix_blocks": pb,
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "roofline": roof, "cpu_baseline": None,
            "e2e": {"value": e2e_v, "unit": unit, "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "copies": E2E_COPIES,
                    "serial_ms_per_step": e2e_serial_ms},
            "gpu_launches": launches, "clocks": clocks.summary()}
    print(json.dumps(line), flush=True)


def run_fp8(args, dev, peaks, rank, world, dist_on):
    """One JSON line for the decode workload on an 8-bit (E4M3) pool."""
    lay = workloads.config_layout(2, args.seed)
    if args.decode_seqs:
        lay = sample_layout(lay, np.arange(min(args.decode_seqs, lay.num_seqs)))
        lay.num_blocks = int(lay.num_blocks * 1.1) + 1
    step = Fp8Step(lay, dev, seed=args.seed + rank)
    clocks = ClockSampler(int(os.environ.get("LOCAL_RANK", "0")))
    ms, attn_ms, launches = time_device(step, args.steps, args.warmup, dist_on, clocks)
    ms = _max_over_ranks(ms, dist_on, dev)
    attn_ms = _max_over_ranks(attn_ms, dist_on, dev)
    if int(step.err.item()):
        raise RuntimeError(f"device error flag {int(step.err.item())}")
    if rank != 0:
        return
    kvb = kv_bytes(lay.seq_lens, lay.num_kv_heads, lay.head_dim, itemsize=1)
    algo = kvb + 2 * lay.num_seqs * lay.num_q_heads * lay.head_dim * 2 + \
        int(np.sum(-(-lay.seq_lens.astype(np.int64) // lay.block_size))) * 4
    ach = algo / (attn_ms * 1e-3) / 1e9
    line = {"metric": "decode KV-read GB/s (8-bit cache)", "value": world * kvb / (ms * 1e-3) / 1e9,
            "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3 cache, fp16 products", "data": "synthetic",
            "config": {"workload": lay.name + " (E4M3 pool)", "ms_attention": attn_ms,
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "roofline": {"bound": "hbm", "achieved": ach, "peak": peaks["hbm"], "unit": "GB/s",
                         "frac": ach / peaks["hbm"]},
            "cpu_baseline": None, "gpu_launches": launches, "clocks": clocks.summary()}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--fused", action="store_true",
                    help="time pa_write_kv_attention instead of pa_write_kv + pa_attention")
    ap.add_argument("--workload",
                    choices=["decode", "prefill", "mixed", "shared", "prefix", "decode_fp8"],
                    default="decode",
                    help="decode is the headline; the others print their own metric")
    ap.add_argument("--cascade", action="store_true",
                    help="shared workload: pa_attention_cascade over the common prefix blocks")
    ap.add_argument("--decode-seqs", type=int, default=0,
                    help="profile case: only the first N decode sequences, pool sized to fit")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        run_reference(args, rank)
        return

    import torch
    import paged_kv_cache_133_gb300 as pa
    pa.load()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_on = world > 1
    if dist_on:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    peaks = load_peaks()
    if args.workload != "decode":
        run_other(args, dev, peaks, rank, world, dist_on)
        return
    lay = workloads.config_layout(2, args.seed)
    if args.decode_seqs:
        lay = sample_layout(lay, np.arange(min(args.decode_seqs, lay.num_seqs)))
        lay.num_blocks = int(lay.num_blocks * 1.1) + 1
    step = Step(lay, dev, seed=args.seed + rank)
    clocks = ClockSampler(local)
    ms, attn_ms, launches = time_device(step, args.steps, args.warmup, dist_on, clocks)
    ms = _max_over_ranks(ms, dist_on, dev)
    attn_ms = _max_over_ranks(attn_ms, dist_on, dev)
    err = int(step.err.item())
    if err:
        raise RuntimeError(f"device error flag {err} during the bench")
    kvb = kv_bytes(lay.seq_lens, lay.num_kv_heads, lay.head_dim)
    value = world * kvb / (ms * 1e-3) / 1e9
    algo = decode_kernel_bytes(lay, np.arange(lay.num_decode_seqs))
    achieved = algo / (attn_ms * 1e-3) / 1e9
    digest = source_digest("decode.cu")
    traffic = measured_traffic("decode_kernel", "decode", digest)
    e2e_ms, h2d, d2h, e2e_serial_ms = time_e2e(step, args.steps, args.warmup, dist_on)
    e2e_serial_ms = _max_over_ranks(e2e_serial_ms, dist_on, dev)
    e2e_ms = _max_over_ranks(e2e_ms, dist_on, dev)
    step.fused = True  # the same step through pa_write_kv_attention, for reference
    fused_ms, _, _ = time_device(step, max(args.steps // 4, 1), args.warmup, dist_on)
    fused_ms = _max_over_ranks(fused_ms, dist_on, dev)
    step.fused = False
    sec = None
    if not args.no_secondary:
        del step
        torch.cuda.empty_cache()
        sec = secondary(dev, args.steps, args.warmup, peaks)
        torch.cuda.empty_cache()
        sec["decode_fp8"] = fp8_leg(dev, args.steps, args.warmup, peaks, ms)
    if rank != 0:
        if dist_on:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    cpu = None if args.no_cpu_baseline else cpu_baseline(lay)
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "decode: 256 seqs x 1 token, history U[512,4096], 32q/32kv, "
                               "head_dim 128, block_size 16, 70000-block pool (seed %d)" % args.seed,
                   "kv_bytes_per_step": kvb, "l2": "inputs larger than L2 (18 GB pool, 10 GB read per step)",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "fused_ms_per_step": fused_ms,
                   "baseline_metric": BASELINE_METRIC},
        "roofline": {"bound": "hbm", "kernel": "decode_kernel (+combine when split)",
                     "achieved": achieved, "peak": peaks["hbm"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm"], "traffic": traffic,
                     "peak_source": peaks["src"], "algorithmic_bytes_per_launch": algo,
                     "ms_per_launch": attn_ms},
        "cpu_baseline": cpu,
        "e2e": {"value": world * kvb / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "copies": E2E_COPIES, "serial_ms_per_step": e2e_serial_ms},
        "gpu_launches": launches,
        "clocks": clocks.summary(),
    }
    if sec:
        line["secondary"] = sec
    print(json.dumps(line), flush=True)
    if dist_on:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
