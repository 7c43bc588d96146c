"""Benchmark: one decode step of the paged quantized-KV path on GB300.

A step is one pass of the whole hot path over one batch: quantize-append of
the step's new tokens (kvq_append) and split-K fused-dequant decode attention
with its merge (kvq_decode_attn: one launch), for every layer of the
workload.  Pages come from the library's host allocator (scattered ids).
Inputs are resident in HBM when the timed region starts; L2 is flushed (a
256 MB write) before every timed step, outside the timed events.

Default workload (N=1): the Llama-3-8B-shaped INT8 layer -- 32 sequences with
lengths uniform in [512, 4096], 32 query / 8 KV heads, head_dim 128, page 16
-- decode step plus 1-token append.  --config selects another workload.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config C] [--impl kvq|reference]

Prints one JSON line (rank 0).  --impl reference times the CPU oracle (the
only reference implementation there is) on the host cores, on a bounded
sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import kvq_inputs as inp  # noqa: E402

METRIC = "paged quantized-KV decode attn GB/s (% of 8 TB/s HBM); append tokens/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 256 << 20


# ---------------------------------------------------------------- accounting
def code_meta_bytes(w: inp.Workload):
    """(code bytes, scale+zero bytes) per (token, KV head) for one of K / V."""
    if w.scheme == "int4":
        return w.head_dim // 2, (w.head_dim // w.group) * 4
    return w.head_dim, 4


def step_plan(w: inp.Workload, lens: np.ndarray):
    """Tokens appended per sequence in one step and the lengths after it."""
    n_new = w.prefill_chunk if w.cid == 5 else w.append_tokens
    n_new = np.minimum(lens, n_new).astype(np.int64)
    return n_new


def algorithmic_bytes(w: inp.Workload, lens: np.ndarray, n_new: np.ndarray) -> dict:
    """Bytes the method must move per step (per layer x layers): never padding."""
    cb, mb = code_meta_bytes(w)
    H, D, P = w.kv_heads, w.head_dim, w.page_size
    B, Hq = len(lens), w.q_heads
    tokens = int(lens.sum())
    kv = tokens * 2 * H * (cb + mb)
    table = int(((lens + P - 1) // P).sum()) * 4
    q = B * Hq * D * 2
    out = B * Hq * D * 4
    decode = kv + table + q + out + B * 4
    T = int(n_new.sum())
    append = T * (2 * H * D * 2 + 8 + 2 * H * (cb + mb))
    L = w.layers
    return {"decode_partial": (kv + table + q + B * 4 + out) * L, "decode": decode * L,
            "append": append * L, "step": (decode + append) * L, "append_tokens": T * L,
            "kv_bytes": kv * L}


def append_line(nb: dict, w: inp.Workload, k1_mean_ms: float, peak_gbs: float) -> dict:
    """The quantize-append launch of a step on its own: tokens per second,
    and its algorithmic bytes (bf16 K/V read, slots read, codes and scales
    written) per second against the HBM peak."""
    T = nb["append_tokens"] // w.layers      # tokens per launch
    b = nb["append"] // w.layers             # algorithmic bytes per launch
    t = k1_mean_ms * 1e-3
    return {"kernel": "append_kernel (quantize-append)", "tokens_per_launch": T,
            "mean_launch_us": round(k1_mean_ms * 1e3, 3), "tokens_per_s": round(T / t, 1),
            "algorithmic_bytes_per_launch": b, "achieved_gbs": round(b / t / 1e9, 2),
            "roofline_tokens_per_s": round(peak_gbs * 1e9 / (b / T), 1) if T else None,
            "frac": round(b / t / 1e9 / peak_gbs, 4)}


def measured_hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def traffic_record(cid: int):
    """DRAM bytes per decode_partial launch from a committed ncu capture, if it
    was taken on the current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "decode_traffic.json")
    try:
        with open(p) as f:
            rec = json.load(f)
    except Exception:
        return None
    import hashlib
    h = hashlib.sha256()
    for name in ("kvq_decode.cuh", "kvq_device.cuh", "kvq_internal.h"):
        with open(os.path.join(ROOT, "dynamically_quantized_paged_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    if rec.get("kernel_source_sha256") != h.hexdigest():
        return None
    entry = rec.get("workloads", {}).get(str(cid))
    return None if entry is None else entry.get("dram_bytes_per_launch")


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest value of x over all ranks (timing: the slowest rank sets
    the job's time).  Uses whatever process group is initialized."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_rank_step: int, world: int, ms_per_step: float) -> float:
    """Whole-job GB/s: every rank moves its own batch (weak scaling) in the
    time of the slowest rank."""
    return world * bytes_per_rank_step / (ms_per_step * 1e-3) / 1e9


# ---------------------------------------------------------------- clocks
STAGE_ALIGN = 256  # byte alignment of each tensor in the host staging buffer


def stage_layout(tensors) -> tuple[list, int]:
    """Byte offsets of `tensors` packed end to end in one staging buffer,
    each at a STAGE_ALIGN-byte boundary, and the buffer's total size."""
    offs, total = [], 0
    for t in tensors:
        total = (total + STAGE_ALIGN - 1) // STAGE_ALIGN * STAGE_ALIGN
        offs.append(total)
        total += t.numel() * t.element_size()
    return offs, total


def stage_view(buf, t, off: int):
    """The region of the uint8 buffer `buf` at byte offset `off`, viewed with
    the dtype and shape of `t`."""
    return buf[off:off + t.numel() * t.element_size()].view(t.dtype).view(t.shape)


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def wait_first(self, timeout_s: float = 10.0) -> None:
        """Returns once the sampler has produced a line (its start-up is done)."""
        t0 = time.time()
        while self.proc is not None and not self.lines and time.time() - t0 < timeout_s:
            time.sleep(0.05)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- the GPU arm
class Bench:
    def __init__(self, w: inp.Workload, device, rank: int):
        import torch
        import dynamically_quantized_paged_gb300 as kvq
        self.torch, self.kvq = torch, kvq
        self.w, self.dev, self.rank = w, device, rank
        self.lens = inp.seq_lens(w)
        self.n_new = step_plan(w, self.lens)
        B, P = w.batch, w.page_size
        need = inp.pages_needed(self.lens, P)
        self.max_pages = int(need.max())
        num_pages = int(need.sum()) + 16
        # page allocation through the library's host allocator (scattered ids)
        self.alloc = kvq.PageAllocator(num_pages, seed=w.seed * 7919 + rank)
        bt = np.full((B, self.max_pages), -1, np.int32)
        for b in range(B):
            bt[b, :need[b]] = self.alloc.alloc(int(need[b]))
        self.bt_host = bt
        dev = device
        self.bt = torch.from_numpy(bt).to(dev)
        self.seq_lens = torch.from_numpy(self.lens).to(dev)
        self.caches, self.q, self.k_new, self.v_new = [], [], [], []
        new_slots = np.concatenate([inp.slots(bt, b, np.arange(self.lens[b] - self.n_new[b], self.lens[b]), P)
                                    for b in range(B)])
        self.slots_new = torch.from_numpy(new_slots).to(dev)
        for layer in range(w.layers):
            c = kvq.PagedKVCache(w.scheme, num_pages, P, w.kv_heads, w.head_dim, device=dev, zero_init=False)
            ks, vs = [], []
            for b in range(B):
                L, n = int(self.lens[b]), int(self.n_new[b])
                for s0 in range(0, L - n, w.prefill_chunk):     # prefill (untimed)
                    s1 = min(L - n, s0 + w.prefill_chunk)
                    k, v = self._rows(layer, b, s0, s1)
                    sl = inp.slots(bt, b, np.arange(s0, s1), P)
                    kvq.append(c, torch.from_numpy(sl).to(dev), k, v)
                k, v = self._rows(layer, b, L - n, L)
                ks.append(k)
                vs.append(v)
            self.k_new.append(torch.cat(ks))
            self.v_new.append(torch.cat(vs))
            self.caches.append(c)
            self.q.append(torch.from_numpy(inp.queries(w, layer).view(np.int16)).to(dev))
        self.out = torch.empty((B, w.q_heads, w.head_dim), dtype=torch.float32, device=dev)
        self.ws = kvq.alloc_workspace(self.caches[0], B, w.q_heads, self.max_pages, device=dev)
        self.flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        torch.cuda.synchronize(dev)
        st = kvq.last_device_error()
        if st != kvq.OK:
            raise RuntimeError(f"set-up failed: {kvq.status_string(st)}")
        self.launches_per_step = 2 * w.layers  # quantize-append + fused decode per layer

    def _rows(self, layer, b, s0, s1):
        k, v = inp.kv_rows(self.w, layer, b, s0, s1)
        t = self.torch
        return (t.from_numpy(k.view(np.int16)).to(self.dev), t.from_numpy(v.view(np.int16)).to(self.dev))

    def step(self, events=None, q=None, k_new=None, v_new=None, slots=None, bt=None, lens=None, out=None,
             stream=None):
        kvq = self.kvq
        q = q or self.q
        k_new, v_new = k_new or self.k_new, v_new or self.v_new
        slots = self.slots_new if slots is None else slots
        bt = self.bt if bt is None else bt
        lens = self.seq_lens if lens is None else lens
        out = self.out if out is None else out
        for layer, c in enumerate(self.caches):
            if events is not None:
                events[layer][2].record()
            kvq.append(c, slots, k_new[layer], v_new[layer], stream=stream)
            if events is not None:
                events[layer][0].record()
            kvq.decode_attn(c, q[layer], bt, lens, out, self.ws, stream=stream)  # one launch, splits merged in place
            if events is not None:
                events[layer][1].record()

    def run(self, steps: int, warmup: int, barrier):
        torch = self.torch
        for _ in range(warmup):
            self.flush.zero_()
            self.step()
        torch.cuda.synchronize(self.dev)
        st = self.kvq.last_device_error()
        if st != self.kvq.OK:
            raise RuntimeError(f"warm-up failed: {self.kvq.status_string(st)}")
        E = torch.cuda.Event
        step_ev = [(E(enable_timing=True), E(enable_timing=True)) for _ in range(steps)]
        # per layer: decode start (= append end), decode end, append start
        k2_ev = [[tuple(E(enable_timing=True) for _ in range(3)) for _ in self.caches] for _ in range(steps)]
        barrier()
        torch.cuda.synchronize(self.dev)
        t0 = time.perf_counter()
        for i in range(steps):
            self.flush.zero_()
            step_ev[i][0].record()
            self.step(events=k2_ev[i])
            step_ev[i][1].record()
        torch.cuda.synchronize(self.dev)
        barrier()
        wall = time.perf_counter() - t0
        status = self.kvq.last_device_error()
        step_ms = [a.elapsed_time(b) for a, b in step_ev]
        k2_ms = [ev[0].elapsed_time(ev[1]) for row in k2_ev for ev in row]
        k1_ms = [ev[2].elapsed_time(ev[0]) for row in k2_ev for ev in row]
        return step_ms, k2_ms, k1_ms, wall, status

    def run_graph(self, steps: int, barrier):
        """The same step recorded once in a CUDA graph (all layers' append and
        decode launches) and replayed: what a serving loop that replays its
        decode step pays, without per-launch host overhead.  The L2 flush
        stays outside the graph and outside the timed events."""
        torch = self.torch
        stream = torch.cuda.Stream(self.dev)
        stream.wait_stream(torch.cuda.current_stream(self.dev))
        with torch.cuda.stream(stream):
            self.step(stream=stream)
        torch.cuda.synchronize(self.dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            self.step(stream=stream)
        for _ in range(3):
            self.flush.zero_()
            graph.replay()
        torch.cuda.synchronize(self.dev)
        E = torch.cuda.Event
        evs = [(E(enable_timing=True), E(enable_timing=True)) for _ in range(steps)]
        barrier()
        torch.cuda.synchronize(self.dev)
        for i in range(steps):
            self.flush.zero_()
            evs[i][0].record()
            graph.replay()
            evs[i][1].record()
        torch.cuda.synchronize(self.dev)
        barrier()
        return [a.elapsed_time(b) for a, b in evs], self.kvq.last_device_error()

    def run_e2e(self, steps: int, warmup: int):
        """The same step through the public API with HOST buffers: a pinned host
        -> device copy of the step's inputs and a device -> host copy of the
        output inside the timed region.  The inputs (queries, new keys and
        values, slots, block tables, lengths) are staged in one pinned buffer
        at 256-byte aligned offsets and go over in ONE copy; the device
        tensors the calls take are views of its device twin."""
        torch = self.torch
        srcs = list(self.q) + list(self.k_new) + list(self.v_new) + [self.slots_new, self.bt, self.seq_lens]
        offs, total = stage_layout(srcs)
        h_buf = torch.empty(total, dtype=torch.uint8).pin_memory()
        d_buf = torch.empty(total, dtype=torch.uint8, device=self.dev)
        for t, off in zip(srcs, offs):
            stage_view(h_buf, t, off).copy_(t.cpu())
        d_views = [stage_view(d_buf, t, off) for t, off in zip(srcs, offs)]
        nl = len(self.q)
        d_q, d_k, d_v = d_views[:nl], d_views[nl:2 * nl], d_views[2 * nl:3 * nl]
        d_slots, d_bt, d_lens = d_views[3 * nl:]
        h_out = torch.empty(self.out.shape, dtype=torch.float32).pin_memory()
        h2d = total
        d2h = h_out.numel() * 4

        def one():
            d_buf.copy_(h_buf, non_blocking=True)
            self.step(q=d_q, k_new=d_k, v_new=d_v, slots=d_slots, bt=d_bt, lens=d_lens)
            h_out.copy_(self.out, non_blocking=True)

        for _ in range(warmup):
            self.flush.zero_()
            one()
        torch.cuda.synchronize(self.dev)
        E = torch.cuda.Event
        evs = [(E(enable_timing=True), E(enable_timing=True)) for _ in range(steps)]
        for i in range(steps):
            self.flush.zero_()
            evs[i][0].record()
            one()
            evs[i][1].record()
        torch.cuda.synchronize(self.dev)
        return [a.elapsed_time(b) for a, b in evs], h2d, d2h


def describe(w: inp.Workload) -> str:
    L = w.lengths
    if L[0] == "fixed":
        lens = f"{L[1]} tokens"
    elif L[0] == "uniform":
        lens = f"lengths U[{L[1]},{L[2]}]"
    else:
        lens = f"lengths lognormal(median {L[1]}, sigma {L[2]}) clipped [{L[3]},{L[4]}]"
    step = f"{w.prefill_chunk}-token chunked append + split-K decode" if w.cid == 5 else \
        "decode step + 1-token append"
    return (f"{w.name}: {w.layers} layer(s), B={w.batch}, {lens}, Hq={w.q_heads}/Hkv={w.kv_heads}, "
            f"d={w.head_dim}, page {w.page_size}, {w.scheme} KV codes, {step}")


# ---------------------------------------------------------------- oracle arms
def oracle_sample_run(w: inp.Workload, rank: int, budget_s: float, steps: int = 1, warmup: int = 0):
    """Times the CPU oracle on a bounded sample of sequences of the workload:
    per step, the oracle appends the step's new tokens and computes the fp64
    decode attention of every query head.  The sample grows until one step
    is estimated to take about budget_s seconds.  Returns (GB/s of
    algorithmic bytes over the sample, threads used, description, per-step
    seconds)."""
    import oracle
    oracle.build()
    lens = inp.seq_lens(w)
    n_new = step_plan(w, lens)
    order = np.random.default_rng(1234 + rank).permutation(len(lens)).tolist()
    probe = _oracle_prepare(w, lens, n_new, order[:1], 0)
    t0 = time.perf_counter()
    _oracle_step(w, probe)
    t_first = max(time.perf_counter() - t0, 1e-4)
    per_token = t_first / max(int(lens[order[0]]), 1)
    chosen, est = [], 0.0
    for b in order:
        chosen.append(int(b))
        est += per_token * int(lens[b])
        if est >= budget_s:
            break
    prepared = _oracle_prepare(w, lens, n_new, chosen, 0)
    for _ in range(warmup):
        _oracle_step(w, prepared)
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        _oracle_step(w, prepared)
        times.append(time.perf_counter() - t0)
    sub_lens = lens[chosen]
    nb = algorithmic_bytes(w, sub_lens, n_new[chosen])
    gbs = nb["step"] / w.layers / statistics.median(times) / 1e9
    desc = (f"{len(chosen)} of {len(lens)} sequences ({int(sub_lens.sum())} cached tokens) of layer 0; "
            f"per step: oracle append of the step's new tokens + fp64 decode of all {w.q_heads} query heads")
    return gbs, oracle.max_threads(), desc, times


def _oracle_prepare(w, lens, n_new, seqs, layer):
    import oracle
    P = w.page_size
    sub = lens[seqs]
    bt, npg = inp.page_table(sub, P, w.seed + 99, spare=1)
    c = oracle.OracleCache(w.scheme, npg, P, w.kv_heads, w.head_dim)
    new = []
    for i, b in enumerate(seqs):
        L, n = int(lens[b]), int(n_new[b])
        k, v = inp.kv_rows(w, layer, b, 0, L)
        c.append(inp.slots(bt, i, np.arange(0, L - n), P), k[: L - n], v[: L - n])
        new.append((inp.slots(bt, i, np.arange(L - n, L), P), k[L - n:], v[L - n:]))
    q = inp.queries(w, layer)[seqs]
    return c, bt, sub, new, q


def _oracle_step(w, prepared):
    c, bt, sub, new, q = prepared
    for slots, k, v in new:
        c.append(slots, k, v)
    return c.decode_attn(q, bt, sub, w.q_heads)


# ---------------------------------------------------------------- main
def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=2, choices=sorted(inp.WORKLOADS))
    ap.add_argument("--impl", default="kvq", choices=["kvq", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=2.0,
                    help="wall seconds of oracle work for the cpu_baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true", help="do not sample nvidia-smi during the timed region")
    ap.add_argument("--no-graph", action="store_true",
                    help="time the eager launches only (default: the step is also replayed from a CUDA graph "
                         "and that time is the headline value)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    w = inp.WORKLOADS[args.config]

    if args.impl == "reference":
        return run_reference(args, w, rank, world)

    import torch
    import torch.distributed as dist
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)

    def barrier():
        if world > 1:
            dist.barrier()

    bench = Bench(w, dev, rank)
    nb = algorithmic_bytes(w, bench.lens, bench.n_new)
    clocks = ClockSampler(local_rank)
    if not args.no_clocks:
        clocks.start()
        clocks.wait_first()
    step_ms, k2_ms, k1_ms, wall, status = bench.run(args.steps, args.warmup, barrier)
    eager_ms_per_step = max_over_ranks(sum(step_ms), world, dev) / args.steps
    graph_ms = None
    if not args.no_graph:
        graph_ms, gstatus = bench.run_graph(args.steps, barrier)
        if status == bench.kvq.OK:
            status = gstatus
    clock_info = clocks.stop()
    timed_ms = graph_ms if graph_ms is not None else step_ms
    total_ms = max_over_ranks(sum(timed_ms), world, dev)
    ms_per_step = total_ms / args.steps
    e2e_ms, h2d, d2h = bench.run_e2e(max(3, args.steps // 2), 3)
    e2e_per_step = max_over_ranks(statistics.mean(e2e_ms), world, dev)

    if rank == 0:
        peak, peak_kind = measured_hbm_peak()
        k2_mean_ms = statistics.mean(k2_ms)
        achieved = nb["decode_partial"] / w.layers / (k2_mean_ms * 1e-3) / 1e9
        value = job_throughput(nb["step"], world, ms_per_step)
        decode_gbs = nb["decode"] / (ms_per_step * 1e-3) / 1e9
        line = {
            "metric": METRIC,
            "value": round(value, 2),
            "unit": "GB/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(ms_per_step, 5),
            "ms_per_step_eager": round(eager_ms_per_step, 5),
            "launch": "cuda_graph_replay" if graph_ms is not None else "eager",
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": describe(w), "batch": w.batch, "layers": w.layers,
                       "cached_tokens": int(bench.lens.sum()), "kv_codes": w.scheme,
                       "l2": "flushed before every timed step (256 MB write, outside the timed events)",
                       "parallelism": f"replicas x{world} (independent batches, no collective)"},
            "hbm_frac_of_8tbs": round(value / NOMINAL_HBM_GBS, 4),
            "decode_kv_gbs_step": round(decode_gbs, 2),
            "decode_tokens_per_s": round(world * w.batch / (ms_per_step * 1e-3), 1),
            "append_tokens_per_s_step": round(world * nb["append_tokens"] / (ms_per_step * 1e-3), 1),
            "algorithmic_bytes_per_step": nb["step"],
            "roofline": {"kernel": "decode_partial_kernel (split-K fused-dequant decode, merge fused)",
                         "bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                         if peak_kind == "measured" else "fallback 6.8 TB/s",
                         "traffic": traffic_record(w.cid),
                         "mean_launch_us": round(k2_mean_ms * 1e3, 3),
                         "algorithmic_bytes_per_launch": nb["decode_partial"] // w.layers},
            "append": append_line(nb, w, statistics.mean(k1_ms), peak),
            "e2e": {"value": round(job_throughput(nb["step"], world, e2e_per_step), 2), "unit": "GB/s",
                    "ms_per_step": round(e2e_per_step, 5), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": bench.launches_per_step * args.steps,
            "clocks": clock_info,
            "wall_s_timed_region": round(wall, 4),
            "step_ms_min_median_max": [round(min(timed_ms), 5), round(statistics.median(timed_ms), 5),
                                       round(max(timed_ms), 5)],
            "device_status": bench.kvq.status_string(status),
        }
        if not args.no_cpu_baseline and world >= 1:
            gbs, cores, desc, _ = oracle_sample_run(w, rank, args.cpu_budget)
            line["cpu_baseline"] = {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                                    "sample": desc}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def run_reference(args, w, rank, world):
    """The reference arm: the CPU oracle on the host cores (rank 0 only)."""
    if rank != 0:
        return
    gbs, cores, desc, times = oracle_sample_run(w, 0, args.cpu_budget, steps=args.steps, warmup=args.warmup)
    ms = statistics.mean(times) * 1e3
    line = {"metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": describe(w), "batch": w.batch, "layers": w.layers, "kv_codes": w.scheme},
            "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "kind": "oracle", "cores": cores,
                             "sample": desc},
            "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
