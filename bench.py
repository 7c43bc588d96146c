"""Benchmark: decode steps of the paged quantized-KV path on GB300.

A step is one pass of the whole hot path over one batch: quantize-append of
the step's new tokens (kvq_append) and split-K fused-dequant decode attention
with its merge (kvq_decode_attn: one launch), for every layer of the
workload; with per-channel K scales (workload 6) the append keeps the new
tokens' bf16 K rows and the pages it fills are sealed (kvq_append_kchan,
kvq_seal_pages) before the decode.  Pages come from the library's host allocator (scattered ids).
Inputs are resident in HBM when the timed region starts; L2 is flushed (a
256 MB write, then a 256 MB read that evicts the write's dirty lines, so their
write-back does not run under the timed kernels) before every timed step,
outside the timed events.

Headline workload (N=1 default): the largest single-GPU configuration, the
8-layer INT4 workload -- 16 sequences x 32768 cached tokens, 32 query / 8 KV
heads, head_dim 128, page 32, asymmetric INT4 in groups of 32 -- decode step
plus 1-token append per layer.  At N=1 the same JSON line carries one
sub-record per other workload (--sub, default 2,3,5,6), each with its own
decode roofline, append figures, end-to-end figure, clocks and CPU baseline.

Timing.  The headline `ms_per_step` is the mean over exactly --steps steps
replayed from a CUDA graph after --warmup untimed steps, bracketed by a
barrier and a device synchronize, max over ranks.  Per-launch kernel figures
(the roofline and append blocks) come from a separate loop of eager steps,
each launch bracketed by CUDA events on the launching stream, repeated for
at least --kernel-seconds per workload so that the clock sampler sees the GPU
under load; the clocks reported are those sampled during that loop.

Multi-GPU (torchrun, N > 1): the batch's sequences are partitioned over the
ranks (longest first onto the least-loaded rank); each rank allocates its own
pages and block-table rows for its share and no data moves between ranks.
`value` is all ranks' algorithmic bytes over the slowest rank's time (total
work fixed as N grows: "scaling": "strong").

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config C] [--sub 2,3,5,6] [--impl kvq|reference]

Prints one JSON line (rank 0).  --impl reference times the CPU oracle (the
only reference implementation there is) on the host cores, on a bounded
sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time
from concurrent.futures import ThreadPoolExecutor

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import kvq_inputs as inp  # noqa: E402

METRIC = "paged quantized-KV decode attn GB/s (% of 8 TB/s HBM); append tokens/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 256 << 20
HEADLINE = 4
HOST_FRACTION = 0.0  # fraction of each layer's page ids in the host tier (--host-fraction)
APPEND_MODE = "separate"  # --append-mode


# ---------------------------------------------------------------- accounting
def code_meta_bytes(w: inp.Workload):
    """(code bytes, scale+zero bytes) per (token, KV head) for one of K / V."""
    if w.scheme == "int4":
        return w.head_dim // 2, (w.head_dim // w.group) * 4
    return w.head_dim, 4


def step_plan(w: inp.Workload, lens: np.ndarray):
    """Tokens appended per sequence in one step."""
    n_new = w.prefill_chunk if w.cid == 5 else w.append_tokens
    return np.minimum(lens, n_new).astype(np.int64)


def algorithmic_bytes(w: inp.Workload, lens: np.ndarray, n_new: np.ndarray) -> dict:
    """Bytes the method must move per step (per layer x layers): never padding.
    Decode: codes and scales of every cached token, the block-table entries of
    the pages in use, the query rows, the lengths and the fp32 output rows.
    Append: the bf16 K/V rows and slot of each new token read, its codes and
    scales written."""
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
    seal = 0
    if w.scheme == "int8kc":
        # per-channel K: the channel factors of every page in use are read;
        # the append also reads the residual slot ids and writes each new
        # token's bf16 K rows (and the factors of a page it opens); the seal
        # of each page the step fills reads its residual rows and ids and
        # writes its K codes, factors and token scales
        decode += table // 4 * H * D * 2
        opened = int(sum(((np.arange(L - n, L) % P) == 0).sum() for L, n in zip(lens, n_new)))
        append += T * (4 + H * D * 2) + opened * H * D * 2
        filled = sealed_pages_of_step(lens, n_new, P)
        seal = filled * (8 + H * (P * D * 2 + P * D + D * 2 + P * 4))
    L = w.layers
    return {"decode": decode * L, "append": append * L, "seal": seal * L, "step": (decode + append + seal) * L,
            "append_tokens": T * L, "kv_bytes": kv * L}


def sealed_pages_of_step(lens, n_new, P: int) -> int:
    """Pages that a step's new tokens complete (their last offset written)."""
    return int(sum(((np.arange(L - n, L) % P) == P - 1).sum() for L, n in zip(lens, n_new)))


def partition_sequences(lens, world: int) -> list:
    """Shares of the batch's sequences for `world` ranks: longest first onto
    the rank with the fewest tokens so far (ties: lower rank, then lower
    sequence index).  Every sequence goes to exactly one rank; each share is
    returned in increasing sequence order."""
    lens = np.asarray(lens, np.int64)
    order = sorted(range(len(lens)), key=lambda b: (-int(lens[b]), b))
    load = [0] * world
    shares = [[] for _ in range(world)]
    for b in order:
        r = min(range(world), key=lambda i: (load[i], i))
        shares[r].append(b)
        load[r] += int(lens[b])
    return [np.array(sorted(s), np.int64) for s in shares]


def append_line(nb: dict, w: inp.Workload, k1_mean_ms: float, peak_gbs: float, fused: bool = False,
                kchan: bool = False) -> dict:
    """The quantize-append launch on its own: tokens per second, and its
    algorithmic bytes (bf16 K/V read, slots read, codes and scales written)
    per second against the HBM peak.  Fused into the decode launch, its time
    is taken as that whole launch's (k1_mean_ms is then the decode's)."""
    T = nb["append_tokens"] // w.layers      # tokens per launch
    # algorithmic bytes per launch (per-channel K: the seal of the pages the
    # step fills runs inside the same timed interval, so its bytes count too)
    b = (nb["append"] + (nb["seal"] if kchan else 0)) // w.layers
    t = k1_mean_ms * 1e-3
    return {"kernel": "fused into the decode launch (its whole time counted)" if fused
            else "append_kernel + seal_kernel of the pages it fills" if kchan
            else "append_kernel (quantize-append)", "tokens_per_launch": T,
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


def kernel_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "dynamically_quantized_paged_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.startswith("kvq_decode") or name in ("kvq_device.cuh", "kvq_internal.h", "kvq_tc.cuh", "kvq_alu.cuh",
                                                     "kvq_quant.cuh"):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + f.read())
    return h.hexdigest()


def traffic_record(cid: int):
    """DRAM bytes per decode launch from a committed ncu capture, if it was
    taken on the current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "decode_traffic.json")
    try:
        with open(p) as f:
            rec = json.load(f)
    except Exception:
        return None
    if rec.get("kernel_source_sha256") != kernel_source_hash():
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


def sum_over_ranks(x: int, world: int, device=None) -> int:
    """The sum of x over all ranks (the job's total work)."""
    if world <= 1:
        return int(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([int(x)], dtype=torch.int64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return int(t.item())


def job_throughput(total_bytes: int, ms_per_step: float) -> float:
    """Whole-job GB/s: all ranks' bytes of one step over the slowest rank's
    step time."""
    return total_bytes / (ms_per_step * 1e-3) / 1e9


# ---------------------------------------------------------------- staging
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


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, enabled: bool = True):
        self.gpu = gpu_index
        self.enabled = enabled
        self.proc = None
        self.lines = []

    def start(self):
        if not self.enabled:
            return self
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            t0 = time.time()
            while not self.lines and time.time() - t0 < 10.0:  # its start-up is done
                time.sleep(0.05)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

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
        for line in self.lines[1:]:  # the first line is taken before the load starts
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
    """One workload's batch share, set up on one GPU: every layer's cache
    filled by chunked appends (untimed), the step's new tokens and queries
    resident, a workspace and an L2 flush buffer."""

    def __init__(self, w: inp.Workload, device, seqs, alloc_seed: int):
        import torch
        import dynamically_quantized_paged_gb300 as kvq
        self.torch, self.kvq = torch, kvq
        self.w, self.dev = w, device
        self.seqs = np.asarray(seqs, np.int64)
        self.lens = inp.seq_lens(w)[self.seqs]
        self.n_new = step_plan(w, self.lens)
        # the decode that appends its step's token (one launch per layer)
        # serves steps of one new token per sequence on the CUDA-core kernel
        # (GQA <= 4 of INT8, FP8, asymmetric INT4)
        eligible = bool(np.all(self.n_new == 1)) and w.scheme in ("int8", "fp8", "int4") and \
            w.q_heads // w.kv_heads <= 4
        self.kchan = w.scheme == "int8kc"
        self.fused = eligible and APPEND_MODE == "fused"
        B, P = len(self.seqs), w.page_size
        need = inp.pages_needed(self.lens, P)
        self.max_pages = int(need.max())
        num_pages = int(need.sum()) + 16
        # page allocation through the library's host allocator (scattered ids)
        self.alloc = kvq.PageAllocator(num_pages, seed=alloc_seed)
        bt = np.full((B, self.max_pages), -1, np.int32)
        for i in range(B):
            bt[i, :need[i]] = self.alloc.alloc(int(need[i]))
        self.bt_host = bt
        dev = device
        self.bt = torch.from_numpy(bt).to(dev)
        self.seq_lens = torch.from_numpy(self.lens).to(dev)
        self.caches, self.q, self.k_new, self.v_new = [], [], [], []
        new_slots = np.concatenate([inp.slots(bt, i, np.arange(self.lens[i] - self.n_new[i], self.lens[i]), P)
                                    for i in range(B)])
        self.slots_new = torch.from_numpy(new_slots).to(dev)
        if self.kchan:  # the new tokens' residual slots, and the pages the step fills
            self.rslots_new = torch.from_numpy((new_slots // P).astype(np.int32)).to(dev)
            full = np.array([bt[i, t // P] for i, L in enumerate(self.lens)
                             for t in range(int(L - self.n_new[i]), int(L)) if t % P == P - 1], np.int32)
            self.seal_new = torch.from_numpy(full).to(dev) if full.size else None
            self.seal_all = []  # per layer: every page sealed by the prefill
        workers = min(16, os.cpu_count() or 1)
        with ThreadPoolExecutor(max_workers=workers) as ex:
            for layer in range(w.layers):
                # the last host pages of the id space live in the cache's host
                # tier (page-locked host memory read over NVLink-C2C)
                host = min(int(round(HOST_FRACTION * num_pages)), num_pages - 1)
                # per-channel K: one residual slot per page id (slot = page id)
                c = kvq.PagedKVCache(w.scheme, num_pages - host, P, w.kv_heads, w.head_dim, device=dev,
                                     zero_init=False, host_pages=host,
                                     resid_slots=num_pages if self.kchan else 0)
                ks, vs = [], []
                # the rows are generated on host threads, a bounded window ahead
                pending = {}
                nxt = 0

                def submit(i):
                    return ex.submit(inp.kv_rows, w, layer, int(self.seqs[i]), 0, int(self.lens[i]))

                for i in range(B):
                    while nxt < B and nxt < i + 2 * workers:
                        pending[nxt] = submit(nxt)
                        nxt += 1
                    k, v = pending.pop(i).result()
                    kd = torch.from_numpy(k.view(np.int16)).to(dev)
                    vd = torch.from_numpy(v.view(np.int16)).to(dev)
                    L, n = int(self.lens[i]), int(self.n_new[i])
                    for s0 in range(0, L - n, w.prefill_chunk):     # prefill (untimed)
                        s1 = min(L - n, s0 + w.prefill_chunk)
                        sl = inp.slots(bt, i, np.arange(s0, s1), P)
                        if self.kchan:
                            kvq.append_kchan(c, torch.from_numpy(sl).to(dev),
                                             torch.from_numpy((sl // P).astype(np.int32)).to(dev),
                                             kd[s0:s1], vd[s0:s1])
                        else:
                            kvq.append(c, torch.from_numpy(sl).to(dev), kd[s0:s1], vd[s0:s1])
                    ks.append(kd[L - n:L].clone())
                    vs.append(vd[L - n:L].clone())
                self.k_new.append(torch.cat(ks))
                self.v_new.append(torch.cat(vs))
                if self.kchan:  # seal every page the prefill filled
                    pre = self.lens - self.n_new
                    pg = np.concatenate([bt[i, :int(pre[i]) // P] for i in range(B)]).astype(np.int32)
                    pgd = torch.from_numpy(pg).to(dev)
                    kvq.seal_pages(c, pgd, pgd)
                    self.seal_all.append(pgd)
                self.caches.append(c)
                self.q.append(torch.from_numpy(np.ascontiguousarray(inp.queries(w, layer)[self.seqs]).view(np.int16)).to(dev))
        self.out = torch.empty((B, w.q_heads, w.head_dim), dtype=torch.float32, device=dev)
        self.ws = kvq.alloc_workspace(self.caches[0], B, w.q_heads, self.max_pages, device=dev)
        self.flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.flush_read = torch.ones(L2_FLUSH_BYTES // 8, dtype=torch.int64, device=dev)
        torch.cuda.synchronize(dev)
        st = kvq.last_device_error()
        if st != kvq.OK:
            raise RuntimeError(f"set-up failed: {kvq.status_string(st)}")
        self.launches_per_step = 2 * w.layers  # quantize-append + fused decode per layer
        if self.kchan and self.seal_new is not None:
            self.launches_per_step += w.layers  # the seal of the pages the step fills

    def flush_l2(self):
        """Evict the step's data from L2: write a buffer larger than L2, then
        read another one, so that the dirty lines of the write are written
        back during the flush rather than while the timed kernels run."""
        self.flush.zero_()
        self.flush_sink = self.flush_read.sum()

    def step(self, events=None, q=None, k_new=None, v_new=None, slots=None, bt=None, lens=None, out=None,
             stream=None, rslots=None, seal=None):
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
            if self.kchan:  # append (keeping the bf16 K rows), then seal the pages it filled
                kvq.append_kchan(c, slots, self.rslots_new if rslots is None else rslots, k_new[layer],
                                 v_new[layer], stream=stream)
                sp = self.seal_new if seal is None else seal
                if sp is not None:
                    kvq.seal_pages(c, sp, sp, stream=stream)
            elif not self.fused:
                kvq.append(c, slots, k_new[layer], v_new[layer], stream=stream)
            if events is not None:
                events[layer][0].record()
            if self.fused:  # one launch: the decode quantizes and stores each sequence's new token itself
                kvq.decode_attn_append(c, k_new[layer], v_new[layer], q[layer], bt, lens, out, self.ws,
                                       stream=stream)
            else:
                kvq.decode_attn(c, q[layer], bt, lens, out, self.ws, stream=stream)  # one launch, splits merged in place
            if events is not None:
                events[layer][1].record()

    def run_eager(self, steps: int, warmup: int, barrier):
        """--steps eager steps after --warmup: per-step events."""
        torch = self.torch
        for _ in range(warmup):
            self.flush_l2()
            self.step()
        torch.cuda.synchronize(self.dev)
        st = self.kvq.last_device_error()
        if st != self.kvq.OK:
            raise RuntimeError(f"warm-up failed: {self.kvq.status_string(st)}")
        E = torch.cuda.Event
        ev = [(E(enable_timing=True), E(enable_timing=True)) for _ in range(steps)]
        barrier()
        torch.cuda.synchronize(self.dev)
        for i in range(steps):
            self.flush_l2()
            ev[i][0].record()
            self.step()
            ev[i][1].record()
        torch.cuda.synchronize(self.dev)
        barrier()
        return [a.elapsed_time(b) for a, b in ev], self.kvq.last_device_error()

    def run_graph(self, steps: int, warmup: int, barrier):
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
        for _ in range(warmup):
            self.flush_l2()
            graph.replay()
        torch.cuda.synchronize(self.dev)
        E = torch.cuda.Event
        evs = [(E(enable_timing=True), E(enable_timing=True)) for _ in range(steps)]
        barrier()
        torch.cuda.synchronize(self.dev)
        t0 = time.perf_counter()
        for i in range(steps):
            self.flush_l2()
            evs[i][0].record()
            graph.replay()
            evs[i][1].record()
        torch.cuda.synchronize(self.dev)
        barrier()
        wall = time.perf_counter() - t0
        self.graph = graph
        return [a.elapsed_time(b) for a, b in evs], wall, self.kvq.last_device_error()

    def kernel_loop(self, seconds: float):
        """Eager steps with every append and decode launch bracketed by CUDA
        events on the launching stream, repeated until `seconds` of wall time
        have passed.  Returns (decode ms per launch, append ms per launch,
        steps run, wall seconds)."""
        torch = self.torch
        E = torch.cuda.Event
        batch = 64
        evs = [[tuple(E(enable_timing=True) for _ in range(3)) for _ in self.caches] for _ in range(batch)]
        k2, k1, n = [], [], 0
        t0 = time.perf_counter()
        while True:
            # the stream first idles (a device-side sleep of ~15 ms) while the
            # host enqueues the batch, so that no launch waits on the host
            # inside a bracketed interval (a step of short launches would
            # otherwise time the host's launch latency, not the kernel)
            torch.cuda._sleep(30_000_000)
            for i in range(batch):
                self.flush_l2()
                self.step(events=evs[i])
            torch.cuda.synchronize(self.dev)
            for row in evs:
                for ev in row:
                    k2.append(ev[0].elapsed_time(ev[1]))
                    k1.append(ev[2].elapsed_time(ev[0]))
            n += batch
            if time.perf_counter() - t0 >= seconds:
                break
        return k2, k1, n, time.perf_counter() - t0

    def run_e2e(self, steps: int, warmup: int):
        """The same step through the public API with HOST buffers: a pinned host
        -> device copy of the step's inputs and a device -> host copy of the
        output inside the timed region.  The inputs (queries, new keys and
        values, slots, block tables, lengths) are staged in one pinned buffer
        at 256-byte aligned offsets and go over in ONE copy; the device
        tensors the calls take are views of its device twin."""
        torch = self.torch
        srcs = list(self.q) + list(self.k_new) + list(self.v_new) + [self.slots_new, self.bt, self.seq_lens]
        if self.kchan:
            srcs += [self.rslots_new] + ([self.seal_new] if self.seal_new is not None else [])
        offs, total = stage_layout(srcs)
        h_buf = torch.empty(total, dtype=torch.uint8).pin_memory()
        d_buf = torch.empty(total, dtype=torch.uint8, device=self.dev)
        for t, off in zip(srcs, offs):
            stage_view(h_buf, t, off).copy_(t.cpu())
        d_views = [stage_view(d_buf, t, off) for t, off in zip(srcs, offs)]
        nl = len(self.q)
        d_q, d_k, d_v = d_views[:nl], d_views[nl:2 * nl], d_views[2 * nl:3 * nl]
        d_slots, d_bt, d_lens = d_views[3 * nl:3 * nl + 3]
        d_rs = d_views[3 * nl + 3] if self.kchan else None
        d_seal = d_views[3 * nl + 4] if self.kchan and self.seal_new is not None else None
        h_out = torch.empty(self.out.shape, dtype=torch.float32).pin_memory()
        h2d = total
        d2h = h_out.numel() * 4

        def one():
            d_buf.copy_(h_buf, non_blocking=True)
            self.step(q=d_q, k_new=d_k, v_new=d_v, slots=d_slots, bt=d_bt, lens=d_lens, rslots=d_rs, seal=d_seal)
            h_out.copy_(self.out, non_blocking=True)

        for _ in range(warmup):
            self.flush_l2()
            one()
        torch.cuda.synchronize(self.dev)
        E = torch.cuda.Event
        evs = [(E(enable_timing=True), E(enable_timing=True)) for _ in range(steps)]
        for i in range(steps):
            self.flush_l2()
            evs[i][0].record()
            one()
            evs[i][1].record()
        torch.cuda.synchronize(self.dev)
        return [a.elapsed_time(b) for a, b in evs], h2d, d2h

    def seal_loop(self, seconds: float):
        """Per-channel K: the seal of every page the prefill filled (layer 0),
        one launch, each bracketed by CUDA events after an L2 flush, repeated
        for `seconds`.  Returns (ms per launch, pages per launch)."""
        torch = self.torch
        E = torch.cuda.Event
        pages = self.seal_all[0]
        c = self.caches[0]
        ms = []
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < seconds:
            evs = [(E(enable_timing=True), E(enable_timing=True)) for _ in range(32)]
            for a, b in evs:
                self.flush_l2()
                a.record()
                self.kvq.seal_pages(c, pages, pages)
                b.record()
            torch.cuda.synchronize(self.dev)
            ms += [a.elapsed_time(b) for a, b in evs]
        return ms, int(pages.numel())

    def close(self):
        self.graph = None
        self.caches, self.q, self.k_new, self.v_new = [], [], [], []
        self.ws = self.flush = self.flush_read = self.out = None
        self.alloc.close()
        self.torch.cuda.empty_cache()


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


def roofline_block(w, nb, k2_ms, peak, peak_kind, fused=False):
    """The decode launch against the HBM roofline; with the append fused into
    it, the launch's algorithmic bytes include the append's."""
    mean = statistics.mean(k2_ms)
    b = (nb["step"] if fused else nb["decode"]) // w.layers
    achieved = b / (mean * 1e-3) / 1e9
    return {"kernel": "decode kernel (split-K fused-dequant decode, merge fused"
                      + (", appends each sequence's new token)" if fused else ")"),
            "bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
            else "fallback 6.8 TB/s",
            "traffic": traffic_record(w.cid), "mean_launch_us": round(mean * 1e3, 3),
            "median_launch_us": round(statistics.median(k2_ms) * 1e3, 3), "launches_timed": len(k2_ms),
            "algorithmic_bytes_per_launch": b, "frac_of_8tbs": round(achieved / NOMINAL_HBM_GBS, 4)}


def measure_workload(w, dev, local_rank, args, world, rank, barrier, headline: bool):
    """Everything the line reports for one workload (this rank's share)."""
    seqs = partition_sequences(inp.seq_lens(w), world)[rank] if world > 1 else np.arange(w.batch)
    bench = Bench(w, dev, seqs, alloc_seed=w.seed * 7919 + rank)
    nb = algorithmic_bytes(w, bench.lens, bench.n_new)
    total_step = sum_over_ranks(nb["step"], world, dev)
    total_decode = sum_over_ranks(nb["decode"], world, dev)
    total_seqs = sum_over_ranks(len(seqs), world, dev)
    total_append = sum_over_ranks(nb["append_tokens"], world, dev)
    steps = args.steps if headline else max(10, args.steps // 2)
    clocks = ClockSampler(local_rank, enabled=not args.no_clocks).start()
    eager_ms, status = bench.run_eager(steps, args.warmup, barrier)
    graph_ms, wall, gstatus = (None, None, status) if args.no_graph else bench.run_graph(steps, args.warmup, barrier)
    k2_ms, k1_ms, loop_steps, loop_wall = bench.kernel_loop(args.kernel_seconds)
    clock_info = clocks.stop()
    if status == bench.kvq.OK:
        status = gstatus
    timed = graph_ms if graph_ms is not None else eager_ms
    ms_per_step = max_over_ranks(sum(timed), world, dev) / steps
    eager_per_step = max_over_ranks(sum(eager_ms), world, dev) / steps
    e2e_ms, h2d, d2h = bench.run_e2e(max(3, steps // 2), 3)
    seal_rec = None
    if bench.kchan:
        s_ms, s_pages = bench.seal_loop(min(args.kernel_seconds, 0.5))
        peak0, _ = measured_hbm_peak()
        H, D, P = w.kv_heads, w.head_dim, w.page_size
        sb = s_pages * (8 + H * (P * D * 2 + P * D + D * 2 + P * 4))
        sm = statistics.mean(s_ms)
        seal_rec = {"kernel": "seal_kernel (per-channel K re-quantization of full pages)",
                    "pages_per_launch": s_pages, "kv_heads": H, "mean_launch_us": round(sm * 1e3, 3),
                    "algorithmic_bytes_per_launch": sb, "achieved_gbs": round(sb / (sm * 1e-3) / 1e9, 2),
                    "peak": peak0, "frac": round(sb / (sm * 1e-3) / 1e9 / peak0, 4),
                    "what": "every page the prefill filled, re-sealed from its residual slot in one launch"}
    e2e_per_step = max_over_ranks(statistics.mean(e2e_ms), world, dev)
    st2 = bench.kvq.last_device_error()
    if status == bench.kvq.OK:
        status = st2
    peak, peak_kind = measured_hbm_peak()
    rec = {
        "value": round(job_throughput(total_step, ms_per_step), 2),
        "ms_per_step": round(ms_per_step, 5),
        "ms_per_step_eager": round(eager_per_step, 5),
        "launch": "cuda_graph_replay" if graph_ms is not None else "eager",
        "steps": steps,
        "config": {"workload": describe(w), "batch": w.batch, "layers": w.layers,
                   "cached_tokens": int(inp.seq_lens(w).sum()), "kv_codes": w.scheme,
                   "l2": "flushed before every timed step (256 MB write, then a 256 MB read, outside the timed events)",
                   "parallelism": (f"sequences partitioned over {world} GPUs, no collective" if world > 1
                                   else "1 GPU"),
                   **({"host_tier_fraction": HOST_FRACTION} if HOST_FRACTION > 0 else {}),
                   "append": ("fused into each layer's decode launch" if bench.fused
                              else "append kernel, then the decode (programmatic launch overlap)")},
        "hbm_frac_of_8tbs": round(job_throughput(total_step, ms_per_step) / NOMINAL_HBM_GBS / max(world, 1), 4),
        "decode_kv_gbs_step": round(job_throughput(total_decode, ms_per_step), 2),
        "decode_tokens_per_s": round(total_seqs / (ms_per_step * 1e-3), 1),
        "append_tokens_per_s_step": round(total_append / (ms_per_step * 1e-3), 1),
        "algorithmic_bytes_per_step": total_step,
        "roofline": roofline_block(w, nb, k2_ms, peak, peak_kind, fused=bench.fused),
        "append": append_line(nb, w, statistics.mean(k2_ms if bench.fused else k1_ms), peak, fused=bench.fused,
                              kchan=bench.kchan),
        **({"seal": seal_rec} if seal_rec is not None else {}),
        "kernel_loop": {"steps": loop_steps, "wall_s": round(loop_wall, 3),
                        "what": "eager steps, each launch bracketed by CUDA events; the clocks below are "
                                "sampled across the timed steps and this loop"},
        "e2e": {"value": round(job_throughput(total_step, e2e_per_step), 2), "unit": "GB/s",
                "ms_per_step": round(e2e_per_step, 5), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": bench.launches_per_step * steps,
        "clocks": clock_info,
        "wall_s_timed_region": round(wall, 4) if wall is not None else None,
        "step_ms_min_median_max": [round(min(timed), 5), round(statistics.median(timed), 5), round(max(timed), 5)],
        "device_status": bench.kvq.status_string(status),
    }
    bench.close()
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        gbs, cores, desc, _ = oracle_sample_run(w, rank, args.cpu_budget)
        rec["cpu_baseline"] = {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                               "sample": desc}
    return rec


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
    kc = w.scheme == "int8kc"  # per-channel K: residual slot = page id; full pages sealed
    c = oracle.OracleCache(w.scheme, npg, P, w.kv_heads, w.head_dim, resid_slots=npg if kc else 0)
    new = []
    for i, b in enumerate(seqs):
        L, n = int(lens[b]), int(n_new[b])
        k, v = inp.kv_rows(w, layer, b, 0, L)
        sl = inp.slots(bt, i, np.arange(0, L - n), P)
        c.append(sl, k[: L - n], v[: L - n], resid_slot=(sl // P).astype(np.int32) if kc else None)
        if kc:
            full = bt[i, :(L - n) // P].astype(np.int32)
            c.seal(full, full)
        sl = inp.slots(bt, i, np.arange(L - n, L), P)
        fill = np.array([bt[i, t // P] for t in range(L - n, L) if t % P == P - 1], np.int32)
        new.append((sl, k[L - n:], v[L - n:], fill))
    q = inp.queries(w, layer)[seqs]
    return c, bt, sub, new, q


def _oracle_step(w, prepared):
    c, bt, sub, new, q = prepared
    kc = w.scheme == "int8kc"
    for slots, k, v, fill in new:
        c.append(slots, k, v, resid_slot=(slots // w.page_size).astype(np.int32) if kc else None)
        if kc and fill.size:
            c.seal(fill, fill)
    return c.decode_attn(q, bt, sub, w.q_heads)


# ---------------------------------------------------------------- main
def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=HEADLINE, choices=sorted(inp.WORKLOADS))
    ap.add_argument("--sub", default="2,3,5,6",
                    help="other workloads measured as sub-records of the line at N=1 ('' for none)")
    ap.add_argument("--impl", default="kvq", choices=["kvq", "reference"])
    ap.add_argument("--kernel-seconds", type=float, default=1.0,
                    help="wall seconds of the per-launch timing loop of each workload")
    ap.add_argument("--cpu-budget", type=float, default=2.0,
                    help="wall seconds of oracle work for each cpu_baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true", help="do not sample nvidia-smi during the timed region")
    ap.add_argument("--layers", type=int, default=0,
                    help="profiling runs only: override the workload's layer count (the per-launch work is "
                         "per layer; the JSON line names the layers it ran)")
    ap.add_argument("--host-fraction", type=float, default=0.0,
                    help="place this fraction of each layer's page ids in the cache's host tier (read in place "
                         "over NVLink-C2C); 0 (default): every page in device memory")
    ap.add_argument("--append-mode", default="separate", choices=["separate", "fused"],
                    help="separate (default): the append kernel, then the decode; fused: each layer's step is "
                         "one decode launch that appends its token itself (steps of one new token per sequence "
                         "on the CUDA-core kernel; elsewhere separate)")
    ap.add_argument("--no-graph", action="store_true",
                    help="time the eager launches only (default: the step is also replayed from a CUDA graph "
                         "and that time is the headline value)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if not 0.0 <= args.host_fraction <= 1.0:
        ap.error("--host-fraction must lie in [0, 1]")
    global HOST_FRACTION, APPEND_MODE
    HOST_FRACTION = args.host_fraction
    APPEND_MODE = args.append_mode

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    w = inp.WORKLOADS[args.config]
    if args.layers > 0:
        import dataclasses
        w = dataclasses.replace(w, layers=args.layers)

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

    head = measure_workload(w, dev, local_rank, args, world, rank, barrier, headline=True)
    subs = {}
    if world == 1:
        for s in [int(x) for x in args.sub.split(",") if x.strip()]:
            if s != args.config:
                subs[str(s)] = measure_workload(inp.WORKLOADS[s], dev, local_rank, args, world, rank, barrier,
                                                headline=False)
    if rank == 0:
        line = {
            "metric": METRIC,
            "value": head.pop("value"),
            "unit": "GB/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": head.pop("ms_per_step"),
            "higher_is_better": True,
            "scaling": "strong",
            "vs_baseline": None,
            "dtype": "f32",
            "data": "synthetic",
        }
        head.pop("steps")
        line.update(head)
        if subs:
            line["workloads"] = subs
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
            "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
            "scaling": "strong",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": describe(w), "batch": w.batch, "layers": w.layers, "kv_codes": w.scheme},
            "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "kind": "oracle", "cores": cores,
                             "sample": desc},
            "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
