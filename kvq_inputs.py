"""Seeded synthetic inputs for the six workloads.

This module holds NO quantization or attention arithmetic: it only draws
random bf16 key/value/query tensors, sequence lengths and page tables.  Both
the CUDA path (tests, bench) and the CPU oracle consume what it produces, so
that the two sides see identical inputs.

Workloads (shapes and distributions as the pages' problem statement and the
workload list fix them; where a distribution parameter is not given, the
plainest choice is taken and stated here):

  1  tiny-int8        1 layer, B=1, 256 tokens, Hq 8 / Hkv 4, d 64, page 16,
                      N(0,1) with 2 outlier (head, channel) pairs x10, INT8,
                      seed 0.
  2  llama3-8b-int8   1 layer, B=32, Hq 32 / Hkv 8, d 128, page 16, lengths
                      uniform in [512, 4096], pages shuffled, N(0,1) with 1 %
                      of the Hkv*d (head, channel) pairs (10) x8, INT8,
                      decode step + 1-token append.
  3  llama3-70b-fp8   1 layer, B=64, Hq 64 / Hkv 8, d 128, page 16, lengths
                      lognormal with median 4096 and sigma 1 (log space),
                      clipped to [1024, 32768]; N(0,1) with 10 heavy-tailed
                      (head, channel) pairs drawn from Student-t nu=4;
                      FP8-E4M3 with an fp32 scale.
  4  int4-g32-8layer  8 layers, B=16, 32768 tokens each, Hq 32 / Hkv 8, d 128,
                      page 32, N(0,1), INT4 asymmetric, group 32, fp16 scale
                      and zero-point; decode looped over the layers.
  5  long-128k-int8   1 layer, B=1, 131072 tokens, Hq 64 / Hkv 8, d 128,
                      page 16, N(0,1), INT8; split-K decode plus 4096-token
                      chunked appends.
  6  llama3-8b-int8kc workload 2's shapes, lengths and rows (same seed) with
                      per-channel K scales: every full page sealed, the open
                      page of each sequence in per-token form; decode step +
                      1-token append + the seal of the pages it fills.

The queries are N(0,1) everywhere.  Every array is a pure function of
(workload seed, layer, sequence), so a sampled check can regenerate exactly
the rows it needs.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    cid: int
    name: str
    scheme: str              # "int8" | "fp8" | "int4" | "int4sym"
    layers: int
    batch: int
    q_heads: int
    kv_heads: int
    head_dim: int
    page_size: int
    lengths: tuple           # ("fixed", L) | ("uniform", lo, hi) | ("lognormal", median, sigma, lo, hi)
    seed: int
    outlier_pairs: int = 0   # number of (kv head, channel) pairs that are outliers
    outlier_gain: float = 1.0
    heavy_pairs: int = 0     # number of (kv head, channel) pairs drawn from Student-t
    heavy_nu: float = 4.0
    append_tokens: int = 1   # tokens appended per sequence in one decode step
    prefill_chunk: int = 4096
    group: int = 32

    @property
    def gqa(self) -> int:
        return self.q_heads // self.kv_heads


WORKLOADS = {
    1: Workload(1, "tiny-int8", "int8", 1, 1, 8, 4, 64, 16, ("fixed", 256), seed=0,
                outlier_pairs=2, outlier_gain=10.0),
    2: Workload(2, "llama3-8b-layer-int8", "int8", 1, 32, 32, 8, 128, 16, ("uniform", 512, 4096),
                seed=2, outlier_pairs=10, outlier_gain=8.0),
    3: Workload(3, "llama3-70b-layer-fp8", "fp8", 1, 64, 64, 8, 128, 16,
                ("lognormal", 4096, 1.0, 1024, 32768), seed=3, heavy_pairs=10, heavy_nu=4.0),
    4: Workload(4, "int4-g32-8layer", "int4", 8, 16, 32, 8, 128, 32, ("fixed", 32768), seed=4),
    5: Workload(5, "long-128k-int8", "int8", 1, 1, 64, 8, 128, 16, ("fixed", 131072), seed=5),
    6: Workload(6, "llama3-8b-layer-int8kc", "int8kc", 1, 32, 32, 8, 128, 16, ("uniform", 512, 4096),
                seed=2, outlier_pairs=10, outlier_gain=8.0),
}


def _rng(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(k) & 0xFFFFFFFF for k in key])))


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round-to-nearest-even (torch)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_float(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def seq_lens(w: Workload) -> np.ndarray:
    kind = w.lengths[0]
    if kind == "fixed":
        return np.full(w.batch, w.lengths[1], np.int32)
    r = _rng(w.seed, 0xA11)
    if kind == "uniform":
        lo, hi = w.lengths[1], w.lengths[2]
        return r.integers(lo, hi + 1, size=w.batch).astype(np.int32)
    if kind == "lognormal":
        med, sigma, lo, hi = w.lengths[1:]
        x = np.exp(r.normal(math.log(med), sigma, size=w.batch))
        return np.clip(np.rint(x), lo, hi).astype(np.int32)
    raise ValueError(kind)


def special_channels(w: Workload, layer: int):
    """(kv_head, channel) pairs that carry outliers / heavy tails in a layer."""
    r = _rng(w.seed, 0xC4A, layer)
    n = max(w.outlier_pairs, w.heavy_pairs)
    if n == 0:
        return np.zeros((0, 2), np.int64)
    flat = r.choice(w.kv_heads * w.head_dim, size=n, replace=False)
    return np.stack([flat // w.head_dim, flat % w.head_dim], axis=1)


def kv_rows(w: Workload, layer: int, b: int, start: int, stop: int):
    """bf16 bits of K and V for tokens [start, stop) of sequence b:
    two uint16 arrays [stop-start, Hkv, D].  Tokens are generated in blocks of
    4096 keyed by (seed, layer, b, block), so any sub-range is reproducible."""
    blk = 4096
    ks, vs = [], []
    for b0 in range(start // blk * blk, stop, blk):
        r = _rng(w.seed, 0x4B56, layer, b, b0 // blk)
        n = blk
        shape = (n, w.kv_heads, w.head_dim)
        k = r.standard_normal(shape, dtype=np.float32)
        v = r.standard_normal(shape, dtype=np.float32)
        ch = special_channels(w, layer)
        if w.heavy_pairs:
            for (h, c) in ch[: w.heavy_pairs]:
                k[:, h, c] = r.standard_t(w.heavy_nu, size=n).astype(np.float32)
                v[:, h, c] = r.standard_t(w.heavy_nu, size=n).astype(np.float32)
        if w.outlier_pairs:
            for (h, c) in ch[: w.outlier_pairs]:
                k[:, h, c] *= w.outlier_gain
                v[:, h, c] *= w.outlier_gain
        lo = max(start, b0) - b0
        hi = min(stop, b0 + blk) - b0
        ks.append(k[lo:hi])
        vs.append(v[lo:hi])
    k = np.concatenate(ks, axis=0) if ks else np.zeros((0, w.kv_heads, w.head_dim), np.float32)
    v = np.concatenate(vs, axis=0) if vs else np.zeros((0, w.kv_heads, w.head_dim), np.float32)
    return to_bf16_bits(k), to_bf16_bits(v)


def queries(w: Workload, layer: int, step: int = 0) -> np.ndarray:
    r = _rng(w.seed, 0x9, layer, step)
    return to_bf16_bits(r.standard_normal((w.batch, w.q_heads, w.head_dim), dtype=np.float32))


def pages_needed(lens: np.ndarray, page_size: int) -> np.ndarray:
    return (np.asarray(lens, np.int64) + page_size - 1) // page_size


def page_table(lens: np.ndarray, page_size: int, seed: int, spare: int = 0,
               max_pages_per_seq: int | None = None):
    """Scattered physical pages for each sequence: a seeded random permutation
    of the pool's page ids handed out in sequence order.  Returns
    (block_table int32 [B, max_pages_per_seq] with -1 in unused entries,
    num_pages)."""
    need = pages_needed(lens, page_size)
    total = int(need.sum())
    num_pages = total + spare
    maxp = int(need.max()) if max_pages_per_seq is None else max_pages_per_seq
    maxp = max(maxp, 1)
    perm = _rng(seed, 0xB10C).permutation(num_pages).astype(np.int32)
    bt = np.full((len(lens), maxp), -1, np.int32)
    pos = 0
    for b, n in enumerate(need):
        bt[b, :n] = perm[pos:pos + n]
        pos += n
    return bt, max(num_pages, 1)


def slots(block_table: np.ndarray, b: int, positions: np.ndarray, page_size: int) -> np.ndarray:
    """Physical slot of each logical position of sequence b (page id * page
    size + offset inside the page)."""
    positions = np.asarray(positions, np.int64)
    return block_table[b, positions // page_size].astype(np.int64) * page_size + positions % page_size
