"""Shared set-up for the GPU parity tests: fills a device cache through the C
ABI and an oracle cache image from the same seeded bf16 inputs, and compares
them."""
from __future__ import annotations

import numpy as np
import torch

import dynamically_quantized_paged_gb300 as kvq
import kvq_inputs as inp
import oracle

ATOL = 1e-2      # attention tolerance: max |gpu - oracle|
MEAN_REL = 2e-3  # attention tolerance: sum |gpu - oracle| / sum |oracle|

DEV = torch.device("cuda:0")


def dev_bits(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(DEV)


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


class Case:
    """One layer: device cache + (optionally partial) oracle cache image."""

    def __init__(self, w: inp.Workload, lens: np.ndarray, layer: int = 0, spare: int = 3,
                 oracle_seqs=None, chunk: int = 4096, table_seed: int | None = None,
                 block_table: np.ndarray | None = None, num_pages: int | None = None,
                 kv_override=None, host_pages: int = 0, extra_host_pages: int = 0):
        """host_pages: the last host_pages of the table's page ids live in the
        cache's host tier; extra_host_pages: more host-tier pages beyond the
        table's ids (targets for moving pages between the tiers)."""
        self.w, self.layer = w, layer
        self.lens = np.asarray(lens, np.int32)
        if block_table is None:
            block_table, num_pages = inp.page_table(self.lens, w.page_size,
                                                    w.seed if table_seed is None else table_seed, spare)
        self.bt, self.num_pages = block_table, num_pages
        self.oracle_seqs = list(range(len(self.lens))) if oracle_seqs is None else list(oracle_seqs)
        self.g = kvq.PagedKVCache(w.scheme, num_pages - host_pages, w.page_size, w.kv_heads, w.head_dim,
                                  device=DEV, host_pages=host_pages + extra_host_pages)
        self.o = oracle.OracleCache(w.scheme, num_pages, w.page_size, w.kv_heads, w.head_dim)
        for b, L in enumerate(self.lens):
            for s0 in range(0, int(L), chunk):
                s1 = min(int(L), s0 + chunk)
                if kv_override is not None:
                    k, v = kv_override(b, s0, s1)
                else:
                    k, v = inp.kv_rows(w, layer, b, s0, s1)
                slots = inp.slots(self.bt, b, np.arange(s0, s1), w.page_size)
                kvq.append(self.g, dev(slots), dev_bits(k), dev_bits(v))
                if b in self.oracle_seqs:
                    assert self.o.append(slots, k, v) == 0
        import dataclasses
        self.q = inp.queries(dataclasses.replace(w, batch=len(self.lens)), layer)
        torch.cuda.synchronize()

    def decode(self, q: np.ndarray | None = None, softmax_scale: float = 0.0, split_calls=False):
        w = self.w
        q = self.q if q is None else q
        out = torch.full((len(self.lens), w.q_heads, w.head_dim), float("nan"), dtype=torch.float32,
                         device=DEV)
        ws = kvq.alloc_workspace(self.g, len(self.lens), w.q_heads, self.bt.shape[1], device=DEV)
        args = (self.g, dev_bits(q), dev(self.bt), dev(self.lens), out, ws, softmax_scale)
        if split_calls:
            kvq.decode_partial(*args)
            kvq.decode_merge(*args)
        else:
            kvq.decode_attn(*args)
        st = kvq.last_device_error()
        assert st == kvq.OK, kvq.status_string(st)
        return out.cpu().numpy().astype(np.float64)

    def oracle_decode(self, seqs=None, q: np.ndarray | None = None, softmax_scale: float = 0.0):
        seqs = self.oracle_seqs if seqs is None else list(seqs)
        q = self.q if q is None else q
        return self.o.decode_attn(q[seqs], self.bt[seqs], self.lens[seqs], self.w.q_heads, softmax_scale)

    def used_rows(self, seqs=None) -> np.ndarray:
        """Pool row indices ([page][head][offset]) written for these sequences."""
        seqs = self.oracle_seqs if seqs is None else seqs
        w = self.w
        rows = []
        for b in seqs:
            t = np.arange(self.lens[b])
            pages = self.bt[b, t // w.page_size].astype(np.int64)
            for h in range(w.kv_heads):
                rows.append((pages * w.kv_heads + h) * w.page_size + t % w.page_size)
        return np.concatenate(rows) if rows else np.zeros(0, np.int64)

    def compare_cache(self, full: bool = True):
        """Bit-exact comparison of codes, scales (and zeros).  full=True compares
        the whole pools (unwritten rows are zero on both sides)."""
        w = self.w
        cb = w.head_dim // 2 if w.scheme in ("int4", "int4sym") else w.head_dim
        mb = {"int4": (w.head_dim // 32) * 2, "int4sym": (w.head_dim // 32) * 4}.get(w.scheme, 4)
        names = ["k_codes", "v_codes", "k_scales", "v_scales"] + (["k_zeros", "v_zeros"] if w.scheme == "int4" else [])
        rows = None if full else self.used_rows()
        for name in names:
            g = self.g.pool(name)  # both tiers, page ids in order
            o = getattr(self.o, name).view(np.uint8).reshape(-1)
            assert not g[o.size:].any(), f"{name}: bytes written past the table's pages"
            g = g[:o.size]
            width = cb if "codes" in name else mb
            if rows is not None:
                g = g.reshape(-1, width)[rows]
                o = o.reshape(-1, width)[rows]
            if not np.array_equal(g, o):
                bad = np.nonzero((g != o).reshape(g.shape[0], -1).any(axis=-1) if g.ndim > 1 else g != o)[0]
                raise AssertionError(f"{name}: {bad.size} rows/bytes differ, first {bad[:5]}")


def attn_errors(got: np.ndarray, ref: np.ndarray):
    d = np.abs(got - ref)
    return float(d.max()), float(d.sum() / max(np.abs(ref).sum(), 1e-300))


def assert_attn_close(got, ref, what=""):
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    max_abs, mean_rel = attn_errors(got, ref)
    assert max_abs <= ATOL and mean_rel <= MEAN_REL, f"{what}: max_abs={max_abs:.3e} mean_rel={mean_rel:.3e}"
    return max_abs, mean_rel
