"""GPU parity of the INT8 scheme with per-channel K scales ("int8kc"): the
append that keeps bf16 residual rows, the seal that re-quantizes a full
page's K per channel, and the tensor-core decode over open and sealed pages,
each against the CPU oracle on the same seeded inputs.  Pools (codes,
scales, channel factors, residual rows) must be bit-exact; attention within
the tolerances of the other schemes.

The per-channel reading ("KV Cache Optimization: Strategies for Faster LLM
Inference", section "KV Cache Quantization: When and How to Compress"): one
K scale per (page, KV head, channel), fixed when the page is sealed from its
bf16 rows."""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

import dynamically_quantized_paged_gb300 as kvq
import kvq_inputs as inp
import oracle
from gpu_harness import DEV, assert_attn_close, dev, dev_bits

pytestmark = pytest.mark.gpu


def _work(H, G, D, P, seed, batch, outliers=3):
    return inp.Workload(0, "kchan", "int8kc", 1, batch, H * G, H, D, P, ("fixed", 0), seed=seed,
                        outlier_pairs=outliers, outlier_gain=12.0)


class KcCase:
    """Device cache and oracle image driven through the same appends and
    seals.  Each logical page of each sequence owns one residual slot
    (page_slot); `steps` final tokens of every sequence are appended one per
    call, as decode steps, and every page is sealed in the call after the
    append that fills it."""

    def __init__(self, w, lens, steps=0, host_pages=0, spare=2, table_seed=None, chunk=4096,
                 seq_slots=False):
        self.w, self.lens = w, np.asarray(lens, np.int32)
        P, H, D = w.page_size, w.kv_heads, w.head_dim
        self.bt, npg = inp.page_table(self.lens, P, w.seed if table_seed is None else table_seed, spare)
        need = inp.pages_needed(self.lens, P)
        # residual slot of logical page i of sequence b: one per sequence when
        # seq_slots (reused page after page), else one per page
        starts = np.concatenate([[0], np.cumsum(need)])
        self.page_slot = lambda b, i: b if seq_slots else int(starts[b] + i)
        nslots = len(self.lens) if seq_slots else int(starts[-1])
        self.g = kvq.PagedKVCache("int8kc", npg - host_pages, P, H, D, device=DEV, host_pages=host_pages,
                                  resid_slots=max(nslots, 1))
        self.o = oracle.OracleCache("int8kc", npg, P, H, D, resid_slots=max(nslots, 1))
        self.rows = {b: inp.kv_rows(w, 0, b, 0, int(L)) for b, L in enumerate(self.lens)}

        def append(tok):  # tok: list of (b, t0, t1)
            if not tok:
                return
            sl = np.concatenate([inp.slots(self.bt, b, np.arange(t0, t1), P) for b, t0, t1 in tok])
            rs = np.concatenate([[self.page_slot(b, t // P) for t in range(t0, t1)] for b, t0, t1 in tok])
            k = np.concatenate([self.rows[b][0][t0:t1] for b, t0, t1 in tok])
            v = np.concatenate([self.rows[b][1][t0:t1] for b, t0, t1 in tok])
            rs = rs.astype(np.int32)
            kvq.append_kchan(self.g, dev(sl), dev(rs), dev_bits(k), dev_bits(v))
            assert self.o.append(sl, k, v, resid_slot=rs) == 0
            full = [(b, t // P) for b, t0, t1 in tok for t in range(t0, t1) if t % P == P - 1]
            if full:  # seal the pages these tokens completed
                pg = np.array([self.bt[b, i] for b, i in full], np.int32)
                sl2 = np.array([self.page_slot(b, i) for b, i in full], np.int32)
                kvq.seal_pages(self.g, dev(pg), dev(sl2))
                assert self.o.seal(pg, sl2) == 0
            self.sealed += len(full)

        self.sealed = 0
        pre = np.maximum(self.lens - steps, 0)
        if seq_slots:  # token by token from the start
            for t in range(int(self.lens.max())):
                append([(b, t, t + 1) for b, L in enumerate(self.lens) if t < L])
        else:
            for c0 in range(0, int(pre.max(initial=0)), chunk):
                append([(b, c0, min(int(L0), c0 + chunk)) for b, L0 in enumerate(pre) if L0 > c0])
            for s in range(steps):
                append([(b, int(L0) + s, int(L0) + s + 1) for b, (L0, L) in enumerate(zip(pre, self.lens))
                        if L0 + s < L])
        self.q = inp.queries(dataclasses.replace(w, batch=len(self.lens)), 0)
        torch.cuda.synchronize()
        st = kvq.last_device_error()
        assert st == kvq.OK, kvq.status_string(st)

    def compare_pools(self):
        for name in ("k_codes", "v_codes", "k_scales", "v_scales", "k_chan"):
            g = self.g.pool(name)
            o = getattr(self.o, name).view(np.uint8).reshape(-1)
            assert g.size == o.size, name
            if not np.array_equal(g, o):
                raise AssertionError(f"{name}: {(g != o).sum()} bytes differ")
        assert np.array_equal(self.g.k_resid.cpu().numpy(), self.o.k_resid.view(np.uint8))

    def decode(self, q=None, bt=None):
        q = self.q if q is None else q
        bt = self.bt if bt is None else bt
        w = self.w
        out = torch.full((len(self.lens), w.q_heads, w.head_dim), float("nan"), dtype=torch.float32, device=DEV)
        ws = kvq.alloc_workspace(self.g, len(self.lens), w.q_heads, bt.shape[1], device=DEV)
        kvq.decode_attn(self.g, dev_bits(q), dev(bt), dev(self.lens), out, ws)
        st = kvq.last_device_error()
        assert st == kvq.OK, kvq.status_string(st)
        return out.cpu().numpy().astype(np.float64)


RAGGED = [0, 1, 15, 16, 17, 40, 77, 130, 33, 64]


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_kchan_append_seal_decode(D, G):
    w = _work(2, G, D, 16, seed=900 + 10 * G + D, batch=len(RAGGED))
    c = KcCase(w, RAGGED, steps=3)
    assert c.sealed > 10
    c.compare_pools()
    got = c.decode()
    ref = c.o.decode_attn(c.q, c.bt, c.lens, w.q_heads)
    assert_attn_close(got, ref, f"int8kc d{D} G{G}")
    assert np.all(got[0] == 0)


def test_kchan_bf16_output_and_two_launch_form():
    """The per-channel decode through the other output paths: bf16 rows equal
    the fp32 rows rounded to nearest even, and the two-launch form
    (partial, then merge) gives bitwise the one-launch output."""
    w = _work(2, 8, 128, 16, seed=956, batch=len(RAGGED))
    c = KcCase(w, RAGGED, steps=2)
    ref32 = c.decode()
    B, Hq, D = len(RAGGED), w.q_heads, w.head_dim
    args = (dev_bits(c.q), dev(c.bt), dev(c.lens))
    ws = kvq.alloc_workspace(c.g, B, Hq, c.bt.shape[1], device=DEV)
    o16 = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=DEV)
    kvq.decode_attn(c.g, *args, o16, ws)
    o2 = torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device=DEV)
    kvq.decode_partial(c.g, *args, o2, ws)
    kvq.decode_merge(c.g, *args, o2, ws)
    assert kvq.last_device_error() == kvq.OK
    want16 = torch.from_numpy(ref32.astype(np.float32)).to(torch.bfloat16)
    assert torch.equal(o16.cpu().view(torch.int16), want16.view(torch.int16))
    assert np.array_equal(o2.cpu().numpy().astype(np.float64), ref32)


def test_kchan_page_32_and_host_tier():
    w = _work(2, 4, 128, 32, seed=951, batch=len(RAGGED))
    c = KcCase(w, RAGGED, steps=5, host_pages=6)
    assert (c.bt >= c.g.num_pages).any()
    c.compare_pools()
    assert_attn_close(c.decode(), c.o.decode_attn(c.q, c.bt, c.lens, w.q_heads), "int8kc page 32, host tier")


def test_kchan_one_residual_slot_per_sequence_reused():
    """Token-by-token appends from the first token, each sequence keeping one
    residual slot that every one of its pages reuses after the previous seal."""
    lens = [35, 20, 48, 1, 16]
    w = _work(2, 4, 64, 16, seed=952, batch=len(lens))
    c = KcCase(w, lens, seq_slots=True)
    assert c.sealed == 2 + 1 + 3 + 0 + 1
    c.compare_pools()
    assert_attn_close(c.decode(), c.o.decode_attn(c.q, c.bt, c.lens, w.q_heads), "int8kc reused slots")


def test_kchan_llama3_8b_layer_shape():
    """The Llama-3-8B layer shape (B = 32, lengths U[512, 4096], 8 KV heads,
    GQA 4, d 128, page 16): a chunked prefill with every full page sealed,
    then two decode steps."""
    lens = inp.seq_lens(inp.WORKLOADS[2])
    w = _work(8, 4, 128, 16, seed=953, batch=len(lens), outliers=10)
    c = KcCase(w, lens, steps=2)
    c.compare_pools()
    assert_attn_close(c.decode(), c.o.decode_attn(c.q, c.bt, c.lens, w.q_heads), "int8kc llama3-8b shape")


def test_kchan_copy_page_moves_channel_factors_between_tiers():
    lens = [64, 40]
    w = _work(2, 4, 128, 16, seed=954, batch=2)
    c = KcCase(w, lens, host_pages=0, spare=3)
    before = c.decode()
    # offload sequence 0's second page to a host page and decode through it
    g2 = kvq.PagedKVCache("int8kc", c.g.num_pages, 16, 2, 128, device=DEV, host_pages=2, resid_slots=1)
    for name in ("k_codes", "v_codes", "k_scales", "v_scales", "k_chan"):
        getattr(g2, name).copy_(getattr(c.g, name))
    src, dst = int(c.bt[0, 1]), c.g.num_pages + 1
    kvq.copy_page(g2, src, dst)
    torch.cuda.synchronize()
    H, D = 2, 128
    chan = g2.pool("k_chan").reshape(-1, H * D * 2)
    assert np.array_equal(chan[src], chan[dst]) and chan[src].any()
    bt2 = c.bt.copy()
    bt2[0, 1] = dst
    c.g, g_old = g2, c.g
    after = c.decode(bt=bt2)
    assert np.array_equal(before, after)


def test_kchan_bad_ids_flagged_and_skipped():
    w = _work(1, 4, 64, 16, seed=955, batch=1)
    c = KcCase(w, [32], spare=2)
    codes_before = c.g.pool("k_codes").copy()
    # a residual slot outside the pool: nothing written for that token
    k = dev_bits(inp.to_bf16_bits(np.ones((1, 1, 64), np.float32)))
    free = int(np.setdiff1d(np.arange(c.g.num_pages), c.bt[c.bt >= 0])[0])
    kvq.append_kchan(c.g, dev(np.array([free * 16], np.int64)), dev(np.array([99], np.int32)), k, k)
    assert kvq.last_device_error() == 4  # KVQ_ERR_BAD_TABLE
    assert np.array_equal(c.g.pool("k_codes"), codes_before)
    # a seal naming a page outside the pool is skipped; the valid pair is done
    kvq.seal_pages(c.g, dev(np.array([10 ** 6, int(c.bt[0, 0])], np.int32)), dev(np.array([0, 0], np.int32)))
    assert kvq.last_device_error() == 4
    assert c.o.seal(np.array([int(c.bt[0, 0])], np.int32), np.array([0], np.int32)) == 0
    c.compare_pools()
    # the fused decode-append has no residual slots: refused
    with pytest.raises(kvq.KvqError) as e:
        out = torch.zeros((1, 4, 64), dtype=torch.float32, device=DEV)
        ws = kvq.alloc_workspace(c.g, 1, 4, c.bt.shape[1], device=DEV)
        kvq.decode_attn_append(c.g, k[0:1], k[0:1], dev_bits(c.q), dev(c.bt), dev(c.lens), out, ws)
    assert e.value.status == 7  # KVQ_ERR_UNSUPPORTED


def test_kchan_step_replayed_from_a_cuda_graph():
    """A per-channel decode step (append of each sequence's token keeping its
    K rows, the seal of the pages it fills, the decode) recorded in a CUDA
    graph and replayed gives the eager step's pools and output bit for bit."""
    lens = np.array([31, 48, 17, 64], np.int32)  # tokens 31, 47 and 63 fill pages
    w = _work(2, 4, 128, 16, seed=957, batch=len(lens))
    c = KcCase(w, lens, steps=1)
    P = w.page_size
    # the step's token of each sequence again (same bytes), its slot, its page's slot
    k_new = np.concatenate([c.rows[b][0][L - 1:L] for b, L in enumerate(lens)])
    v_new = np.concatenate([c.rows[b][1][L - 1:L] for b, L in enumerate(lens)])
    sl = np.concatenate([inp.slots(c.bt, b, np.array([L - 1]), P) for b, L in enumerate(lens)])
    rs = np.array([c.page_slot(b, (L - 1) // P) for b, L in enumerate(lens)], np.int32)
    fill = [(b, (L - 1) // P) for b, L in enumerate(lens) if (L - 1) % P == P - 1]
    pg = np.array([c.bt[b, i] for b, i in fill], np.int32)
    ps = np.array([c.page_slot(b, i) for b, i in fill], np.int32)
    dk, dv, dsl, drs, dpg, dps = (dev_bits(k_new), dev_bits(v_new), dev(sl), dev(rs), dev(pg), dev(ps))
    dq, dbt, dlen = dev_bits(c.q), dev(c.bt), dev(c.lens)
    B, Hq, D = len(lens), w.q_heads, w.head_dim
    ws = kvq.alloc_workspace(c.g, B, Hq, c.bt.shape[1], device=DEV)
    out = torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device=DEV)

    def step(stream=None):
        kvq.append_kchan(c.g, dsl, drs, dk, dv, stream=stream)
        kvq.seal_pages(c.g, dpg, dps, stream=stream)
        kvq.decode_attn(c.g, dq, dbt, dlen, out, ws, stream=stream)

    step()
    torch.cuda.synchronize()
    eager = out.cpu().numpy().copy()
    pools = {n: c.g.pool(n).copy() for n in ("k_codes", "v_codes", "k_scales", "v_scales", "k_chan")}
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step(stream=s)
    out.fill_(float("nan"))
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert kvq.last_device_error() == kvq.OK
    assert np.array_equal(out.cpu().numpy(), eager)
    for n, a in pools.items():
        assert np.array_equal(c.g.pool(n), a), n
    c.compare_pools()
    assert_attn_close(eager.astype(np.float64), c.o.decode_attn(c.q, c.bt, c.lens, Hq), "int8kc graph step")


def test_kchan_page_48():
    """A page size that is a multiple of 16 but not a power of two: the seal
    walks its page in three 16-token chunks."""
    lens = [47, 48, 49, 100, 5]
    w = _work(2, 2, 64, 48, seed=958, batch=len(lens))
    c = KcCase(w, lens, steps=2)
    assert c.sealed >= 4
    c.compare_pools()
    assert_attn_close(c.decode(), c.o.decode_attn(c.q, c.bt, c.lens, w.q_heads), "int8kc page 48")


def test_kchan_sealed_page_reopened():
    """A sealed page that is freed and reused: the token appended at its
    offset 0 sets its channel factors back to 1.0 (every head) and takes the
    token rule; the pools match the oracle, which does the same."""
    lens = [32]
    w = _work(2, 4, 128, 16, seed=959, batch=1)
    c = KcCase(w, lens, spare=2)
    page = int(c.bt[0, 0])
    chan_before = c.g.pool("k_chan").view(np.uint16).reshape(-1, 2, 128)[page].copy()
    assert np.any(chan_before != 0x3C00)     # sealed: factors other than 1.0
    r = np.random.default_rng(5)
    k = inp.to_bf16_bits(r.standard_normal((1, 2, 128)).astype(np.float32))
    v = inp.to_bf16_bits(r.standard_normal((1, 2, 128)).astype(np.float32))
    sl = np.array([page * 16], np.int64)
    rs = np.array([c.page_slot(0, 0)], np.int32)
    kvq.append_kchan(c.g, dev(sl), dev(rs), dev_bits(k), dev_bits(v))
    assert c.o.append(sl, k, v, resid_slot=rs) == 0
    torch.cuda.synchronize()
    assert kvq.last_device_error() == kvq.OK
    chan = c.g.pool("k_chan").view(np.uint16).reshape(-1, 2, 128)[page]
    assert np.all(chan == 0x3C00)
    c.compare_pools()
