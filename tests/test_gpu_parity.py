"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Codes, scales and zero-points must be bit-exact; attention must be within
max-abs 1e-2 and mean-rel 2e-3 of the oracle's fp64 attention over the same
dequantized cache.  Covers the five workloads at full size (sampled where the
oracle would take minutes), ragged and degenerate shapes, tie-breaking
inputs, page-permutation invariance and the device-side error flags."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU-only machines, never run there
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import dynamically_quantized_paged_gb300 as kvq  # noqa: E402
import kvq_inputs as inp  # noqa: E402
import oracle  # noqa: E402
from gpu_harness import Case, DEV, assert_attn_close, dev, dev_bits  # noqa: E402


def small(scheme, Hq, Hkv, D, P, seed=7, outliers=2):
    return inp.Workload(0, "edge", scheme, 1, 1, Hq, Hkv, D, P, ("fixed", 0), seed=seed,
                        outlier_pairs=outliers, outlier_gain=8.0)


# ------------------------------------------------------------- full workloads
@pytest.mark.parametrize("cid", [1, 2, 5])
def test_workload_full_parity(cid):
    w = inp.WORKLOADS[cid]
    case = Case(w, inp.seq_lens(w))
    case.compare_cache(full=True)
    got = case.decode()
    ref = case.oracle_decode()
    assert_attn_close(got, ref, f"workload {cid}")


def test_workload3_fp8_70b_layer():
    """Every sequence's codes and scales bit-exact (whole pools); attention on a
    seeded sample of sequences (the fp64 oracle takes minutes on all 64)."""
    w = inp.WORKLOADS[3]
    lens = inp.seq_lens(w)
    r = np.random.default_rng(33)
    sample = sorted(set(r.choice(len(lens), 6, replace=False).tolist()) | {int(np.argmax(lens)), int(np.argmin(lens))})
    case = Case(w, lens)
    case.compare_cache(full=True)
    got = case.decode()
    ref = case.oracle_decode(seqs=sample)
    assert_attn_close(got[sample], ref, "workload 3 (sampled sequences)")


def test_workload4_int4_eight_layers():
    """All 8 layers: every sequence's codes, scales and zero-points bit-exact
    (whole pools); attention on two sequences per layer."""
    w = inp.WORKLOADS[4]
    lens = inp.seq_lens(w)
    for layer in range(w.layers):
        sample = [layer % w.batch, (layer * 5 + 3) % w.batch]
        case = Case(w, lens, layer=layer)
        case.compare_cache(full=True)
        got = case.decode()
        assert_attn_close(got[sample], case.oracle_decode(seqs=sample), f"workload 4 layer {layer}")
        del case
        torch.cuda.empty_cache()


def test_int4sym_eight_layer_shapes():
    """The 8-layer INT4 workload's shapes (16 x 32768 tokens, Hq 32 / Hkv 8,
    d 128, page 32) under symmetric INT4, one layer: whole pools bit-exact,
    attention on three sequences."""
    import dataclasses
    w = dataclasses.replace(inp.WORKLOADS[4], scheme="int4sym", layers=1)
    lens = inp.seq_lens(w)
    case = Case(w, lens)
    case.compare_cache(full=True)
    got = case.decode()
    sample = [0, 7, 15]
    assert_attn_close(got[sample], case.oracle_decode(seqs=sample), "symmetric INT4, 8-layer shapes")


@pytest.mark.parametrize("shape", [("int8", 32, 8, 128, 16), ("int4", 32, 8, 128, 32), ("fp8", 64, 8, 128, 16),
                                   ("int4sym", 16, 8, 64, 16)], ids=lambda s: "-".join(map(str, s)))
def test_bf16_output_is_the_rounded_fp32_output(shape):
    """kvq_decode_attn_out with bf16 output writes, element for element, the
    fp32 output of kvq_decode_attn rounded to nearest even: final rows of
    whole segments, merged split segments (a 40000-token sequence) and the
    zero rows of empty sequences, on both decode kernels."""
    scheme, Hq, Hkv, D, P = shape
    w = small(scheme, Hq, Hkv, D, P)
    lens = np.array([1, 0, 300, 5000, 17, 40000], np.int32)
    case = Case(w, lens, oracle_seqs=[])
    ref32 = case.decode()
    out = torch.full((len(lens), Hq, D), float("nan"), dtype=torch.bfloat16, device=DEV)
    ws = kvq.alloc_workspace(case.g, len(lens), Hq, case.bt.shape[1], device=DEV)
    kvq.decode_attn(case.g, dev_bits(case.q), dev(case.bt), dev(case.lens), out, ws)
    assert kvq.last_device_error() == kvq.OK
    want = torch.from_numpy(ref32.astype(np.float32)).to(torch.bfloat16)
    assert torch.equal(out.cpu().view(torch.int16), want.view(torch.int16))


# ------------------------------------------------------------- edge cases
SHAPES = [  # scheme, Hq, Hkv, D, P
    ("int8", 8, 8, 64, 16), ("int8", 8, 4, 64, 16), ("int8", 16, 4, 128, 32), ("int8", 32, 4, 128, 16),
    ("fp8", 4, 4, 128, 16), ("fp8", 16, 8, 64, 32), ("fp8", 32, 8, 128, 16), ("fp8", 8, 2, 128, 48),
    ("int4", 8, 8, 128, 32), ("int4", 16, 8, 64, 16), ("int4", 16, 4, 128, 16), ("int4", 64, 8, 128, 32),
    # the remaining (head_dim, GQA ratio) instantiations of each scheme
    ("int8", 16, 16, 128, 16), ("int8", 16, 8, 128, 16), ("int8", 16, 4, 64, 16), ("int8", 32, 4, 64, 16),
    ("fp8", 8, 8, 64, 16), ("fp8", 16, 8, 128, 16), ("fp8", 32, 8, 64, 16), ("fp8", 64, 8, 64, 16),
    ("int4", 8, 8, 64, 16), ("int4", 32, 16, 128, 16), ("int4", 32, 8, 64, 16), ("int4", 64, 8, 64, 16),
    # symmetric INT4: every (head_dim, GQA ratio) instantiation
    ("int4sym", 8, 8, 128, 16), ("int4sym", 8, 8, 64, 32), ("int4sym", 16, 8, 128, 16), ("int4sym", 16, 8, 64, 16),
    ("int4sym", 16, 4, 128, 32), ("int4sym", 32, 8, 64, 16), ("int4sym", 64, 8, 128, 16), ("int4sym", 32, 4, 64, 16),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "-".join(map(str, s)))
def test_ragged_and_degenerate_lengths(shape):
    scheme, Hq, Hkv, D, P = shape
    w = small(scheme, Hq, Hkv, D, P)
    lens = np.array([1, 0, 17, 15, 16, 300, 2049, 33, 0, 5000, 129], np.int32)
    case = Case(w, lens, spare=5)
    case.compare_cache(full=True)
    got = case.decode()
    ref = case.oracle_decode()
    assert_attn_close(got, ref, str(shape))
    assert np.all(got[1] == 0) and np.all(got[8] == 0)  # empty sequences give zero rows


def test_single_sequence_many_splits_and_custom_scale():
    w = small("int8", 16, 2, 128, 16)
    case = Case(w, np.array([40000], np.int32))
    case.compare_cache(full=True)
    for scale in (0.0, 0.05):
        got = case.decode(softmax_scale=scale)
        assert_attn_close(got, case.oracle_decode(softmax_scale=scale), f"scale {scale}")


def test_page_permutation_is_bitwise_invariant():
    w = small("fp8", 16, 4, 128, 16)
    lens = np.array([700, 3000, 45, 1600], np.int32)
    a = Case(w, lens, table_seed=1, oracle_seqs=[])
    b = Case(w, lens, table_seed=2, oracle_seqs=[], spare=40)
    assert not np.array_equal(a.bt, b.bt)
    assert np.array_equal(a.decode(), b.decode())


def test_workspace_garbage_is_harmless():
    """The workspace needs no initialization: arbitrary bytes in it (stale
    arrival counters included) must not change the result."""
    w = small("int8", 32, 8, 128, 16)
    lens = np.array([9000, 40, 2000, 0, 777], np.int32)
    case = Case(w, lens)
    ref = case.oracle_decode()
    for fill in (0x00, 0xFF, 0xA5):
        out = torch.full((len(lens), 32, 128), float("nan"), dtype=torch.float32, device=DEV)
        ws = kvq.alloc_workspace(case.g, len(lens), 32, case.bt.shape[1], device=DEV)
        ws.fill_(fill)
        kvq.decode_attn(case.g, dev_bits(case.q), dev(case.bt), dev(lens), out, ws)
        assert kvq.last_device_error() == kvq.OK
        assert_attn_close(out.cpu().numpy().astype(np.float64), ref, f"fill {fill:#x}")


def test_two_launch_form_matches_one_call():
    w = small("int4", 32, 4, 128, 32)
    case = Case(w, np.array([5000, 70, 2300], np.int32), oracle_seqs=[])
    assert np.array_equal(case.decode(), case.decode(split_calls=True))


# ------------------------------------------------------------- crafted inputs
def _tie_rows(scheme, D):
    """Rows whose quotients land exactly on rounding ties."""
    f = np.zeros((4, D), np.float32)
    if scheme == "int8":       # absmax 127 -> scale 1: x.5 ties
        f[:, 0] = 127.0
        f[:, 1:] = (np.arange(1, D) % 40 - 20) + 0.5
        f[3] = 0.0             # all-zero row: scale 1.0, zero codes
    elif scheme == "fp8":      # absmax 448 -> scale 1: E4M3 midpoints
        vals = np.array([oracle.e4m3_value(c) for c in range(0x7F)])
        mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
        f[:, 0] = 448.0
        f[:, 1:] = np.resize(np.concatenate([mids, -mids]), D - 1)
        f[3] = 0.0
    elif scheme == "int4sym":  # group absmax 7 -> scale 1: x.5 ties
        f[:] = np.resize((np.arange(2 * D) % 14 - 7) + 0.5, (4, D))
        f[:, ::32] = 7.0
        f[1, ::32] = -7.0                                      # negative absmax
        f[2, :32] = 0.0                                        # an all-zero group
        f[2, 32:64] = np.float32(2.0 ** -30) * (np.arange(32) % 7 - 3)  # a tiny group
        f[3] = 0.0                                             # an all-zero row
    else:                      # INT4: constant groups, tiny minima, exact ties
        f[0] = 0.5
        f[1] = np.tile(np.concatenate([[-1.5, 6.0, 0.0, 0.25, 0.75, 1.25], np.full(26, 2.0)]), D // 32)
        f[2] = np.float32(2.0 ** -30) * (np.arange(D) % 7)
        f[3] = 0.0
    return inp.to_bf16_bits(f)


@pytest.mark.parametrize("scheme", ["int8", "fp8", "int4", "int4sym"])
def test_tie_breaking_and_zero_rows_bit_exact(scheme):
    D, H = 128, 2
    w = small(scheme, 4, H, D, 16)
    rows = _tie_rows(scheme, D)

    def kv(b, s0, s1):
        n = s1 - s0
        k = np.stack([rows[(s0 + i) % 4] for i in range(n)])[:, None, :].repeat(H, axis=1)
        v = np.stack([rows[(s0 + i + 1) % 4] for i in range(n)])[:, None, :].repeat(H, axis=1)
        return np.ascontiguousarray(k), np.ascontiguousarray(v)

    case = Case(w, np.array([64, 23], np.int32), kv_override=kv)
    case.compare_cache(full=True)
    assert_attn_close(case.decode(), case.oracle_decode(), scheme)


@pytest.mark.parametrize("scheme", ["int8", "fp8", "int4", "int4sym"])
def test_tiny_magnitude_rows_bit_exact(scheme):
    """Rows (and 32-channel groups) whose largest magnitude is tiny, down to
    the smallest bf16 subnormal: the reciprocal of such a scale overflows, so
    the append must take the exact quotient; codes and scales equal the
    oracle's."""
    D, H, P = 128, 1, 16
    r = np.random.default_rng(41)
    bits = []
    for top in (0x0001, 0x0003, 0x0010, 0x007F, 0x0080, 0x0100, 0x0800, 0x0C00):  # subnormals .. ~1e-36
        for _ in range(4):
            row = r.integers(0, top + 1, size=D).astype(np.uint16)
            row[r.integers(0, D)] = top
            row[r.random(D) < 0.5] |= 0x8000
            bits.append(row)
    rows = np.stack(bits)
    T = rows.shape[0]
    k = rows.reshape(T, H, D)
    v = np.ascontiguousarray(k[::-1])
    slots = np.arange(T, dtype=np.int64)
    npg = (T + P - 1) // P
    g = kvq.PagedKVCache(scheme, npg, P, H, D, device=DEV)
    o = oracle.OracleCache(scheme, npg, P, H, D)
    kvq.append(g, dev(slots), dev_bits(k), dev_bits(v))
    assert o.append(slots, k, v) == 0
    torch.cuda.synchronize()
    assert kvq.last_device_error() == kvq.OK
    names = ["k_codes", "v_codes", "k_scales", "v_scales"] + (["k_zeros", "v_zeros"] if scheme == "int4" else [])
    for name in names:
        got = g.codes_rowmajor(name[0]).reshape(-1) if "codes" in name else getattr(g, name).cpu().numpy()
        want = getattr(o, name).view(np.uint8)
        bad = np.nonzero(got.view(np.uint8) != want)[0]
        assert bad.size == 0, f"{scheme} {name}: {bad.size} bytes differ, first at {bad[:5]}"


# ------------------------------------------------------------- device-side errors
def test_bad_page_id_is_flagged_not_faulted():
    w = small("int8", 8, 4, 64, 16)
    case = Case(w, np.array([100, 50], np.int32), oracle_seqs=[])
    bt = case.bt.copy()
    bt[0, 2] = case.num_pages + 1000  # outside the pool
    out = torch.zeros((2, 8, 64), dtype=torch.float32, device=DEV)
    ws = kvq.alloc_workspace(case.g, 2, 8, bt.shape[1], device=DEV)
    kvq.decode_attn(case.g, dev_bits(case.q), dev(bt), dev(case.lens), out, ws)
    assert kvq.last_device_error() == 4
    assert kvq.last_device_error() == 0  # reading clears the flag
    assert torch.isfinite(out).all()
    kvq.validate_tables(case.g, dev(bt), dev(case.lens))
    assert kvq.last_device_error() == 4


def test_sequence_longer_than_its_table_is_flagged():
    w = small("int8", 8, 4, 64, 16)
    case = Case(w, np.array([64], np.int32), oracle_seqs=[])
    lens = np.array([64 + 10 * 16 * case.bt.shape[1]], np.int32)
    out = torch.zeros((1, 8, 64), dtype=torch.float32, device=DEV)
    ws = kvq.alloc_workspace(case.g, 1, 8, case.bt.shape[1], device=DEV)
    kvq.decode_attn(case.g, dev_bits(case.q), dev(case.bt), dev(lens), out, ws)
    assert kvq.last_device_error() == 4


def test_append_slot_outside_pool_is_flagged_and_negative_slots_skipped():
    w = small("fp8", 8, 4, 64, 16)
    g = kvq.PagedKVCache("fp8", 2, 16, 4, 64, device=DEV)
    k, v = inp.kv_rows(w, 0, 0, 0, 3)
    kvq.append(g, dev(np.array([-1, 5, 32], np.int64)), dev_bits(k), dev_bits(v))
    assert kvq.last_device_error() == 4
    codes = g.k_codes.cpu().numpy().reshape(2, 4, 16, 64)
    assert codes[0, :, 5].any() and not codes[0, :, 0].any() and not codes[1].any()
    # a block table given to append is checked too
    bt = np.array([[0, 1, 7]], np.int32)
    kvq.append(g, dev(np.array([1], np.int64)), dev_bits(k[:1]), dev_bits(v[:1]), block_table=dev(bt))
    assert kvq.last_device_error() == 4


def test_graph_replay_matches_eager_call():
    """A decode_attn captured in a CUDA graph and replayed several times on
    one workspace gives the eager call's output bit for bit (the arrival
    counters are cleared by each call, so the replayed generation is
    harmless)."""
    w = small("int8", 32, 8, 128, 16)
    lens = np.array([9000, 40, 2000, 0, 777, 3000], np.int32)
    case = Case(w, lens, oracle_seqs=[])
    ref = case.decode()
    q, bt, sl = dev_bits(case.q), dev(case.bt), dev(lens)
    out = torch.full((len(lens), 32, 128), float("nan"), dtype=torch.float32, device=DEV)
    ws = kvq.alloc_workspace(case.g, len(lens), 32, case.bt.shape[1], device=DEV)
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):  # warm-up outside capture (sets kernel attributes)
        kvq.decode_attn(case.g, q, bt, sl, out, ws, stream=stream)
    torch.cuda.current_stream().wait_stream(stream)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        kvq.decode_attn(case.g, q, bt, sl, out, ws, stream=stream)
    for _ in range(3):
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert kvq.last_device_error() == kvq.OK
        assert np.array_equal(out.cpu().numpy().astype(np.float64), ref)


def test_decode_right_after_append_sees_the_new_tokens():
    """The decode is launched so that it may be scheduled while the append
    ahead of it on the stream still runs.  Appending each sequence's newest
    token and decoding at once, with no synchronization between the two
    calls, must attend over that token: eagerly, and replayed from a CUDA
    graph holding both calls."""
    w = small("int8", 32, 8, 128, 16)
    full = np.array([3001, 17, 4096, 1, 800, 2500], np.int32)
    bt, num_pages = inp.page_table(full, w.page_size, w.seed, 3)
    case = Case(w, full - 1, block_table=bt, num_pages=num_pages)
    ks, vs, sl = [], [], []
    for b, L in enumerate(full):
        k, v = inp.kv_rows(w, 0, b, int(L) - 1, int(L))
        ks.append(k)
        vs.append(v)
        sl.append(inp.slots(bt, b, np.array([L - 1]), w.page_size))
    k_new, v_new, s_new = np.concatenate(ks), np.concatenate(vs), np.concatenate(sl)
    assert case.o.append(s_new, k_new, v_new) == 0
    ref = case.o.decode_attn(case.q, bt, full, w.q_heads, 0.0)

    d_s, d_k, d_v = dev(s_new), dev_bits(k_new), dev_bits(v_new)
    q, d_bt, d_len = dev_bits(case.q), dev(bt), dev(full)
    out = torch.full((len(full), w.q_heads, w.head_dim), float("nan"), dtype=torch.float32, device=DEV)
    ws = kvq.alloc_workspace(case.g, len(full), w.q_heads, bt.shape[1], device=DEV)
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        kvq.append(case.g, d_s, d_k, d_v, stream=stream)
        kvq.decode_attn(case.g, q, d_bt, d_len, out, ws, stream=stream)
    stream.synchronize()
    assert kvq.last_device_error() == kvq.OK
    eager = out.cpu().numpy().astype(np.float64)
    assert_attn_close(eager, ref, "decode right after append")
    case.compare_cache(full=True)

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        kvq.append(case.g, d_s, d_k, d_v, stream=stream)
        kvq.decode_attn(case.g, q, d_bt, d_len, out, ws, stream=stream)
    for _ in range(3):
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert kvq.last_device_error() == kvq.OK
        assert np.array_equal(out.cpu().numpy().astype(np.float64), eager)


def quotient_sweep_rows(D=128):
    """bf16 rows (as uint16 bits) in which every positive bf16 value x <= a
    appears, with alternating signs, next to a row maximum a: for a of every
    one of the 128 bf16 mantissas at three exponents.  With a fixed, the 8-bit
    scale is a / qmax, so each row sweeps every bf16 quotient x / s the
    append can meet at that scale mantissa, the ones within a hair of a
    rounding midpoint included."""
    rows = []
    for e in (120, 127, 133):
        for m in range(128):
            a = (e << 7) | m
            xs = np.arange(0, a + 1, dtype=np.uint16)
            xs[1::2] |= 0x8000
            n = D - 1
            pad = (-xs.size) % n
            xs = np.concatenate([xs, np.zeros(pad, np.uint16)]).reshape(-1, n)
            r = np.empty((xs.shape[0], D), np.uint16)
            r[:, 0] = a
            r[:, 1:] = xs
            rows.append(r)
    return np.concatenate(rows)


@pytest.mark.parametrize("scheme", ["int8", "fp8", "int4", "int4sym"])
def test_append_quotient_sweep_bit_exact(scheme):
    """The append divides by the scale with a fast reciprocal product and
    falls back to the exact IEEE quotient only near a rounding midpoint.
    Over every bf16 value at every scale mantissa (~6.3M quotients; the sign
    alternates) its codes, scales and zero-points equal the oracle's, which
    divides exactly every time."""
    D, P, H = 128, 16, 1
    rows = quotient_sweep_rows(D)
    T = rows.shape[0]
    num_pages = (T + P - 1) // P
    k = rows.reshape(T, H, D)
    v = np.ascontiguousarray(k[::-1])
    slots = np.arange(T, dtype=np.int64)
    g = kvq.PagedKVCache(scheme, num_pages, P, H, D, device=DEV)
    o = oracle.OracleCache(scheme, num_pages, P, H, D)
    kvq.append(g, dev(slots), dev_bits(k), dev_bits(v))
    assert o.append(slots, k, v) == 0
    torch.cuda.synchronize()
    assert kvq.last_device_error() == kvq.OK
    names = ["k_codes", "v_codes", "k_scales", "v_scales"] + (["k_zeros", "v_zeros"] if scheme == "int4" else [])
    for name in names:
        got = g.codes_rowmajor(name[0]).reshape(-1) if "codes" in name else getattr(g, name).cpu().numpy()
        want = getattr(o, name).view(np.uint8)
        bad = np.nonzero(got.view(np.uint8) != want)[0]
        assert bad.size == 0, f"{scheme} {name}: {bad.size} bytes differ, first at {bad[:5]}"


@pytest.mark.parametrize("scheme", ["int8", "fp8", "int4", "int4sym"])
def test_shared_prefix_pages_with_copy_on_write(scheme):
    """Sequence B reuses the pages of sequence A's first 100 tokens (six full
    pages shared through the allocator's reference counts); the page where
    the prefix ends is copied with kvq_copy_page before B appends its own
    tokens past the prefix.  The pools equal an oracle cache in which B's
    tokens were all appended into B's own slots, and both sequences decode
    within tolerance."""
    w = small(scheme, 32, 8, 128, 16)
    P, H, D = w.page_size, w.kv_heads, w.head_dim
    La, Lp, Lb = 117, 100, 150
    num_pages = 24
    alloc = kvq.PageAllocator(num_pages, 11)
    g = kvq.PagedKVCache(scheme, num_pages, P, H, D, device=DEV)
    o = oracle.OracleCache(scheme, num_pages, P, H, D)
    ka, va = inp.kv_rows(w, 0, 0, 0, La)
    kb, vb = inp.kv_rows(w, 0, 1, 0, Lb)
    kb[:Lp], vb[:Lp] = ka[:Lp], va[:Lp]          # the shared prefix: the same tokens

    pages_a = alloc.alloc((La + P - 1) // P)
    n_full = Lp // P                              # 6 pages wholly inside the prefix
    alloc.share(pages_a[:n_full + 1])             # B's table starts with A's first 7 pages
    own = alloc.alloc(1)[0]                       # copy-on-write of the page the prefix ends in
    pages_b = pages_a[:n_full] + [own] + alloc.alloc((Lb + P - 1) // P - n_full - 1)
    alloc.free([pages_a[n_full]])                 # B drops its reference to A's page
    bt = np.full((2, len(pages_b)), -1, np.int32)
    bt[0, :len(pages_a)] = pages_a
    bt[1] = pages_b
    assert [alloc.refcount(x) for x in pages_a[:n_full + 1]] == [2] * n_full + [1]

    sa = inp.slots(bt, 0, np.arange(La), P)
    kvq.append(g, dev(sa), dev_bits(ka), dev_bits(va))
    kvq.copy_page(g, pages_a[n_full], own)
    sb = inp.slots(bt, 1, np.arange(Lp, Lb), P)
    kvq.append(g, dev(sb), dev_bits(kb[Lp:]), dev_bits(vb[Lp:]))

    assert o.append(sa, ka, va) == 0
    assert o.append(inp.slots(bt, 1, np.arange(Lb), P), kb, vb) == 0
    torch.cuda.synchronize()
    assert kvq.last_device_error() == kvq.OK
    names = ["k_codes", "v_codes", "k_scales", "v_scales"] + (["k_zeros", "v_zeros"] if scheme == "int4" else [])
    for name in names:
        got = g.codes_rowmajor(name[0]).reshape(-1) if "codes" in name else getattr(g, name).cpu().numpy()
        assert np.array_equal(got.view(np.uint8), getattr(o, name).view(np.uint8)), name

    import dataclasses
    q = inp.queries(dataclasses.replace(w, batch=2), 0)
    lens = np.array([La, Lb], np.int32)
    out = torch.full((2, w.q_heads, D), float("nan"), dtype=torch.float32, device=DEV)
    ws = kvq.alloc_workspace(g, 2, w.q_heads, bt.shape[1], device=DEV)
    kvq.decode_attn(g, dev_bits(q), dev(bt), dev(lens), out, ws)
    assert kvq.last_device_error() == kvq.OK
    ref = o.decode_attn(q, bt, lens, w.q_heads, 0.0)
    assert_attn_close(out.cpu().numpy().astype(np.float64), ref, f"{scheme} shared prefix")
    alloc.close()


# ------------------------------------------------------------ host (cold) tier
@pytest.mark.parametrize("scheme", ["int8", "fp8", "int4", "int4sym"])
@pytest.mark.parametrize("Hq", [32, 64], ids=["gqa4", "gqa8"])
def test_host_tier_pages_are_written_and_read_in_place(scheme, Hq):
    """Half of the pool's pages live in the host tier (page-locked host
    memory): the append writes them and both decode kernels (GQA 4 on the CUDA
    cores, GQA 8 on the tensor cores) read them in place.  The pools over both
    tiers equal the oracle's one-tier pool byte for byte, and the decode equals
    that of an all-device cache with the same tables bit for bit."""
    w = small(scheme, Hq, 8, 128, 16)
    lens = np.array([700, 1, 2049, 16, 333, 0, 1500], np.int32)
    a = Case(w, lens, spare=4, table_seed=3)
    split = Case(w, lens, spare=4, table_seed=3, host_pages=a.num_pages // 2)
    assert split.g.num_pages + split.g.host_pages == a.num_pages
    used = np.unique(split.bt[split.bt >= 0])
    assert (used >= split.g.num_pages).any() and (used < split.g.num_pages).any()
    split.compare_cache(full=True)
    got = split.decode()
    assert np.array_equal(got, a.decode())
    assert_attn_close(got, split.oracle_decode(), f"{scheme} G{Hq // 8} host tier")


@pytest.mark.parametrize("scheme", ["int8", "int4"])
def test_pages_offloaded_to_the_host_tier_and_fetched_back(scheme):
    """kvq_copy_page moves pages between the tiers: every other page of the
    first sequence goes to free host-tier pages (offload; the block table is
    rewritten), then comes back to fresh device pages (fetch).  The decode
    is bit-identical after each move, and a token appended while its page is
    host-resident lands there."""
    w = small(scheme, 32, 8, 128, 16)
    lens = np.array([1000, 300], np.int32)
    c = Case(w, lens, spare=70, extra_host_pages=40)
    ref = c.decode()
    ever_used = set(c.bt[c.bt >= 0].tolist())
    n0 = (int(lens[0]) + 15) // 16
    moved = list(range(0, n0, 2))
    homes = c.bt[0, moved].copy()
    for j, lp in enumerate(moved):           # offload
        dst = c.g.num_pages + j
        kvq.copy_page(c.g, int(c.bt[0, lp]), dst)
        c.bt[0, lp] = dst
    assert all(c.g.tier_of(int(x)) == "host" for x in c.bt[0, moved])
    assert np.array_equal(c.decode(), ref)
    used = set(c.bt[c.bt >= 0].tolist())
    fresh = [x for x in range(c.g.num_pages) if x not in used and x not in set(homes.tolist())][:len(moved)]
    assert len(fresh) == len(moved)
    for lp, dst in zip(moved, fresh):        # fetch
        kvq.copy_page(c.g, int(c.bt[0, lp]), dst)
        c.bt[0, lp] = dst
    assert all(c.g.tier_of(int(x)) == "device" for x in c.bt[0, moved])
    assert np.array_equal(c.decode(), ref)
    # append one token into a host-resident page: the page's bytes match
    # the same append into a device page
    host_page = c.g.num_pages + 39
    dev_page = [x for x in range(c.g.num_pages) if x not in ever_used and x not in fresh][0]  # never written
    k, v = inp.kv_rows(w, 0, 5, 0, 1)
    kvq.append(c.g, dev(np.array([host_page * 16 + 3], np.int64)), dev_bits(k), dev_bits(v))
    kvq.append(c.g, dev(np.array([dev_page * 16 + 3], np.int64)), dev_bits(k), dev_bits(v))
    torch.cuda.synchronize()
    assert kvq.last_device_error() == kvq.OK
    for name in ["k_codes", "v_codes", "k_scales", "v_scales"] + (["k_zeros", "v_zeros"] if scheme == "int4" else []):
        pool = c.g.pool(name)
        per_page = pool.size // (c.g.num_pages + c.g.host_pages)
        hp = pool[host_page * per_page:(host_page + 1) * per_page]
        dp = pool[dev_page * per_page:(dev_page + 1) * per_page]
        assert hp.any() and np.array_equal(hp, dp), name


@pytest.mark.parametrize("scheme", ["int8", "fp8", "int4", "int4sym", "int8kc"])
def test_batched_page_copies_across_tiers(scheme):
    """kvq_copy_pages moves a batch of pages in one launch: device pages to
    free host-tier pages, host pages to free device pages and a device page
    to another (copy-on-write), every pool byte for byte as the pools' host
    copies predict; a pair naming a page outside both tiers is flagged and
    skipped.  The decode is bit-identical through the moved pages."""
    if scheme == "int8kc":
        from test_gpu_kchan import KcCase, _work
        w = _work(8, 4, 128, 16, seed=961, batch=2)
        c = KcCase(w, [1000, 300], host_pages=20, spare=40)
    else:
        w = small(scheme, 32, 8, 128, 16)
        c = Case(w, np.array([1000, 300], np.int32), spare=40, host_pages=20, extra_host_pages=20)
    ref = c.decode()
    total = c.g.num_pages + c.g.host_pages
    used = set(c.bt[c.bt >= 0].tolist())
    free_dev = [x for x in range(c.g.num_pages) if x not in used]
    free_host = [x for x in range(c.g.num_pages, total) if x not in used]
    dev_used = [x for x in c.bt[0] if 0 <= x < c.g.num_pages][:8]
    host_used = [x for x in c.bt.reshape(-1) if x >= c.g.num_pages][:4]
    assert len(dev_used) == 8 and len(host_used) >= 2
    pairs = [(int(a), int(b)) for a, b in zip(dev_used[:5], free_host)]                 # offload
    pairs += [(int(a), int(b)) for a, b in zip(host_used, free_dev[:len(host_used)])]    # fetch
    pairs += [(int(dev_used[5]), int(free_dev[len(host_used)]))]                         # copy-on-write
    names = ["k_codes", "v_codes", "k_scales", "v_scales"] + (["k_zeros", "v_zeros"] if scheme == "int4" else []) + \
        (["k_chan"] if scheme == "int8kc" else [])
    before = {n: c.g.pool(n).reshape(total, -1).copy() for n in names}
    src = np.array([a for a, _ in pairs] + [total + 5], np.int32)
    dst = np.array([b for _, b in pairs] + [free_dev[-1]], np.int32)
    kvq.copy_pages(c.g, dev(src), dev(dst))
    torch.cuda.synchronize()
    assert kvq.last_device_error() == 4  # KVQ_ERR_BAD_TABLE: the pair outside both tiers
    for n in names:
        want = before[n].copy()
        for a, b in pairs:
            want[b] = before[n][a]
        assert np.array_equal(c.g.pool(n).reshape(total, -1), want), n
    bt2 = c.bt.copy()
    for a, b in pairs:
        bt2[c.bt == a] = b
    assert np.array_equal(c.decode(bt=bt2) if scheme == "int8kc" else _decode_with(c, bt2), ref)


def _decode_with(c, bt):
    saved = c.bt
    c.bt = bt
    try:
        return c.decode()
    finally:
        c.bt = saved


# --------------------------------------------------- decode that appends its token
@pytest.mark.parametrize("scheme,Hq,D,P", [("int8", 32, 128, 16), ("int8", 8, 64, 32), ("fp8", 16, 128, 16),
                                           ("int4", 32, 128, 32), ("int4", 16, 64, 16), ("int8", 64, 128, 16),
                                           ("int4sym", 32, 128, 16)],
                         ids=lambda x: str(x))
@pytest.mark.parametrize("host", [False, True], ids=["device", "host-tier"])
def test_decode_that_appends_its_token_equals_append_then_decode(scheme, Hq, D, P, host):
    """kvq_decode_attn_append (one launch on the CUDA-core kernel, the
    append kernel then the decode on the tensor-core one) leaves the same
    pools and the same output, bit for bit, as kvq_append of each sequence's
    new token followed by kvq_decode_attn; also replayed from a CUDA graph,
    with part of the pages in the host tier, and with bf16 output."""
    w = small(scheme, Hq, 8, D, P)
    full = np.array([3001, 17, 1, 0, 800, 2500, 32, 33], np.int32)
    bt, num_pages = inp.page_table(full, P, w.seed, 3)
    hp = num_pages // 3 if host else 0
    a = Case(w, np.maximum(full - 1, 0), block_table=bt, num_pages=num_pages, host_pages=hp)
    b = Case(w, np.maximum(full - 1, 0), block_table=bt, num_pages=num_pages, host_pages=hp, oracle_seqs=[])
    H = w.kv_heads
    k_new = np.zeros((len(full), H, D), np.uint16)
    v_new = np.zeros((len(full), H, D), np.uint16)
    for i, L in enumerate(full):
        if L > 0:
            k, v = inp.kv_rows(w, 0, i, int(L) - 1, int(L))
            k_new[i], v_new[i] = k.reshape(H, D), v.reshape(H, D)
    live = np.nonzero(full > 0)[0]
    slots = np.concatenate([inp.slots(bt, int(i), np.array([full[i] - 1]), P) for i in live])
    assert a.o.append(slots, k_new[live].reshape(-1, H, D), v_new[live].reshape(-1, H, D)) == 0
    ref = a.o.decode_attn(a.q, bt, full, w.q_heads, 0.0)

    q, d_bt, d_len = dev_bits(a.q), dev(bt), dev(full)
    # a: the fused call
    out_a = torch.full((len(full), w.q_heads, D), float("nan"), dtype=torch.float32, device=DEV)
    ws_a = kvq.alloc_workspace(a.g, len(full), w.q_heads, bt.shape[1], device=DEV)
    kvq.decode_attn_append(a.g, dev_bits(k_new), dev_bits(v_new), q, d_bt, d_len, out_a, ws_a)
    assert kvq.last_device_error() == kvq.OK
    # b: append then decode
    out_b = torch.full_like(out_a, float("nan"))
    ws_b = kvq.alloc_workspace(b.g, len(full), w.q_heads, bt.shape[1], device=DEV)
    kvq.append(b.g, dev(slots), dev_bits(k_new[live]), dev_bits(v_new[live]))
    kvq.decode_attn(b.g, q, d_bt, d_len, out_b, ws_b)
    assert kvq.last_device_error() == kvq.OK
    got = out_a.cpu().numpy().astype(np.float64)
    assert np.array_equal(got, out_b.cpu().numpy().astype(np.float64))
    for name in kvq.POOLS:
        ga, gb = a.g.pool(name), b.g.pool(name)
        assert (ga is None and gb is None) or np.array_equal(ga, gb), name
    a.compare_cache(full=True)
    assert_attn_close(got, ref, f"{scheme} decode with append")
    assert np.all(got[3] == 0)  # the empty sequence

    # replayed from a CUDA graph (the token is re-quantized to the same bytes)
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    dk, dv = dev_bits(k_new), dev_bits(v_new)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        kvq.decode_attn_append(a.g, dk, dv, q, d_bt, d_len, out_a, ws_a, stream=stream)
    for _ in range(2):
        out_a.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert kvq.last_device_error() == kvq.OK
        assert np.array_equal(out_a.cpu().numpy().astype(np.float64), got)
    a.compare_cache(full=True)
    # bf16 output: the fp32 result rounded to nearest even
    out16 = torch.empty((len(full), w.q_heads, D), dtype=torch.bfloat16, device=DEV)
    kvq.decode_attn_append(a.g, dk, dv, q, d_bt, d_len, out16, ws_a)
    assert kvq.last_device_error() == kvq.OK
    assert torch.equal(out16, out_a.to(torch.bfloat16))
