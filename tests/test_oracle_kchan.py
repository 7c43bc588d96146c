"""Pins for the oracle's per-channel K scheme ("int8kc"): the page rule, the
append that keeps residual rows, the seal, and the decode over open and
sealed pages.  Each check rests on something other than the oracle's own
code: a torch restatement of the rule, hand-made blocks with exact ties, a
block on which the rule must coincide with the (separately pinned) INT8
token rule, invariants and error bounds, and a brute-force fp64 attention
written here from the definition.

The rule ("KV Cache Optimization: Strategies for Faster LLM Inference",
section "KV Cache Quantization: When and How to Compress": per-channel keeps
more than per-tensor; the absmax rule of "Dynamic KV Cache Quantization for
Fast LLM Inference", section "Understanding Dynamic Quantization
Techniques", taken down each channel of a page's K): s_j = max_t |x| / 127,
S = max_j s_j, r_j = fp16 round-up of s_j / S, e_j = r_j * S, code =
round-half-even(x / e_j) in [-127, 127], every token scale S.

CPU only (no GPU marker)."""
import math

import numpy as np
import pytest
import torch

import kvq_inputs as inp
import oracle


def bf16(values):
    return inp.to_bf16_bits(np.asarray(values, np.float32))


def torch_kchan(xb: np.ndarray):
    """The rule restated with torch CPU fp32 ops and numpy binary16."""
    x = torch.from_numpy(inp.bf16_bits_to_float(xb))          # [P][D] fp32
    s = x.abs().amax(dim=0) / 127.0                           # fp32 division
    S = s.max()
    P, D = x.shape
    if S == 0:
        return (np.zeros((P, D), np.int8), np.full(D, 0x3C00, np.uint16), np.ones(P, np.float32))
    ratio = (s / S).numpy()                                   # fp32 division
    h = ratio.astype(np.float16)                              # nearest
    below = h.astype(np.float32) < ratio
    h = np.where(below, np.nextafter(h, np.float16(np.inf)), h)  # round up
    e = torch.from_numpy(h.astype(np.float32)) * S            # fp32 product
    q = torch.round(x / e).clamp(-127, 127)
    q = torch.where(e == 0, torch.zeros_like(q), q)
    return q.to(torch.int8).numpy(), h.view(np.uint16), np.full(P, S.item(), np.float32)


def outlier_block(r, P=16, D=128, n_out=4, gain=40.0):
    x = r.standard_normal((P, D)).astype(np.float32)
    x[:, r.choice(D, n_out, replace=False)] *= gain
    return bf16(x)


# ------------------------------------------------------------- the page rule ----
def test_kchan_page_matches_torch_restatement():
    r = np.random.default_rng(71)
    for trial in range(240):
        P = [16, 32, 48][trial % 3]
        D = [64, 128][(trial // 2) % 2]
        mag = r.choice([1e-3, 1.0, 50.0])
        xb = outlier_block(r, P, D, n_out=int(r.integers(0, 6)), gain=float(r.choice([1.0, 8.0, 60.0])))
        xb = bf16(inp.bf16_bits_to_float(xb) * mag)
        if trial % 5 == 0:  # an all-zero channel
            xb[:, r.integers(D)] = 0
        c, ch, tok = oracle.quant_kchan_page(xb)
        rc, rch, rtok = torch_kchan(xb)
        assert np.array_equal(ch, rch), trial
        assert np.array_equal(tok, rtok), trial
        assert np.array_equal(c, rc), trial


def test_kchan_hand_block_with_exact_ties():
    """Every channel's largest magnitude is 127 * 2^-3, so every s_j is 2^-3,
    r_j = 1.0 and e_j = 2^-3; entries at (k + 1/2) 2^-3 are exact ties and
    go to the even neighbour."""
    P, D = 16, 64
    x = np.zeros((P, D), np.float32)
    x[0, :] = 127 / 8
    x[1, :] = -127 / 8
    x[2, :] = 2.5 / 8     # tie 2.5 -> 2
    x[3, :] = 3.5 / 8     # tie 3.5 -> 4
    x[4, :] = -0.5 / 8    # tie -0.5 -> -0
    x[5, :] = 1.0 / 8 + 1 / 64  # 1.125 -> 1
    x[6, ::2] = 126.5 / 8  # tie 126.5 -> 126
    c, ch, tok = oracle.quant_kchan_page(bf16(x))
    assert np.all(ch == 0x3C00)
    assert np.all(tok == np.float32(127 / 8 / 127))
    assert np.all(c[0] == 127) and np.all(c[1] == -127)
    assert np.all(c[2] == 2) and np.all(c[3] == 4) and np.all(c[4] == 0) and np.all(c[5] == 1)
    assert np.all(c[6, ::2] == 126) and np.all(c[6, 1::2] == 0)
    assert np.all(c[7:] == 0)


def test_kchan_reduces_to_the_int8_token_rule_when_rows_and_channels_share_absmax():
    """If every token row and every channel of a block has the same largest
    magnitude A, the channel rule's effective scale is A / 127 for every
    channel, which is the INT8 token rule's scale of every row: the codes
    must be those of the (separately pinned) token rule."""
    r = np.random.default_rng(72)
    for trial in range(40):
        P, D = 16, [64, 128][trial % 2]
        A = float(r.choice([0.5, 3.0, 96.0]))
        x = r.uniform(-0.99 * A, 0.99 * A, (P, D)).astype(np.float32)
        sign = np.where(r.random(D) < 0.5, -1.0, 1.0)
        x[np.arange(D) % P, np.arange(D)] = sign * A  # each channel and each row reaches A
        xb = bf16(x)
        assert np.all(np.abs(inp.bf16_bits_to_float(xb)).max(axis=0) == np.float32(A))
        c, ch, tok = oracle.quant_kchan_page(xb)
        assert np.all(ch == 0x3C00)
        for t in range(P):
            rc, rs = oracle.quant_int8_row(xb[t])
            assert np.array_equal(c[t], rc)
            assert tok[t] == rs


def test_kchan_invariants_and_error_bound():
    r = np.random.default_rng(73)
    for trial in range(100):
        P, D = [16, 48][trial % 2], 128
        xb = outlier_block(r, P, D, n_out=int(r.integers(0, 8)), gain=float(r.choice([4.0, 30.0])))
        x = inp.bf16_bits_to_float(xb).astype(np.float64)
        c, ch, tok = oracle.quant_kchan_page(xb)
        rj = ch.view(np.float16).astype(np.float64)
        S = float(tok[0])
        assert np.all(tok == tok[0]) and S == np.float32(np.abs(x).max()) / np.float32(127)
        assert np.all(np.abs(c.astype(np.int64)) <= 127)
        assert np.all((rj > 0) & (rj <= 1.0)) and rj.max() == 1.0
        # the rounding up of r_j keeps every channel's peak on the code 127
        normal = rj >= 2.0 ** -14
        assert np.all(np.abs(c.astype(np.int64)).max(axis=0)[normal] == 127)
        # round trip within half an effective scale e_j (the fp32 product),
        # plus the fp32 rounding of the quotient x / e_j (|x / e_j| <= 127)
        e = (rj.astype(np.float32) * np.float32(S)).astype(np.float64)
        err = np.abs(c.astype(np.float64) * e[None, :] - x)
        assert np.all(err <= e[None, :] * (0.5 + 128 * 2.0 ** -24))


def test_kchan_zero_block_and_zero_channel():
    z = np.zeros((16, 64), np.uint16)
    c, ch, tok = oracle.quant_kchan_page(z)
    assert np.all(c == 0) and np.all(ch == 0x3C00) and np.all(tok == 1.0)
    r = np.random.default_rng(74)
    xb = outlier_block(r, 16, 64, n_out=0)
    xb[:, 5] = 0x8000  # -0.0
    c, ch, tok = oracle.quant_kchan_page(xb)
    assert ch[5] == 0 and np.all(c[:, 5] == 0)


def test_kchan_keeps_more_than_the_token_rule_on_outlier_channels():
    """The pages' claim for per-channel scales: with a few outlier channels,
    the ordinary channels keep far more precision than under one scale per
    token."""
    r = np.random.default_rng(75)
    xb = outlier_block(r, 16, 128, n_out=4, gain=40.0)
    x = inp.bf16_bits_to_float(xb).astype(np.float64)
    c, ch, tok = oracle.quant_kchan_page(xb)
    kc = c * ch.view(np.float16).astype(np.float64)[None, :] * tok[:, None]
    tk = np.stack([oracle.quant_int8_row(xb[t])[0] * np.float64(oracle.quant_int8_row(xb[t])[1])
                   for t in range(16)])
    ordinary = np.abs(x).max(axis=0) < 10
    e_kc = np.abs(kc - x)[:, ordinary].mean()
    e_tk = np.abs(tk - x)[:, ordinary].mean()
    assert e_kc * 10 < e_tk


# ---------------------------------------------------------- append and seal ----
def _kc_cache(npg, P, H, D, slots=4):
    return oracle.OracleCache("int8kc", npg, P, H, D, resid_slots=slots)


def test_kchan_open_pages_store_the_int8_token_rule_and_decode_like_int8():
    """Before any seal, the scheme is the INT8 token scheme: identical codes
    and scales, channel factors 1.0, and a bit-identical decode."""
    lens = np.array([5, 33, 16], np.int32)
    H, D, P, Hq = 2, 64, 16, 4
    w = inp.Workload(0, "t", "int8", 1, len(lens), Hq, H, D, P, ("fixed", 0), seed=81,
                     outlier_pairs=3, outlier_gain=10.0)
    bt, npg = inp.page_table(lens, P, 81, spare=2)
    a = oracle.OracleCache("int8", npg, P, H, D)
    b = _kc_cache(npg, P, H, D)
    for s, L in enumerate(lens):
        k, v = inp.kv_rows(w, 0, s, 0, L)
        sl = inp.slots(bt, s, np.arange(L), P)
        assert a.append(sl, k, v) == 0
        assert b.append(sl, k, v, resid_slot=np.full(L, -1, np.int32)) == 0
    for name in ("k_codes", "v_codes", "k_scales", "v_scales"):
        assert np.array_equal(getattr(a, name), getattr(b, name)), name
    used = np.unique(bt[bt >= 0])
    assert np.all(b.k_chan.reshape(npg, H, D)[used] == 0x3C00)
    q = inp.queries(w, 0)
    assert np.array_equal(a.decode_attn(q, bt, lens, Hq), b.decode_attn(q, bt, lens, Hq))


def test_kchan_residual_rows_and_seal_place_the_page_rule():
    """The residual slot holds the appended bf16 K rows at their offsets; a
    seal writes, for every KV head, exactly the page rule of those rows; V is
    untouched; out-of-range ids are rejected and skipped."""
    H, D, P = 2, 128, 16
    r = np.random.default_rng(82)
    cache = _kc_cache(4, P, H, D, slots=3)
    k = np.stack([outlier_block(r, P, D) for _ in range(H)], axis=1)  # [P][H][D]
    v = bf16(r.standard_normal((P, H, D)))
    page, rs = 2, 1
    sl = np.arange(P, dtype=np.int64) + page * P
    order = r.permutation(P)  # tokens may arrive in any order, over several calls
    for part in np.array_split(order, 3):
        assert cache.append(sl[part], k[part], v[part], resid_slot=np.full(part.size, rs, np.int32)) == 0
    res = cache.k_resid.reshape(3, H, P, D)
    assert np.array_equal(res[rs], k.transpose(1, 0, 2))
    v_before = cache.v_codes.copy(), cache.v_scales.copy()
    assert cache.seal(np.array([page, 9], np.int32), np.array([rs, 0], np.int32)) == -1
    for h in range(H):
        c, ch, tok = oracle.quant_kchan_page(k[:, h])
        row0 = (page * H + h) * P
        assert np.array_equal(cache.k_codes.reshape(-1, D)[row0:row0 + P].view(np.int8), c)
        assert np.array_equal(cache.k_chan.reshape(-1, H, D)[page, h], ch)
        assert np.array_equal(cache.k_scales[row0:row0 + P], tok)
    assert np.array_equal(cache.v_codes, v_before[0]) and np.array_equal(cache.v_scales, v_before[1])
    # a bad residual slot in an append writes nothing for that token
    assert cache.append(np.array([0], np.int64), k[:1], v[:1], resid_slot=np.array([3], np.int32)) == -1
    assert np.all(cache.k_codes.reshape(-1, D)[0] == 0)


def test_kchan_reopened_page_resets_its_channel_factors():
    H, D, P = 1, 64, 16
    r = np.random.default_rng(83)
    cache = _kc_cache(2, P, H, D, slots=1)
    k = outlier_block(r, P, D).reshape(P, 1, D)
    sl = np.arange(P, dtype=np.int64)
    cache.append(sl, k, k, resid_slot=np.zeros(P, np.int32))
    cache.seal(np.array([0], np.int32), np.array([0], np.int32))
    assert np.any(cache.k_chan[:D] != 0x3C00)
    # the page is freed and reused: its first token reopens it
    k2 = bf16(r.standard_normal((1, 1, D)))
    cache.append(np.array([0], np.int64), k2, k2, resid_slot=np.zeros(1, np.int32))
    assert np.all(cache.k_chan[:D] == 0x3C00)
    c, s = oracle.quant_int8_row(k2[0, 0])
    assert np.array_equal(cache.k_codes[:D].view(np.int8), c) and cache.k_scales[0] == s


def dense_kc(cache, kv, rows):
    """This test's own dequantization of per-channel K pools (numpy float16
    for the channel factors)."""
    D, P, H = cache.head_dim, cache.page_size, cache.num_kv_heads
    codes = (cache.k_codes if kv == 0 else cache.v_codes).reshape(-1, D)[rows].view(np.int8).astype(np.float64)
    sc = (cache.k_scales if kv == 0 else cache.v_scales)[rows].astype(np.float64)[:, None]
    if kv == 1:
        return codes * sc
    ch = cache.k_chan.reshape(-1, D)[rows // P].view(np.float16).astype(np.float64)
    return codes * ch * sc


def test_kchan_decode_over_sealed_and_open_pages_matches_brute_force():
    lens = np.array([40, 16, 1, 0, 77], np.int32)
    H, D, P, Hq = 2, 64, 16, 8
    w = inp.Workload(0, "t", "int8", 1, len(lens), Hq, H, D, P, ("fixed", 0), seed=84,
                     outlier_pairs=3, outlier_gain=20.0)
    bt, npg = inp.page_table(lens, P, 84, spare=2)
    cache = _kc_cache(npg, P, H, D, slots=len(lens))
    sealed = 0
    for s, L in enumerate(lens):
        k, v = inp.kv_rows(w, 0, s, 0, L)
        for t in range(L):  # one token at a time, sealing each page as it fills
            assert cache.append(inp.slots(bt, s, np.array([t]), P), k[t:t + 1], v[t:t + 1],
                                resid_slot=np.array([s], np.int32)) == 0
            if t % P == P - 1:
                assert cache.seal(np.array([bt[s, t // P]], np.int32), np.array([s], np.int32)) == 0
                sealed += 1
    assert sealed == 40 // 16 + 1 + 77 // 16
    q = inp.queries(w, 0)
    got = cache.decode_attn(q, bt, lens, Hq)
    qf = inp.bf16_bits_to_float(q).astype(np.float64).reshape(len(lens), Hq, D)
    G = Hq // H
    for b, L in enumerate(lens):
        if L == 0:
            assert np.all(got[b] == 0)
            continue
        t = np.arange(L)
        for hq in range(Hq):
            rows = (bt[b, t // P].astype(np.int64) * H + hq // G) * P + t % P
            K, V = dense_kc(cache, 0, rows), dense_kc(cache, 1, rows)
            sc = K @ qf[b, hq] / math.sqrt(D)
            p = np.exp(sc - sc.max())
            np.testing.assert_allclose(got[b, hq], p @ V / p.sum(), rtol=1e-12, atol=1e-12)


def test_kchan_sealed_decode_is_closer_to_the_unquantized_attention():
    """With outlier channels in K, attention over sealed per-channel pages is
    closer to the attention over the bf16 keys than the INT8 token scheme."""
    lens = np.array([256], np.int32)
    H, D, P, Hq = 1, 128, 16, 4
    w = inp.Workload(0, "t", "int8", 1, 1, Hq, H, D, P, ("fixed", 0), seed=85,
                     outlier_pairs=4, outlier_gain=30.0)
    bt, npg = inp.page_table(lens, P, 85)
    k, v = inp.kv_rows(w, 0, 0, 0, 256)
    sl = inp.slots(bt, 0, np.arange(256), P)
    a = oracle.OracleCache("int8", npg, P, H, D)
    a.append(sl, k, v)
    b = _kc_cache(npg, P, H, D, slots=npg)
    pg = bt[0, np.arange(256) // P].astype(np.int32)
    b.append(sl, k, v, resid_slot=np.arange(256, dtype=np.int32) // P)
    b.seal(pg[::P], np.arange(256 // P, dtype=np.int32))
    q = inp.queries(w, 0)
    ka = inp.bf16_bits_to_float(k).astype(np.float64)[:, 0]
    va = np.stack([oracle.quant_int8_row(v[t, 0])[0] * np.float64(oracle.quant_int8_row(v[t, 0])[1])
                   for t in range(256)])
    qf = inp.bf16_bits_to_float(q).astype(np.float64).reshape(Hq, D)
    exact = []
    for hq in range(Hq):
        sc = ka @ qf[hq] / math.sqrt(D)
        p = np.exp(sc - sc.max())
        exact.append(p @ va / p.sum())
    exact = np.stack(exact)
    ea = np.abs(a.decode_attn(q, bt, lens, Hq)[0] - exact).max()
    eb = np.abs(b.decode_attn(q, bt, lens, Hq)[0] - exact).max()
    assert eb < ea
