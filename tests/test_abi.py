"""The C ABI on the host (no GPU needed): the library loads, exports every
entry point include/kvq.h declares, sizes pools by the pages' bytes-per-token
rule, checks arguments before touching the device, and its page allocator
reproduces the oracle's seeded free list."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import dynamically_quantized_paged_gb300 as kvq
import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "kvq.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_function_is_exported():
    names = declared_functions()
    assert len(names) >= 14
    assert sorted(kvq.EXPORTS) == names
    lib = ctypes.CDLL(kvq.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings():
    seen = set()
    for s in range(9):
        txt = kvq.status_string(s)
        assert txt and txt not in seen
        seen.add(txt)
    assert kvq.status_string(99) == "unknown status"


@pytest.mark.parametrize("scheme,bits", [("int8", 8), ("fp8", 8), ("int4", 4), ("int4sym", 4)])
def test_cache_bytes_match_printed_bytes_per_token(scheme, bits):
    # 80 layers, 8 KV heads, head_dim 128: K+V codes per token
    code, scale, zero = kvq.cache_bytes(scheme, 3, 16, 8, 128)
    per_token_layer_codes = 2 * code // (3 * 16)
    assert per_token_layer_codes * 80 == oracle.kv_bytes_per_token(80, 8, 128, bits)
    per_token_layer_meta = 2 * (scale + zero) // (3 * 16)
    assert per_token_layer_meta == oracle.scale_bytes_per_token(1, 8, 128, scheme)


def test_cache_bytes_rejects_bad_geometry():
    with pytest.raises(kvq.KvqError) as e:
        kvq.cache_bytes("int8", 0, 16, 8, 128)
    assert e.value.status == 1
    with pytest.raises(kvq.KvqError) as e:
        kvq.cache_bytes("int8", 4, 16, 8, 96)
    assert e.value.status == 7


def test_allocator_matches_oracle_free_list_and_semantics():
    for n, seed in ((1, 0), (10, 7), (1000, 123456789)):
        a = kvq.PageAllocator(n, seed)
        got = a.alloc(n)
        assert got == oracle.free_list(n, seed)[::-1].tolist()
        assert a.free_count == 0
        with pytest.raises(kvq.KvqError) as e:
            a.alloc(1)
        assert e.value.status == 3  # out of pages: the pages' out-of-memory case
        if n >= 3:
            a.free(got[:3])
            assert a.free_count == 3
            assert a.alloc(2) == [got[2], got[1]]  # last freed, first reused
        a.close()


def test_allocator_rejects_bad_frees():
    a = kvq.PageAllocator(8, 1)
    pages = a.alloc(4)
    for bad in ([99], [-1], [pages[0], pages[0]]):
        with pytest.raises(kvq.KvqError):
            a.free(bad)
    assert a.free_count == 4  # nothing was freed by the failed calls
    a.free(pages[:1])
    with pytest.raises(kvq.KvqError):
        a.free(pages[:1])  # double free
    a.close()


def test_allocator_shared_pages_reference_counts():
    """Shared prefix pages: allocation gives one reference, share adds, free
    drops, and a page goes back on the free list with its last reference."""
    a = kvq.PageAllocator(6, 3)
    p = a.alloc(3)
    assert [a.refcount(x) for x in p] == [1, 1, 1]
    a.share([p[0], p[1], p[0]])                      # p0 now held 3 times, p1 twice
    assert [a.refcount(x) for x in p] == [3, 2, 1]
    a.free([p[0], p[1]])
    assert [a.refcount(x) for x in p] == [2, 1, 1] and a.free_count == 3
    a.free([p[1], p[0], p[0], p[2]])                 # p1, p0, p2 lose their last references
    assert [a.refcount(x) for x in p] == [0, 0, 0] and a.free_count == 6
    assert a.alloc(3) == [p[2], p[0], p[1]]          # pushed in the order they were released
    a.close()


def test_allocator_share_and_free_reject_without_changing_anything():
    a = kvq.PageAllocator(5, 9)
    p = a.alloc(2)
    free_page = next(x for x in range(5) if x not in p)
    for bad in ([99], [-1], [free_page], [p[0], free_page]):
        with pytest.raises(kvq.KvqError) as e:
            a.share(bad)
        assert e.value.status == 1
    with pytest.raises(kvq.KvqError):
        a.free([p[0], p[0]])                          # two drops, one reference
    a.share([p[0]])
    with pytest.raises(kvq.KvqError):
        a.free([p[0], p[0], p[0], p[1]])              # three drops, two references
    assert [a.refcount(x) for x in p] == [2, 1] and a.free_count == 3
    with pytest.raises(kvq.KvqError):
        a.refcount(5)
    a.close()


def test_allocator_matches_a_plain_model_under_random_operations():
    """Random alloc / share / free sequences against a plain model of the
    header's rules: a stack of free ids (pop from the end, push released ids
    in call order) and a count per page; failed calls change nothing."""
    n, seed = 40, 77
    a = kvq.PageAllocator(n, seed)
    stack = oracle.free_list(n, seed).tolist()
    refs = [0] * n
    r = np.random.default_rng(5)
    for _ in range(3000):
        op = r.integers(3)
        held = [i for i in range(n) if refs[i] > 0]
        if op == 0:
            k = int(r.integers(0, 4))
            if k > len(stack):
                with pytest.raises(kvq.KvqError):
                    a.alloc(k)
                continue
            got = a.alloc(k)
            want = [stack.pop() for _ in range(k)]
            assert got == want
            for x in want:
                refs[x] = 1
        else:
            pool = held + [int(r.integers(n))] if held else [int(r.integers(n))]
            ids = [int(r.choice(pool)) for _ in range(int(r.integers(1, 4)))]
            counts = {x: ids.count(x) for x in ids}
            ok = all(refs[x] > 0 for x in ids) and (op == 1 or all(counts[x] <= refs[x] for x in ids))
            if not ok:
                with pytest.raises(kvq.KvqError):
                    (a.share if op == 1 else a.free)(ids)
            elif op == 1:
                a.share(ids)
                for x in ids:
                    refs[x] += 1
            else:
                a.free(ids)
                for x in ids:
                    refs[x] -= 1
                    if refs[x] == 0:
                        stack.append(x)
        assert a.free_count == len(stack)
        assert [a.refcount(i) for i in range(n)] == refs
    a.close()


def test_copy_page_argument_errors_before_any_device_access():
    c = fake_cache(num_pages=4)
    for src, dst in ((0, 0), (-1, 1), (0, 4), (4, 0)):
        assert kvq.lib.kvq_copy_page(ctypes.byref(c), src, dst, None) == 1
    assert kvq.lib.kvq_copy_page(None, 0, 1, None) == 1
    assert kvq.lib.kvq_copy_page(ctypes.byref(fake_cache(head_dim=96)), 0, 1, None) == 7


def fake_cache(scheme=1, head_dim=128, page_size=16, heads=8, align=256, group=32, num_pages=4, host_pages=0,
               resid_slots=0, k_chan=True, host_k_chan=True, k_resid=True):
    base = 1 << 20  # never dereferenced: argument checks run before any device access
    p = lambda i: base + i * (1 << 16) + (0 if align >= 16 else align)
    h = lambda i: p(6 + i) if host_pages > 0 else None
    kc = scheme == 5
    return kvq.CacheStruct(scheme, num_pages, page_size, heads, head_dim, group if scheme == 3 else 0,
                           p(0), p(1), p(2), p(3), p(4) if scheme == 3 else None,
                           p(5) if scheme == 3 else None,
                           host_pages, h(0), h(1), h(2), h(3), h(4) if scheme == 3 else None,
                           h(5) if scheme == 3 else None,
                           p(12) if kc and k_chan else None,
                           p(13) if kc and host_k_chan and host_pages > 0 else None,
                           p(14) if kc and k_resid and resid_slots > 0 else None, resid_slots)


def test_cache_struct_layout_matches_the_header():
    """The binding's mirror of kvq_cache: field order and offsets as in
    include/kvq.h (int32 fields, then the six pools, then the host tier)."""
    hdr = open(os.path.join(ROOT, "include", "kvq.h")).read()
    body = re.search(r"typedef struct kvq_cache \{(.*?)\} kvq_cache;", hdr, re.S).group(1)
    names = re.findall(r"^\s*(?:int32_t|void\*)\s+(\w+);", body, re.M)
    assert names == [f[0] for f in kvq.CacheStruct._fields_]
    off = {f[0]: getattr(kvq.CacheStruct, f[0]).offset for f in kvq.CacheStruct._fields_}
    assert off["k_codes"] == 24 and off["host_pages"] == 72 and off["host_k_codes"] == 80
    assert off["k_chan"] == 128 and off["k_resid"] == 144 and off["resid_slots"] == 152
    assert ctypes.sizeof(kvq.CacheStruct) == 160


def test_batched_page_copy_argument_errors_before_any_device_access():
    c = fake_cache(num_pages=4, host_pages=3)
    L = kvq.lib
    assert L.kvq_copy_pages(ctypes.byref(c), None, None, 0, None) == 0     # nothing to do
    assert L.kvq_copy_pages(ctypes.byref(c), None, None, -1, None) == 1
    assert L.kvq_copy_pages(ctypes.byref(c), None, 1 << 20, 2, None) == 1
    assert L.kvq_copy_pages(ctypes.byref(c), 1 << 20, (1 << 20) + 2, 2, None) == 1  # misaligned
    assert L.kvq_copy_pages(None, 1 << 20, 1 << 21, 2, None) == 1


def test_kchan_sizes_and_argument_errors_before_any_device_access():
    """The per-channel K scheme's pools, its append, seal and the refusal of
    the fused decode-append: every rule of the header checked on the host."""
    c, r = ctypes.c_size_t(), ctypes.c_size_t()
    assert kvq.lib.kvq_kchan_bytes(10, 16, 8, 128, 3, ctypes.byref(c), ctypes.byref(r)) == 0
    assert c.value == 10 * 8 * 128 * 2 and r.value == 3 * 8 * 16 * 128 * 2
    assert kvq.lib.kvq_kchan_bytes(10, 16, 8, 96, 3, None, None) == 7
    assert kvq.lib.kvq_kchan_bytes(10, 16, 8, 128, -1, None, None) == 1
    assert kvq.cache_bytes("int8kc", 10, 16, 8, 128) == kvq.cache_bytes("int8", 10, 16, 8, 128)
    ok = fake_cache(scheme=5, resid_slots=2)
    # the channel-factor pool is required; the residual pool when it has slots
    assert call_append(fake_cache(scheme=5, k_chan=False)) == 1
    assert call_append(fake_cache(scheme=5, resid_slots=2, k_resid=False)) == 1
    assert call_append(fake_cache(scheme=5, resid_slots=-1)) == 1
    assert call_append(fake_cache(scheme=5, host_pages=2, host_k_chan=False)) == 1
    assert call_append(ok, T=0) == 0  # valid: nothing to launch
    L = kvq.lib
    # append_kchan: scheme, alignment of the residual-slot array
    assert L.kvq_append_kchan(ctypes.byref(fake_cache(scheme=1)), None, 0, 1, None, None, None, None, 0, None) == 2
    assert L.kvq_append_kchan(ctypes.byref(ok), None, 0, 1, None, (1 << 20) + 2, None, None, 0, None) == 1
    assert L.kvq_append_kchan(ctypes.byref(fake_cache(scheme=5)), None, 0, 1, None, 1 << 20, None, None, 0,
                              None) == 1  # residual slots named, but the cache has none
    assert L.kvq_append_kchan(ctypes.byref(ok), None, 0, 1, None, 1 << 20, None, None, 0, None) == 0
    # seal: scheme, residual pool, n
    assert L.kvq_seal_pages(ctypes.byref(fake_cache(scheme=1)), None, None, 0, None) == 2
    assert L.kvq_seal_pages(ctypes.byref(fake_cache(scheme=5)), None, None, 0, None) == 1
    assert L.kvq_seal_pages(ctypes.byref(ok), None, None, -1, None) == 1
    assert L.kvq_seal_pages(ctypes.byref(ok), None, None, 0, None) == 0
    assert L.kvq_seal_pages(ctypes.byref(ok), None, None, 3, None) == 1  # null arrays
    # the fused decode-append needs residual slots: refused
    args = [None] * 6 + [0, 1, 4, 1, ctypes.c_float(0.0), None, ctypes.c_size_t(0), None]
    assert L.kvq_decode_attn_append(ctypes.byref(ok), *args) == 7


def test_host_tier_argument_errors_before_any_device_access():
    """A host tier needs its pools (16-byte aligned; zero-point pools for
    asymmetric INT4) and a non-negative size; page ids of both tiers are
    valid copy_page arguments, ids past both are not."""
    c = fake_cache(num_pages=4, host_pages=3)
    for src, dst in ((0, 7), (7, 0), (-1, 5), (6, 6)):
        assert kvq.lib.kvq_copy_page(ctypes.byref(c), src, dst, None) == 1
    assert call_append(fake_cache(host_pages=-1)) == 1
    c = fake_cache(host_pages=2)
    c.host_v_scales = None
    assert call_append(c) == 1
    c = fake_cache(host_pages=2)
    c.host_k_codes += 8
    assert call_append(c) == 1
    c = fake_cache(scheme=3, host_pages=2)
    c.host_v_zeros = None
    assert call_append(c) == 1
    # both tiers count toward the 2^31-slot limit of 32-bit slot indexing
    assert call_append(fake_cache(num_pages=1 << 26, host_pages=1 << 26)) == 1


def call_append(c, scheme=None, T=1, k=1 << 24, v=1 << 25, slots=1 << 26):
    return kvq.lib.kvq_append(ctypes.byref(c), None, 0, 1, slots, k, v, T,
                              c.scheme if scheme is None else scheme, None)


def test_append_argument_errors_before_any_launch():
    assert kvq.lib.kvq_append(None, None, 0, 1, None, None, None, 0, 1, None) == 1
    assert call_append(fake_cache(), scheme=2) == 2            # scheme mismatch
    assert call_append(fake_cache(head_dim=96)) == 7           # unsupported head_dim
    assert call_append(fake_cache(page_size=8)) == 7           # page not a multiple of 16
    assert call_append(fake_cache(align=8)) == 1               # misaligned pool
    assert call_append(fake_cache(scheme=3, group=64)) == 7    # INT4 group must be 32
    assert call_append(fake_cache(), T=-1) == 1
    assert call_append(fake_cache(), k=(1 << 24) + 2) == 1     # misaligned k
    assert call_append(fake_cache(), T=0) == 0                 # nothing to do
    c = fake_cache(scheme=3)
    c.k_zeros = None
    assert call_append(c) == 1                                 # INT4 needs zero pools
    assert call_append(fake_cache(num_pages=1 << 27)) == 1     # 2^31 slots: beyond 32-bit indexing
    assert call_append(fake_cache(), T=1 << 27) == 1           # 2^31 rows (2^27 tokens x 8 heads x K,V)


def call_decode(c, B=2, Hq=32, maxp=4, ws_bytes=1 << 30, q=1 << 24):
    return kvq.lib.kvq_decode_attn(ctypes.byref(c), q, 1 << 25, 1 << 26, 1 << 27, B, Hq, maxp, 0.0,
                                   1 << 28, ws_bytes, None)


def test_decode_argument_errors_before_any_launch():
    c = fake_cache()
    assert call_decode(c, Hq=30) == 1          # not a multiple of the KV heads
    assert call_decode(c, Hq=24) == 7          # GQA ratio 3
    assert call_decode(c, Hq=128) == 7         # GQA ratio 16
    assert call_decode(c, B=5000) == 1         # more sequences than one call plans for
    assert call_decode(c, maxp=0) == 1
    assert call_decode(c, B=0) == 0            # empty batch: nothing to do
    assert call_decode(c, q=(1 << 24) + 4) == 1


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_device_calls_report_cuda_error_without_a_gpu():
    c = fake_cache()
    n = ctypes.c_size_t()
    assert kvq.lib.kvq_decode_workspace_bytes(ctypes.byref(c), 2, 32, 4, ctypes.byref(n)) == 5
    assert call_decode(c) == 5
    assert call_append(fake_cache()) == 5
    assert kvq.lib.kvq_last_device_error(None) == 5
    assert kvq.lib.kvq_copy_page(ctypes.byref(c), 0, 1, None) == 5


def test_no_oracle_in_product_path():
    """The product package never imports or links the oracle."""
    pkg = os.path.dirname(kvq.__file__)
    for root, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(root, f)).read()
                assert "import oracle" not in text and "liboracle" not in text and "kvq_oracle" not in text, f


def test_decode_attn_out_rejects_an_unknown_output_dtype():
    """The output dtype is checked before anything else: no device needed."""
    import ctypes
    st = kvq.lib.kvq_decode_attn_out(None, None, None, None, None, 7, 1, 8, 1, ctypes.c_float(0.0), None, 0, None)
    assert st == 1  # KVQ_ERR_INVALID_ARG



def test_decode_attn_append_argument_errors_before_any_launch():
    c = fake_cache()
    call = lambda c, dt=0, Hq=32: kvq.lib.kvq_decode_attn_append(  # noqa: E731
        ctypes.byref(c), 1 << 23, 1 << 22, 1 << 24, 1 << 25, 1 << 26, 1 << 27, dt, 2, Hq, 4, 0.0,
        1 << 28, 1 << 30, None)
    assert call(c, dt=7) == 1                  # unknown output dtype
    assert call(c, Hq=24) == 7                 # GQA ratio 3
    assert call(fake_cache(head_dim=96)) == 7  # unsupported head_dim
    assert kvq.lib.kvq_decode_attn_append(None, None, None, None, None, None, None, 0, 2, 32, 4, 0.0,
                                          None, 0, None) == 1
