"""Dynamic KV-cache quantization with fused-dequantization paged decode
attention for NVIDIA GB300 (sm_103a).

Thin Python binding over the C ABI in ``include/kvq.h`` (``libkvq.so``, built
in-tree by ``build.py``).  This module only marshals arguments: torch tensors
are passed as raw device pointers with the current CUDA stream; every step of
the computation runs in the library's CUDA kernels.  There is no CPU
fallback: if the library is missing, importing this package raises.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvq.so")

INT8, FP8, INT4, INT4SYM, INT8KC = 1, 2, 3, 4, 5
SCHEMES = {"int8": INT8, "fp8": FP8, "int4": INT4, "int4sym": INT4SYM, "int8kc": INT8KC}

OK = 0
OUT_F32, OUT_BF16 = 0, 1  # kvq_out_dtype
STATUS_NAMES = {0: "KVQ_OK", 1: "KVQ_ERR_INVALID_ARG", 2: "KVQ_ERR_SCHEME_MISMATCH",
                3: "KVQ_ERR_OUT_OF_PAGES", 4: "KVQ_ERR_BAD_TABLE", 5: "KVQ_ERR_CUDA",
                6: "KVQ_ERR_DEVICE_TIMEOUT", 7: "KVQ_ERR_UNSUPPORTED", 8: "KVQ_ERR_WORKSPACE"}

# Every function the header declares (checked against include/kvq.h by the tests).
EXPORTS = ["kvq_status_string", "kvq_cache_bytes", "kvq_append", "kvq_decode_workspace_bytes",
           "kvq_decode_attn", "kvq_decode_partial", "kvq_decode_merge", "kvq_validate_tables",
           "kvq_last_device_error", "kvq_allocator_create", "kvq_allocator_destroy",
           "kvq_alloc_pages", "kvq_free_pages", "kvq_allocator_free_count", "kvq_decode_attn_noalloc",
           "kvq_share_pages", "kvq_page_refcount", "kvq_copy_page", "kvq_decode_attn_out",
           "kvq_decode_attn_append", "kvq_kchan_bytes", "kvq_append_kchan", "kvq_seal_pages", "kvq_copy_pages"]


class KvqError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)} ({status_string(status)})")


class CacheStruct(ctypes.Structure):
    _fields_ = [("scheme", ctypes.c_int32), ("num_pages", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("group", ctypes.c_int32),
                ("k_codes", ctypes.c_void_p), ("v_codes", ctypes.c_void_p),
                ("k_scales", ctypes.c_void_p), ("v_scales", ctypes.c_void_p),
                ("k_zeros", ctypes.c_void_p), ("v_zeros", ctypes.c_void_p),
                ("host_pages", ctypes.c_int32),
                ("host_k_codes", ctypes.c_void_p), ("host_v_codes", ctypes.c_void_p),
                ("host_k_scales", ctypes.c_void_p), ("host_v_scales", ctypes.c_void_p),
                ("host_k_zeros", ctypes.c_void_p), ("host_v_zeros", ctypes.c_void_p),
                ("k_chan", ctypes.c_void_p), ("host_k_chan", ctypes.c_void_p),
                ("k_resid", ctypes.c_void_p), ("resid_slots", ctypes.c_int32)]


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built: run `python dynamically_quantized_paged_gb300/build.py` "
                          "(or __graft_entry__.build()); there is no fallback path")
    L = ctypes.CDLL(LIB_PATH)
    P, i32, i64p = ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p
    cachep = ctypes.POINTER(CacheStruct)
    sz = ctypes.POINTER(ctypes.c_size_t)
    L.kvq_status_string.argtypes, L.kvq_status_string.restype = [ctypes.c_int], ctypes.c_char_p
    L.kvq_cache_bytes.argtypes = [i32, i32, i32, i32, i32, sz, sz, sz]
    L.kvq_append.argtypes = [cachep, P, i32, i32, i64p, P, P, i32, i32, P]
    L.kvq_decode_workspace_bytes.argtypes = [cachep, i32, i32, i32, sz]
    dec = [cachep, P, P, P, P, i32, i32, i32, ctypes.c_float, P, ctypes.c_size_t, P]
    L.kvq_decode_attn.argtypes = dec
    L.kvq_decode_attn_out.argtypes = [cachep, P, P, P, P, i32, i32, i32, i32, ctypes.c_float, P, ctypes.c_size_t, P]
    L.kvq_decode_attn_append.argtypes = [cachep, P, P, P, P, P, P, i32, i32, i32, i32, ctypes.c_float, P,
                                         ctypes.c_size_t, P]
    L.kvq_decode_partial.argtypes = dec
    L.kvq_decode_merge.argtypes = dec
    L.kvq_validate_tables.argtypes = [cachep, P, P, i32, i32, P]
    L.kvq_decode_attn_noalloc.argtypes = [cachep, P, P, P, P, i32, i32, i32, ctypes.c_float, P]
    L.kvq_last_device_error.argtypes = [P]
    L.kvq_allocator_create.argtypes, L.kvq_allocator_create.restype = [i32, ctypes.c_uint64], P
    L.kvq_allocator_destroy.argtypes, L.kvq_allocator_destroy.restype = [P], None
    L.kvq_alloc_pages.argtypes = [P, i32, P]
    L.kvq_free_pages.argtypes = [P, i32, P]
    L.kvq_allocator_free_count.argtypes, L.kvq_allocator_free_count.restype = [P], i32
    L.kvq_share_pages.argtypes = [P, i32, P]
    L.kvq_page_refcount.argtypes = [P, i32, ctypes.POINTER(ctypes.c_int32)]
    L.kvq_copy_page.argtypes = [cachep, i32, i32, P]
    L.kvq_kchan_bytes.argtypes = [i32, i32, i32, i32, i32, sz, sz]
    L.kvq_append_kchan.argtypes = [cachep, P, i32, i32, i64p, P, P, P, i32, P]
    L.kvq_seal_pages.argtypes = [cachep, P, P, i32, P]
    L.kvq_copy_pages.argtypes = [cachep, P, P, i32, P]
    for name in EXPORTS:
        getattr(L, name)  # every declared entry point must be exported
    return L


lib = _load()


def status_string(status: int) -> str:
    return lib.kvq_status_string(status).decode()


def _check(status: int, what: str) -> None:
    if status != OK:
        raise KvqError(status, what)


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    if stream is None:
        if not torch.cuda.is_available():
            return None
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream) if hasattr(stream, "cuda_stream") else stream


def cache_bytes(scheme: str | int, num_pages: int, page_size: int, num_kv_heads: int,
                head_dim: int) -> tuple[int, int, int]:
    """(code_bytes, scale_bytes, zero_bytes) of one K (or V) pool."""
    sid = SCHEMES.get(scheme, scheme)
    c, s, z = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib.kvq_cache_bytes(sid, num_pages, page_size, num_kv_heads, head_dim,
                               ctypes.byref(c), ctypes.byref(s), ctypes.byref(z)), "kvq_cache_bytes")
    return c.value, s.value, z.value


def kchan_bytes(num_pages: int, page_size: int, num_kv_heads: int, head_dim: int,
                resid_slots: int) -> tuple[int, int]:
    """(chan_bytes, resid_bytes) of the per-channel K scheme's extra pools."""
    c, r = ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib.kvq_kchan_bytes(num_pages, page_size, num_kv_heads, head_dim, resid_slots,
                               ctypes.byref(c), ctypes.byref(r)), "kvq_kchan_bytes")
    return c.value, r.value


POOLS = ("k_codes", "v_codes", "k_scales", "v_scales", "k_zeros", "v_zeros", "k_chan")


class PagedKVCache:
    """One layer's paged quantized cache: six caller-owned device pools (torch
    uint8 tensors) laid out as include/kvq.h describes, and optionally a host
    tier of host_pages more pages (page ids num_pages .. num_pages +
    host_pages - 1) in page-locked host memory that the kernels read and
    write in place.  The per-channel K scheme ("int8kc") adds the channel
    factors k_chan (both tiers) and a device residual pool k_resid of
    resid_slots slots."""

    def __init__(self, scheme: str, num_pages: int, page_size: int, num_kv_heads: int,
                 head_dim: int, device="cuda", zero_init: bool = True, host_pages: int = 0,
                 resid_slots: int = 0):
        self.scheme = scheme
        self.sid = SCHEMES[scheme]
        self.num_pages, self.page_size = num_pages, page_size
        self.num_kv_heads, self.head_dim = num_kv_heads, head_dim
        self.host_pages = host_pages
        self.group = 32 if scheme in ("int4", "int4sym") else 0
        cb, sb, zb = cache_bytes(scheme, num_pages, page_size, num_kv_heads, head_dim)
        alloc = torch.zeros if zero_init else torch.empty
        self.k_codes = alloc(cb, dtype=torch.uint8, device=device)
        self.v_codes = alloc(cb, dtype=torch.uint8, device=device)
        self.k_scales = alloc(sb, dtype=torch.uint8, device=device)
        self.v_scales = alloc(sb, dtype=torch.uint8, device=device)
        self.k_zeros = alloc(zb, dtype=torch.uint8, device=device) if zb else None
        self.v_zeros = alloc(zb, dtype=torch.uint8, device=device) if zb else None
        kc = scheme == "int8kc"
        self.resid_slots = resid_slots if kc else 0
        chb, rsb = kchan_bytes(num_pages, page_size, num_kv_heads, head_dim, self.resid_slots) if kc else (0, 0)
        self.k_chan = alloc(chb, dtype=torch.uint8, device=device) if kc else None
        self.k_resid = alloc(rsb, dtype=torch.uint8, device=device) if rsb else None
        self.host = {}
        if host_pages > 0:
            hcb, hsb, hzb = cache_bytes(scheme, host_pages, page_size, num_kv_heads, head_dim)
            hchb = kchan_bytes(host_pages, page_size, num_kv_heads, head_dim, 0)[0] if kc else 0
            for name, nb in (("k_codes", hcb), ("v_codes", hcb), ("k_scales", hsb), ("v_scales", hsb),
                             ("k_zeros", hzb), ("v_zeros", hzb), ("k_chan", hchb)):
                self.host[name] = torch.zeros(nb, dtype=torch.uint8).pin_memory() if nb else None
        hp = lambda n: self.host[n].data_ptr() if self.host.get(n) is not None else None  # noqa: E731
        dp = lambda t: t.data_ptr() if t is not None else None  # noqa: E731
        self.struct = CacheStruct(self.sid, num_pages, page_size, num_kv_heads, head_dim, self.group,
                                  self.k_codes.data_ptr(), self.v_codes.data_ptr(),
                                  self.k_scales.data_ptr(), self.v_scales.data_ptr(),
                                  self.k_zeros.data_ptr() if zb else None,
                                  self.v_zeros.data_ptr() if zb else None,
                                  host_pages, hp("k_codes"), hp("v_codes"), hp("k_scales"),
                                  hp("v_scales"), hp("k_zeros"), hp("v_zeros"),
                                  dp(self.k_chan), hp("k_chan"), dp(self.k_resid), self.resid_slots)

    def tier_of(self, page: int) -> str:
        """"device" or "host": where page id `page` lives."""
        return "device" if page < self.num_pages else "host"

    def pool(self, name: str):
        """Host copy of one pool over both tiers (uint8, page ids in order:
        the device tier, then the host tier)."""
        d = getattr(self, name)
        if d is None:
            return None
        d = d.cpu().numpy()
        h = self.host.get(name)
        return d if h is None else np.concatenate([d, h.numpy()])

    def codes_rowmajor(self, which: str):
        """Host copy of the K or V codes (which = "k" or "v") over both tiers as
        uint8 [num_pages + host_pages][num_kv_heads][page_size][code bytes per token]."""
        t = self.pool(which + "_codes")
        cb = self.head_dim // 2 if self.scheme in ("int4", "int4sym") else self.head_dim
        return t.reshape(self.num_pages + self.host_pages, self.num_kv_heads, self.page_size, cb)

    @property
    def nbytes(self) -> int:
        return sum(t.numel() for t in (self.k_codes, self.v_codes, self.k_scales, self.v_scales,
                                       self.k_zeros, self.v_zeros, self.k_chan) if t is not None)


def copy_page(cache: PagedKVCache, src: int, dst: int, stream=None) -> None:
    """kvq_copy_page: copy page src into page dst (every pool), within a tier
    (copy-on-write) or between the device and host tiers (offload, fetch)."""
    _check(lib.kvq_copy_page(ctypes.byref(cache.struct), src, dst, _stream(stream)), "kvq_copy_page")


def copy_pages(cache: PagedKVCache, src: torch.Tensor, dst: torch.Tensor, stream=None) -> None:
    """kvq_copy_pages: copy every pool of page src[i] into page dst[i] (int32
    [n] device arrays; either tier), one launch for the whole batch."""
    n = src.numel()
    if dst.numel() != n or src.element_size() != 4 or dst.element_size() != 4:
        raise ValueError("kvq_copy_pages: src and dst must be int32 [n]")
    _check(lib.kvq_copy_pages(ctypes.byref(cache.struct), _ptr(src), _ptr(dst), n, _stream(stream)),
           "kvq_copy_pages")


def append(cache: PagedKVCache, slot_mapping: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
           block_table: torch.Tensor | None = None, stream=None) -> None:
    """kvq_append: quantize bf16 k, v [T, Hkv, d] into the slots slot_mapping
    (int64 [T]) of the cache."""
    T = slot_mapping.numel()
    if slot_mapping.element_size() != 8 or k.shape != v.shape or k.numel() != T * cache.num_kv_heads * cache.head_dim \
            or k.element_size() != 2:
        raise ValueError("kvq_append: slot_mapping must be int64 [T]; k, v bf16 [T, Hkv, d]")
    B, maxp = (block_table.shape[0], block_table.shape[1]) if block_table is not None else (0, 1)
    _check(lib.kvq_append(ctypes.byref(cache.struct), _ptr(block_table), B, maxp, _ptr(slot_mapping),
                          _ptr(k), _ptr(v), T, cache.sid, _stream(stream)), "kvq_append")


def append_kchan(cache: PagedKVCache, slot_mapping: torch.Tensor, resid_slot: torch.Tensor | None,
                 k: torch.Tensor, v: torch.Tensor, block_table: torch.Tensor | None = None, stream=None) -> None:
    """kvq_append_kchan: kvq_append for the per-channel K scheme, keeping each
    token's bf16 K rows in residual slot resid_slot[t] (int32 [T]; -1 or
    None: none)."""
    T = slot_mapping.numel()
    if slot_mapping.element_size() != 8 or k.shape != v.shape or k.numel() != T * cache.num_kv_heads * cache.head_dim \
            or k.element_size() != 2 or (resid_slot is not None and (resid_slot.numel() != T
                                                                     or resid_slot.element_size() != 4)):
        raise ValueError("kvq_append_kchan: slot_mapping int64 [T]; resid_slot int32 [T]; k, v bf16 [T, Hkv, d]")
    B, maxp = (block_table.shape[0], block_table.shape[1]) if block_table is not None else (0, 1)
    _check(lib.kvq_append_kchan(ctypes.byref(cache.struct), _ptr(block_table), B, maxp, _ptr(slot_mapping),
                                _ptr(resid_slot), _ptr(k), _ptr(v), T, _stream(stream)), "kvq_append_kchan")


def seal_pages(cache: PagedKVCache, pages: torch.Tensor, resid_slots: torch.Tensor, stream=None) -> None:
    """kvq_seal_pages: re-quantize K of pages[i] per channel from residual
    slot resid_slots[i] (both int32 [n], device)."""
    n = pages.numel()
    if resid_slots.numel() != n or pages.element_size() != 4 or resid_slots.element_size() != 4:
        raise ValueError("kvq_seal_pages: pages and resid_slots must be int32 [n]")
    _check(lib.kvq_seal_pages(ctypes.byref(cache.struct), _ptr(pages), _ptr(resid_slots), n, _stream(stream)),
           "kvq_seal_pages")


def decode_workspace_bytes(cache: PagedKVCache, num_seqs: int, num_q_heads: int,
                           max_pages_per_seq: int) -> int:
    n = ctypes.c_size_t()
    _check(lib.kvq_decode_workspace_bytes(ctypes.byref(cache.struct), num_seqs, num_q_heads,
                                          max_pages_per_seq, ctypes.byref(n)),
           "kvq_decode_workspace_bytes")
    return n.value


def alloc_workspace(cache: PagedKVCache, num_seqs: int, num_q_heads: int, max_pages_per_seq: int,
                    device="cuda") -> torch.Tensor:
    n = decode_workspace_bytes(cache, num_seqs, num_q_heads, max_pages_per_seq)
    return torch.empty(n, dtype=torch.uint8, device=device)


def _decode_call(fn, name, cache, q, block_table, seq_lens, out, workspace, softmax_scale, stream, bf16_ok=False):
    B = seq_lens.numel()
    if q.dim() != 3 or q.shape[0] != B or q.shape[2] != cache.head_dim or tuple(out.shape) != tuple(q.shape) \
            or block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError(f"{name}: shapes q{tuple(q.shape)} out{tuple(out.shape)} "
                         f"block_table{tuple(block_table.shape)} seq_lens[{B}] do not agree")
    out_ok = out.dtype == torch.float32 or (bf16_ok and out.dtype == torch.bfloat16)
    if q.element_size() != 2 or not out_ok or seq_lens.element_size() != 4 or block_table.element_size() != 4:
        raise ValueError(f"{name}: q must be bf16 bits, out fp32{' or bf16' if bf16_ok else ''}, tables int32")
    Hq = q.shape[1]
    if bf16_ok:  # kvq_decode_attn_out: the output dtype rides along
        dt = OUT_BF16 if out.dtype == torch.bfloat16 else OUT_F32
        _check(fn(ctypes.byref(cache.struct), _ptr(q), _ptr(block_table), _ptr(seq_lens), _ptr(out), dt, B, Hq,
                  block_table.shape[1], float(softmax_scale), _ptr(workspace), workspace.numel(),
                  _stream(stream)), name)
        return
    _check(fn(ctypes.byref(cache.struct), _ptr(q), _ptr(block_table), _ptr(seq_lens), _ptr(out), B, Hq,
              block_table.shape[1], float(softmax_scale), _ptr(workspace), workspace.numel(),
              _stream(stream)), name)


def decode_attn(cache: PagedKVCache, q: torch.Tensor, block_table: torch.Tensor,
                seq_lens: torch.Tensor, out: torch.Tensor, workspace: torch.Tensor,
                softmax_scale: float = 0.0, stream=None) -> torch.Tensor:
    """kvq_decode_attn: out[B, Hq, d] = paged GQA decode attention of
    q[B, Hq, d] (bf16) over the quantized cache; out fp32, or bf16 (through
    kvq_decode_attn_out: the fp32 result rounded to nearest even)."""
    if out.dtype == torch.bfloat16:
        _decode_call(lib.kvq_decode_attn_out, "kvq_decode_attn_out", cache, q, block_table, seq_lens, out,
                     workspace, softmax_scale, stream, bf16_ok=True)
    else:
        _decode_call(lib.kvq_decode_attn, "kvq_decode_attn", cache, q, block_table, seq_lens, out,
                     workspace, softmax_scale, stream)
    return out


def decode_attn_append(cache: PagedKVCache, k_new: torch.Tensor, v_new: torch.Tensor, q: torch.Tensor,
                       block_table: torch.Tensor, seq_lens: torch.Tensor, out: torch.Tensor,
                       workspace: torch.Tensor, softmax_scale: float = 0.0, stream=None) -> torch.Tensor:
    """kvq_decode_attn_append: one decode step that appends its own token --
    k_new, v_new bf16 [B, Hkv, d] are each sequence's new key and value,
    stored at position seq_lens[b] - 1 (seq_lens include them) -- then the
    attention of q over the whole cache into out (fp32 or bf16).  The same
    pools and output as append followed by decode_attn."""
    B = seq_lens.numel()
    if k_new.shape != v_new.shape or k_new.numel() != B * cache.num_kv_heads * cache.head_dim \
            or k_new.element_size() != 2:
        raise ValueError("kvq_decode_attn_append: k_new, v_new must be bf16 [B, Hkv, d]")
    if q.dim() != 3 or q.shape[0] != B or tuple(out.shape) != tuple(q.shape) or block_table.shape[0] != B:
        raise ValueError("kvq_decode_attn_append: shapes of q, out, block_table, seq_lens do not agree")
    if out.dtype not in (torch.float32, torch.bfloat16) or q.element_size() != 2 \
            or seq_lens.element_size() != 4 or block_table.element_size() != 4:
        raise ValueError("kvq_decode_attn_append: q bf16, out fp32 or bf16, tables int32")
    dt = OUT_BF16 if out.dtype == torch.bfloat16 else OUT_F32
    _check(lib.kvq_decode_attn_append(ctypes.byref(cache.struct), _ptr(k_new), _ptr(v_new), _ptr(q),
                                      _ptr(block_table), _ptr(seq_lens), _ptr(out), dt, B, q.shape[1],
                                      block_table.shape[1], float(softmax_scale), _ptr(workspace),
                                      workspace.numel(), _stream(stream)), "kvq_decode_attn_append")
    return out


def decode_attn_noalloc(cache: PagedKVCache, q: torch.Tensor, block_table: torch.Tensor,
                        seq_lens: torch.Tensor, out: torch.Tensor, softmax_scale: float = 0.0,
                        stream=None) -> torch.Tensor:
    """kvq_decode_attn_noalloc: decode_attn without a workspace, for callers
    that cannot allocate device memory; it uses the library's own fixed
    scratch array (KVQ_STATIC_SCRATCH_BYTES per GPU), so calls that overlap
    on the GPU race on it."""
    B = seq_lens.numel()
    if q.dim() != 3 or q.shape[0] != B or tuple(out.shape) != tuple(q.shape) or block_table.shape[0] != B:
        raise ValueError("kvq_decode_attn_noalloc: shapes of q, out, block_table, seq_lens do not agree")
    _check(lib.kvq_decode_attn_noalloc(ctypes.byref(cache.struct), _ptr(q), _ptr(block_table), _ptr(seq_lens),
                                       _ptr(out), B, q.shape[1], block_table.shape[1], float(softmax_scale),
                                       _stream(stream)), "kvq_decode_attn_noalloc")
    return out


def decode_partial(cache, q, block_table, seq_lens, out, workspace, softmax_scale=0.0, stream=None):
    _decode_call(lib.kvq_decode_partial, "kvq_decode_partial", cache, q, block_table, seq_lens, out,
                 workspace, softmax_scale, stream)


def decode_merge(cache, q, block_table, seq_lens, out, workspace, softmax_scale=0.0, stream=None):
    _decode_call(lib.kvq_decode_merge, "kvq_decode_merge", cache, q, block_table, seq_lens, out,
                 workspace, softmax_scale, stream)


def validate_tables(cache: PagedKVCache, block_table: torch.Tensor, seq_lens: torch.Tensor,
                    stream=None) -> None:
    _check(lib.kvq_validate_tables(ctypes.byref(cache.struct), _ptr(block_table), _ptr(seq_lens),
                                   block_table.shape[0], block_table.shape[1], _stream(stream)),
           "kvq_validate_tables")


def last_device_error(stream=None) -> int:
    """Synchronizes the stream; returns (and clears) the device error status."""
    return lib.kvq_last_device_error(_stream(stream))


class PageAllocator:
    """Host page allocator (kvq_allocator_*): scattered page ids handed out on
    demand from a seeded shuffled free list."""

    def __init__(self, num_pages: int, seed: int = 0):
        self._h = lib.kvq_allocator_create(num_pages, seed)
        if not self._h:
            raise KvqError(1, "kvq_allocator_create")
        self.num_pages = num_pages

    def alloc(self, n: int) -> list[int]:
        out = (ctypes.c_int32 * max(n, 1))()
        _check(lib.kvq_alloc_pages(self._h, n, out), "kvq_alloc_pages")
        return list(out[:n])

    def free(self, pages) -> None:
        """Drops one reference per listed id (kvq_free_pages)."""
        arr = (ctypes.c_int32 * max(len(pages), 1))(*pages)
        _check(lib.kvq_free_pages(self._h, len(pages), arr), "kvq_free_pages")

    def share(self, pages) -> None:
        """Adds one reference per listed id (kvq_share_pages)."""
        arr = (ctypes.c_int32 * max(len(pages), 1))(*pages)
        _check(lib.kvq_share_pages(self._h, len(pages), arr), "kvq_share_pages")

    def refcount(self, page: int) -> int:
        out = ctypes.c_int32(0)
        _check(lib.kvq_page_refcount(self._h, page, ctypes.byref(out)), "kvq_page_refcount")
        return out.value

    @property
    def free_count(self) -> int:
        return lib.kvq_allocator_free_count(self._h)

    def close(self) -> None:
        if self._h:
            lib.kvq_allocator_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
