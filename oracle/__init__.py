"""CPU oracle for dynamic KV-cache quantization and paged decode attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference legs may import this package.  The
product library (``dynamically_quantized_paged_gb300``) never imports it, and
this package imports nothing from the product.

The arithmetic lives in ``kvq_oracle.c`` (plain C, fp32 steps exactly as
written, fp64 attention); this module only compiles it with gcc and passes
numpy arrays through ctypes.  Every function cites the page passage it
follows in the C source.

Pins (checked by the CPU tests, independent of the oracle's own code):
worked hand examples of the INT8 rule, torch's rounding and float8 casts,
exhaustive binary16 neighbour checks, round-trip error bounds, closed-form
attention cases, brute-force dense attention and page-permutation
invariance, and the pages' printed bytes-per-token figures.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvq_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

INT8, FP8, INT4, INT4SYM, INT8KC = 1, 2, 3, 4, 5
SCHEME_IDS = {"int8": INT8, "fp8": FP8, "int4": INT4, "int4sym": INT4SYM, "int8kc": INT8KC}


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FP contraction)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fno-fast-math", "-ffp-contract=off", "-fopenmp",
           "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Cache(ctypes.Structure):
    _fields_ = [("scheme", ctypes.c_int32), ("num_pages", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("group", ctypes.c_int32),
                ("k_codes", ctypes.c_void_p), ("v_codes", ctypes.c_void_p),
                ("k_scales", ctypes.c_void_p), ("v_scales", ctypes.c_void_p),
                ("k_zeros", ctypes.c_void_p), ("v_zeros", ctypes.c_void_p),
                ("k_chan", ctypes.c_void_p), ("k_resid", ctypes.c_void_p),
                ("resid_slots", ctypes.c_int32)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            P, c_i32, c_u16 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint16
            L.orc_bf16_to_float.argtypes, L.orc_bf16_to_float.restype = [c_u16], ctypes.c_float
            L.orc_fp16_value.argtypes, L.orc_fp16_value.restype = [c_u16], ctypes.c_double
            L.orc_fp16_round_down.argtypes, L.orc_fp16_round_down.restype = [ctypes.c_float], c_u16
            L.orc_fp16_round_up.argtypes, L.orc_fp16_round_up.restype = [ctypes.c_float], c_u16
            L.orc_e4m3_value.argtypes, L.orc_e4m3_value.restype = [ctypes.c_uint8], ctypes.c_double
            L.orc_e4m3_encode.argtypes, L.orc_e4m3_encode.restype = [ctypes.c_float], ctypes.c_uint8
            L.orc_quant_int8_row.argtypes = [P, ctypes.c_int, P, P]
            L.orc_quant_fp8_row.argtypes = [P, ctypes.c_int, P, P]
            L.orc_quant_int4_row.argtypes = [P, ctypes.c_int, ctypes.c_int, P, P, P]
            L.orc_quant_int4sym_row.argtypes = [P, ctypes.c_int, ctypes.c_int, P, P]
            L.orc_append.argtypes, L.orc_append.restype = [ctypes.POINTER(_Cache), P, P, P, c_i32], ctypes.c_int
            L.orc_append_kc.argtypes = [ctypes.POINTER(_Cache), P, P, P, P, c_i32]
            L.orc_append_kc.restype = ctypes.c_int
            L.orc_seal_pages.argtypes, L.orc_seal_pages.restype = [ctypes.POINTER(_Cache), P, P, c_i32], ctypes.c_int
            L.orc_quant_kchan_page.argtypes = [P, ctypes.c_int, ctypes.c_int, P, P, P]
            L.orc_decode_attn.argtypes = [ctypes.POINTER(_Cache), P, P, P, c_i32, c_i32, c_i32,
                                          ctypes.c_double, P]
            L.orc_decode_attn.restype = ctypes.c_int
            L.orc_free_list.argtypes = [c_i32, ctypes.c_uint64, P]
            L.orc_splitmix64.argtypes, L.orc_splitmix64.restype = [ctypes.POINTER(ctypes.c_uint64)], ctypes.c_uint64
            L.orc_set_threads.argtypes = [ctypes.c_int]
            L.orc_max_threads.restype = ctypes.c_int
            _lib = L
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


# ---- scalar format helpers -------------------------------------------------------
def fp16_value(bits: int) -> float:
    return lib().orc_fp16_value(bits)


def fp16_round_down(x: float) -> int:
    return lib().orc_fp16_round_down(x)


def fp16_round_up(x: float) -> int:
    return lib().orc_fp16_round_up(x)


def e4m3_value(code: int) -> float:
    return lib().orc_e4m3_value(code)


def e4m3_encode(y: float) -> int:
    return lib().orc_e4m3_encode(y)


def splitmix64_stream(seed: int, n: int) -> list[int]:
    st = ctypes.c_uint64(seed)
    return [lib().orc_splitmix64(ctypes.byref(st)) for _ in range(n)]


# ---- per-row quantizers (x: uint16 bf16 bits) -------------------------------------
def quant_int8_row(x: np.ndarray):
    x = np.ascontiguousarray(x, dtype=np.uint16)
    codes = np.empty(x.size, np.int8)
    sc = np.empty(1, np.float32)
    lib().orc_quant_int8_row(_p(x), x.size, _p(codes), _p(sc))
    return codes, sc[0]


def quant_fp8_row(x: np.ndarray):
    x = np.ascontiguousarray(x, dtype=np.uint16)
    codes = np.empty(x.size, np.uint8)
    sc = np.empty(1, np.float32)
    lib().orc_quant_fp8_row(_p(x), x.size, _p(codes), _p(sc))
    return codes, sc[0]


def quant_int4_row(x: np.ndarray, group: int = 32):
    x = np.ascontiguousarray(x, dtype=np.uint16)
    n = x.size
    packed = np.empty(n // 2, np.uint8)
    sc = np.empty(n // group, np.uint16)
    zp = np.empty(n // group, np.uint16)
    lib().orc_quant_int4_row(_p(x), n, group, _p(packed), _p(sc), _p(zp))
    return packed, sc, zp


def quant_int4sym_row(x: np.ndarray, group: int = 32):
    """Symmetric INT4 of one bf16 row (bits): packed two's-complement nibbles
    and one fp32 scale per group (scale = group absmax / 7)."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    n = x.size
    packed = np.empty(n // 2, np.uint8)
    sc = np.empty(n // group, np.float32)
    lib().orc_quant_int4sym_row(_p(x), n, group, _p(packed), _p(sc))
    return packed, sc


def quant_kchan_page(x: np.ndarray):
    """Per-channel INT8 of one (page, KV head) K block x[P][D] (bf16 bits):
    codes [P][D] int8, channel factors [D] (fp16 bits), token scales [P] fp32."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    P, D = x.shape
    codes = np.empty((P, D), np.int8)
    chan = np.empty(D, np.uint16)
    tok = np.empty(P, np.float32)
    lib().orc_quant_kchan_page(_p(x), P, D, _p(codes), _p(chan), _p(tok))
    return codes, chan, tok


def unpack_int4sym(packed: np.ndarray) -> np.ndarray:
    """The signed codes of a packed symmetric INT4 row (even channel in the
    low nibble, two's complement)."""
    lo = (packed & 0xF).astype(np.int16)
    hi = (packed >> 4).astype(np.int16)
    q = np.empty(packed.size * 2, np.int16)
    q[0::2], q[1::2] = lo, hi
    return np.where(q >= 8, q - 16, q)


# ---- paged cache image ---------------------------------------------------------------
class OracleCache:
    """Host image of one layer's paged quantized cache (numpy arrays).

    Layout: codes [page][kv_head][page_size][head_dim] (INT4 and symmetric
    INT4: head_dim/2 bytes, two codes per byte), scales [page][kv_head]
    [page_size] fp32 (INT4: fp16 bits [..][head_dim/group], plus zeros of the
    same shape; symmetric INT4: fp32 [..][head_dim/group], no zeros).  The
    per-channel K scheme ("int8kc") is INT8 plus channel factors k_chan
    [page][kv_head][head_dim] (fp16 bits) and a residual pool k_resid
    [resid_slots][kv_head][page_size][head_dim] (bf16 bits)."""

    def __init__(self, scheme: str, num_pages: int, page_size: int, num_kv_heads: int,
                 head_dim: int, group: int = 32, resid_slots: int = 0):
        self.scheme = scheme
        self.sid = SCHEME_IDS[scheme]
        self.num_pages, self.page_size = num_pages, page_size
        self.num_kv_heads, self.head_dim = num_kv_heads, head_dim
        self.group = group if scheme in ("int4", "int4sym") else 0
        rows = num_pages * num_kv_heads * page_size
        cb = head_dim // 2 if scheme in ("int4", "int4sym") else head_dim
        self.k_codes = np.zeros(rows * cb, np.uint8)
        self.v_codes = np.zeros(rows * cb, np.uint8)
        if scheme == "int4sym":
            ng = head_dim // group
            self.k_scales = np.zeros(rows * ng, np.float32)
            self.v_scales = np.zeros(rows * ng, np.float32)
            self.k_zeros = self.v_zeros = None
        elif scheme == "int4":
            ng = head_dim // group
            self.k_scales = np.zeros(rows * ng, np.uint16)
            self.v_scales = np.zeros(rows * ng, np.uint16)
            self.k_zeros = np.zeros(rows * ng, np.uint16)
            self.v_zeros = np.zeros(rows * ng, np.uint16)
        else:
            self.k_scales = np.zeros(rows, np.float32)
            self.v_scales = np.zeros(rows, np.float32)
            self.k_zeros = self.v_zeros = None
        self.resid_slots = resid_slots if scheme == "int8kc" else 0
        if scheme == "int8kc":
            self.k_chan = np.zeros(num_pages * num_kv_heads * head_dim, np.uint16)
            self.k_resid = np.zeros(max(self.resid_slots, 1) * num_kv_heads * page_size * head_dim, np.uint16)
        else:
            self.k_chan = self.k_resid = None

    def _struct(self) -> _Cache:
        z = lambda a: None if a is None else a.ctypes.data
        return _Cache(self.sid, self.num_pages, self.page_size, self.num_kv_heads, self.head_dim,
                      self.group, z(self.k_codes), z(self.v_codes), z(self.k_scales),
                      z(self.v_scales), z(self.k_zeros), z(self.v_zeros), z(self.k_chan),
                      z(self.k_resid), self.resid_slots)

    def append(self, slot_mapping: np.ndarray, k_bits: np.ndarray, v_bits: np.ndarray,
               resid_slot: np.ndarray | None = None) -> int:
        """resid_slot (per-channel K only): int32 [T], the residual slot that
        keeps each token's bf16 K row (-1: none)."""
        slot_mapping = np.ascontiguousarray(slot_mapping, np.int64)
        k_bits = np.ascontiguousarray(k_bits, np.uint16)
        v_bits = np.ascontiguousarray(v_bits, np.uint16)
        T = slot_mapping.size
        assert k_bits.size == T * self.num_kv_heads * self.head_dim == v_bits.size
        s = self._struct()
        if resid_slot is None:
            return lib().orc_append(ctypes.byref(s), _p(slot_mapping), _p(k_bits), _p(v_bits), T)
        resid_slot = np.ascontiguousarray(resid_slot, np.int32)
        assert resid_slot.size == T
        return lib().orc_append_kc(ctypes.byref(s), _p(slot_mapping), _p(resid_slot), _p(k_bits),
                                   _p(v_bits), T)

    def seal(self, pages: np.ndarray, resid_slots: np.ndarray) -> int:
        """Per-channel K: re-quantize each page's K per channel from its
        residual slot (pages[i] from resid_slots[i])."""
        pages = np.ascontiguousarray(pages, np.int32)
        resid_slots = np.ascontiguousarray(resid_slots, np.int32)
        assert pages.size == resid_slots.size
        s = self._struct()
        return lib().orc_seal_pages(ctypes.byref(s), _p(pages), _p(resid_slots), pages.size)

    def decode_attn(self, q_bits: np.ndarray, block_table: np.ndarray, seq_lens: np.ndarray,
                    num_q_heads: int, softmax_scale: float = 0.0) -> np.ndarray:
        q_bits = np.ascontiguousarray(q_bits, np.uint16)
        block_table = np.ascontiguousarray(block_table, np.int32)
        seq_lens = np.ascontiguousarray(seq_lens, np.int32)
        B = seq_lens.size
        maxp = block_table.shape[1] if block_table.ndim == 2 else block_table.size // max(B, 1)
        out = np.zeros((B, num_q_heads, self.head_dim), np.float64)
        s = self._struct()
        rc = lib().orc_decode_attn(ctypes.byref(s), _p(q_bits), _p(block_table), _p(seq_lens), B,
                                   num_q_heads, maxp, softmax_scale, _p(out))
        if rc != 0:
            raise ValueError("oracle: block table entry outside the page pool")
        return out


def free_list(num_pages: int, seed: int) -> np.ndarray:
    """Initial free list (allocation pops from the end)."""
    out = np.empty(num_pages, np.int32)
    lib().orc_free_list(num_pages, seed, _p(out))
    return out


def set_threads(n: int) -> None:
    lib().orc_set_threads(n)


def max_threads() -> int:
    return lib().orc_max_threads()


def kv_bytes_per_token(num_layers: int, num_kv_heads: int, head_dim: int, bits: int) -> float:
    """K and V codes per token over all layers: 2 x layers x KV heads x head_dim
    x bytes per element ([P2] "Technical Architecture"; one factor of two, the
    one for K and V; scale overhead is counted separately)."""
    return 2 * num_layers * num_kv_heads * head_dim * bits / 8


def scale_bytes_per_token(num_layers: int, num_kv_heads: int, head_dim: int, scheme: str,
                          group: int = 32) -> int:
    """Scale (and zero-point) overhead per token over all layers."""
    if scheme == "int4":
        return 2 * num_layers * num_kv_heads * (head_dim // group) * (2 + 2)
    if scheme == "int4sym":
        return 2 * num_layers * num_kv_heads * (head_dim // group) * 4
    return 2 * num_layers * num_kv_heads * 4
