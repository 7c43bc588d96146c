"""kvq_decode_attn_noalloc: decode attention for callers that cannot
allocate device memory (code inside another framework's memory pool, or a
latency-critical path that cannot take an allocation's synchronization).
It runs the same kernel, with the same plan, as kvq_decode_attn on a scratch
array compiled into the library, so its output must equal kvq_decode_attn's
bit for bit, call after call -- also when consecutive calls have different
shapes and schemes, so that each call finds the previous call's partials where
its own arrival counters live.

This file is collected last on purpose; it must pass both on its own in a
fresh process and after the other GPU tests."""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import dynamically_quantized_paged_gb300 as kvq  # noqa: E402
import kvq_inputs as inp  # noqa: E402
from gpu_harness import Case, DEV, dev, dev_bits  # noqa: E402

SCRATCH_BYTES = 16 << 20  # KVQ_STATIC_SCRATCH_BYTES


def _noalloc_abi(case, q, bt, sl, out, Hq):
    """One call through the C ABI (ctypes), on the current stream."""
    return kvq.lib.kvq_decode_attn_noalloc(
        ctypes.byref(case.g.struct), ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(bt.data_ptr()),
        ctypes.c_void_p(sl.data_ptr()), ctypes.c_void_p(out.data_ptr()), sl.numel(), Hq, bt.shape[1], 0.0,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _case(scheme, Hq, Hkv, lens, seed):
    w = inp.Workload(0, "noalloc", scheme, 1, 1, Hq, Hkv, 128, 16, ("fixed", 0), seed=seed,
                     outlier_pairs=2, outlier_gain=8.0)
    return Case(w, np.asarray(lens, np.int32), oracle_seqs=[])


# Consecutive calls alternate batch size, head count and scheme; each problem
# has a sequence long enough to be split across CTAs (cross-CTA merge through
# the arrival counters) and an empty one.
PROBLEMS = [
    ("int8", 32, 8, [3000, 17, 0, 20000, 511], 11),
    ("fp8", 64, 8, [9000, 0, 40], 12),
    ("int4", 16, 4, [1, 12000, 0, 700, 5000, 33, 2048], 13),
    ("int8", 16, 8, [25000, 0], 14),
    ("int8kc", 32, 8, [6000, 0, 900], 15),  # per-channel K (pages open: token rule, factors 1.0)
]


def test_noalloc_equals_workspace_call_across_shapes():
    cases = [_case(*p) for p in PROBLEMS]
    refs = [c.decode() for c in cases]  # kvq_decode_attn with a torch-allocated workspace
    for round_ in range(2):  # two calls of each, in alternating order
        for (scheme, Hq, Hkv, lens, _), case, ref in zip(PROBLEMS, cases, refs):
            need = kvq.decode_workspace_bytes(case.g, len(lens), Hq, case.bt.shape[1])
            assert need <= SCRATCH_BYTES
            q, bt, sl = dev_bits(case.q), dev(case.bt), dev(case.lens)
            out = torch.full((len(lens), Hq, 128), float("nan"), dtype=torch.float32, device=DEV)
            st = _noalloc_abi(case, q, bt, sl, out, Hq)
            assert st == kvq.OK, kvq.status_string(st)
            assert kvq.last_device_error() == kvq.OK
            got = out.cpu().numpy().astype(np.float64)
            assert np.array_equal(got, ref), f"{scheme} Hq={Hq} call {round_}: differs from kvq_decode_attn"
            assert all(np.all(got[b] == 0) for b, L in enumerate(lens) if L == 0)


def test_noalloc_python_binding():
    scheme, Hq, Hkv, lens, seed = PROBLEMS[0]
    case = _case(scheme, Hq, Hkv, lens, seed)
    ref = case.decode()
    out = torch.full((len(lens), Hq, 128), float("nan"), dtype=torch.float32, device=DEV)
    kvq.decode_attn_noalloc(case.g, dev_bits(case.q), dev(case.bt), dev(case.lens), out)
    assert kvq.last_device_error() == kvq.OK
    assert np.array_equal(out.cpu().numpy().astype(np.float64), ref)


def test_noalloc_rejects_problems_beyond_the_array():
    """A problem whose workspace need exceeds the array gets KVQ_ERR_WORKSPACE
    and nothing is enqueued: the output keeps its contents."""
    g = None
    for Hkv in (64, 128, 256, 512):
        cand = kvq.PagedKVCache("int8", 1, 16, Hkv, 128, device=DEV)
        B = 4096
        if kvq.decode_workspace_bytes(cand, B, 8 * Hkv, 1) > SCRATCH_BYTES:
            g = cand
            break
    assert g is not None, "no problem needing more than the array was found"
    Hq = 8 * g.num_kv_heads
    # nothing is read before the size check: small stand-in buffers suffice
    q = torch.zeros(64, dtype=torch.int16, device=DEV)
    bt = torch.zeros((B, 1), dtype=torch.int32, device=DEV)
    sl = torch.zeros(B, dtype=torch.int32, device=DEV)
    out = torch.full((64,), 7.0, dtype=torch.float32, device=DEV)
    st = kvq.lib.kvq_decode_attn_noalloc(
        ctypes.byref(g.struct), ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(bt.data_ptr()),
        ctypes.c_void_p(sl.data_ptr()), ctypes.c_void_p(out.data_ptr()), B, Hq, 1, 0.0,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 8  # KVQ_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert kvq.last_device_error() == kvq.OK
    assert torch.all(out == 7.0)
