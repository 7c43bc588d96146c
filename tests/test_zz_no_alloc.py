"""kvq_decode_attn_noalloc: decode attention for callers that cannot
allocate device memory (code inside another framework's memory pool, or a
latency-critical path that cannot take an allocation's synchronization).
It runs the same kernels as kvq_decode_attn on a scratch array compiled into
the library, so its output must match kvq_decode_attn's, call after call.

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
from gpu_harness import ATOL, MEAN_REL, Case, DEV, attn_errors, dev, dev_bits  # noqa: E402


@pytest.mark.parametrize("scheme,Hq,Hkv", [("int8", 32, 8), ("fp8", 64, 8), ("int4", 16, 4)])
def test_noalloc_matches_workspace_call_twice(scheme, Hq, Hkv):
    w = inp.Workload(0, "noalloc", scheme, 1, 1, Hq, Hkv, 128, 16, ("fixed", 0), seed=11,
                     outlier_pairs=2, outlier_gain=8.0)
    # several sequences, one long enough to be split across CTAs, one empty
    lens = np.array([3000, 17, 0, 20000, 511], np.int32)
    case = Case(w, lens, oracle_seqs=[])
    q, bt, sl = dev_bits(case.q), dev(case.bt), dev(lens)
    ref = case.decode()  # kvq_decode_attn with a torch-allocated workspace
    need = kvq.decode_workspace_bytes(case.g, len(lens), Hq, bt.shape[1])
    assert need <= 16 << 20  # KVQ_STATIC_SCRATCH_BYTES
    for _ in range(2):
        out = torch.full((len(lens), Hq, 128), float("nan"), dtype=torch.float32, device=DEV)
        st = kvq.lib.kvq_decode_attn_noalloc(ctypes.byref(case.g.struct), ctypes.c_void_p(q.data_ptr()),
                                             ctypes.c_void_p(bt.data_ptr()), ctypes.c_void_p(sl.data_ptr()),
                                             ctypes.c_void_p(out.data_ptr()), len(lens), Hq, bt.shape[1],
                                             0.0, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == kvq.OK, kvq.status_string(st)
        assert kvq.last_device_error() == kvq.OK
        got = out.cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(got))
        max_abs, mean_rel = attn_errors(got, ref)
        assert max_abs <= ATOL and mean_rel <= MEAN_REL, (max_abs, mean_rel)
        assert np.all(got[2] == 0)
