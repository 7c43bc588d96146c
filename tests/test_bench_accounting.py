"""The bench's algorithmic byte counts, checked against hand computations
for small steps (CPU only).  These are the numerators of every GB/s and
roofline figure the bench prints."""
import dataclasses

import numpy as np

import bench
import kvq_inputs as inp


def _w(scheme, H=2, D=64, P=16, Hq=4):
    return dataclasses.replace(inp.WORKLOADS[2], scheme=scheme, kv_heads=H, head_dim=D, page_size=P, q_heads=Hq,
                               batch=2, layers=1)


def test_int8_decode_and_append_bytes():
    w = _w("int8")
    lens = np.array([20, 16])          # 36 cached tokens, pages 2 + 1
    n_new = np.array([1, 1])
    nb = bench.algorithmic_bytes(w, lens, n_new)
    H, D, Hq, B = 2, 64, 4, 2
    kv = 36 * 2 * H * (D + 4)          # K and V codes plus fp32 scales, every cached token
    decode = kv + 3 * 4 + B * Hq * D * 2 + B * Hq * D * 4 + B * 4   # + table, q, out, lengths
    append = 2 * (2 * H * D * 2 + 8 + 2 * H * (D + 4))              # bf16 rows + slot in, codes + scales out
    assert nb["decode"] == decode and nb["append"] == append and nb["seal"] == 0
    assert nb["step"] == decode + append and nb["append_tokens"] == 2


def test_int4_group_metadata_bytes():
    w = _w("int4", D=128)
    nb = bench.algorithmic_bytes(w, np.array([32]), np.array([1]))
    H, D = 2, 128
    per_token = 2 * H * (D // 2 + (D // 32) * 4)   # packed codes, fp16 scale + zero per 32-channel group
    assert nb["kv_bytes"] == 32 * per_token


def test_per_channel_k_adds_factors_residual_rows_and_the_seal():
    w = _w("int8kc")
    P, H, D, Hq = 16, 2, 64, 4
    lens = np.array([16, 33])          # sequence 0's token completes page 0; sequence 1's opens page 2
    n_new = np.array([1, 1])
    base = bench.algorithmic_bytes(_w("int8"), lens, n_new)
    nb = bench.algorithmic_bytes(w, lens, n_new)
    pages = 1 + 3
    assert nb["decode"] == base["decode"] + pages * H * D * 2           # the pages' channel factors
    opened = 1                                                          # position 32 is offset 0
    assert nb["append"] == base["append"] + 2 * (4 + H * D * 2) + opened * H * D * 2
    assert bench.sealed_pages_of_step(lens, n_new, P) == 1              # position 15 fills page 0
    assert nb["seal"] == 1 * (8 + H * (P * D * 2 + P * D + D * 2 + P * 4))
    assert nb["step"] == nb["decode"] + nb["append"] + nb["seal"]


def test_chunked_append_counts_every_new_token():
    w = dataclasses.replace(inp.WORKLOADS[5], batch=1)
    lens = inp.seq_lens(w)
    n_new = bench.step_plan(w, lens)
    assert int(n_new.sum()) == w.prefill_chunk
    nb = bench.algorithmic_bytes(w, lens, n_new)
    assert nb["append"] == w.prefill_chunk * (2 * w.kv_heads * w.head_dim * 2 + 8 + 2 * w.kv_heads * (w.head_dim + 4))
