"""The bench's multi-rank host logic on CPU with world_size-2 gloo ranks:
the path shards by sequences (each rank takes a share of the batch with its
own pages and block-table rows) with no data-path collective; the only
exchanges are the max over ranks of the timed duration and the sum of the
ranks' work."""
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import kvq_inputs as inp
    ms = [3.0, 5.0][rank]  # rank 1 is the slow one
    worst = bench.max_over_ranks(ms, world)
    work = bench.sum_over_ranks([1_000_000_000, 500_000_000][rank], world)
    value = bench.job_throughput(work, worst)
    # each rank's share of every workload, and the bytes it moves per step
    shares, totals = {}, {}
    for cid, w in inp.WORKLOADS.items():
        lens = inp.seq_lens(w)
        mine = bench.partition_sequences(lens, world)[rank]
        nb = bench.algorithmic_bytes(w, lens[mine], bench.step_plan(w, lens[mine]))
        shares[cid] = mine.tolist()
        totals[cid] = (bench.sum_over_ranks(nb["step"], world), bench.sum_over_ranks(len(mine), world))
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, worst, work, value, shares, totals))


def test_two_ranks_split_the_batch_and_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    import bench
    import kvq_inputs as inp
    for rank, worst, work, value, shares, totals in res:
        assert worst == 5.0
        assert work == 1_500_000_000
        assert value == pytest.approx(1.5 / 5e-3)  # 1.5 GB in the slowest rank's 5 ms
    for cid, w in inp.WORKLOADS.items():
        lens = inp.seq_lens(w)
        a, b = res[0][4][cid], res[1][4][cid]
        # the shares cover every sequence exactly once
        assert sorted(a + b) == list(range(w.batch))
        # the ranks' bytes add up to the single-GPU step's
        whole = bench.algorithmic_bytes(w, lens, bench.step_plan(w, lens))["step"]
        assert res[0][5][cid] == res[1][5][cid] == (whole, w.batch)


def test_partition_balances_tokens_and_is_deterministic():
    import bench
    import kvq_inputs as inp
    for cid, w in inp.WORKLOADS.items():
        lens = inp.seq_lens(w)
        for world in (1, 2, 3, 4, 8):
            shares = bench.partition_sequences(lens, world)
            assert len(shares) == world
            assert sorted(np.concatenate(shares).tolist()) == list(range(w.batch))
            assert all(np.all(np.diff(s) > 0) for s in shares)
            loads = [int(lens[s].sum()) for s in shares]
            # longest-first greedy: no rank exceeds the mean by more than the longest sequence
            assert max(loads) <= sum(loads) / world + int(lens.max())
            again = bench.partition_sequences(lens, world)
            assert all(np.array_equal(x, y) for x, y in zip(shares, again))


def test_single_rank_is_the_identity():
    import bench
    assert bench.max_over_ranks(2.5, 1) == 2.5
    assert bench.sum_over_ranks(7, 1) == 7
    assert bench.job_throughput(10**9, 1.0) == pytest.approx(1000.0)


def test_end_to_end_staging_layout_round_trips():
    """The end-to-end step stages every input tensor in one pinned buffer:
    offsets are aligned, regions do not overlap, and each view reads back its
    tensor exactly."""
    import torch
    import bench
    g = torch.Generator().manual_seed(7)
    srcs = [torch.randn(3, 5, 8, generator=g).to(torch.bfloat16),
            torch.randint(0, 1 << 40, (37,), generator=g, dtype=torch.int64),
            torch.randint(-1, 100, (4, 9), generator=g, dtype=torch.int32),
            torch.randint(0, 100, (1,), generator=g, dtype=torch.int32),
            torch.empty(0, dtype=torch.int32)]
    offs, total = bench.stage_layout(srcs)
    ends = [o + t.numel() * t.element_size() for o, t in zip(offs, srcs)]
    assert all(o % bench.STAGE_ALIGN == 0 for o in offs)
    assert all(e <= o for e, o in zip(ends, offs[1:]))
    assert total == ends[-1]
    buf = torch.full((total,), 0xAB, dtype=torch.uint8)
    for t, o in zip(srcs, offs):
        bench.stage_view(buf, t, o).copy_(t)
    for t, o in zip(srcs, offs):
        v = bench.stage_view(buf, t, o)
        assert v.dtype == t.dtype and v.shape == t.shape and v.is_contiguous()
        assert torch.equal(v, t)
