"""The bench's multi-rank host logic on CPU with world_size-2 gloo ranks:
the path shards by sequence batches with no data-path collective; the only
exchange is the max over ranks of the timed duration."""
import os
import socket

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
    ms = [3.0, 5.0][rank]  # rank 1 is the slow one
    worst = bench.max_over_ranks(ms, world)
    value = bench.job_throughput(1_000_000_000, world, worst)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, worst, value))


def test_two_ranks_take_the_slowest_time_and_sum_the_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, worst, value in res:
        assert worst == 5.0
        assert value == pytest.approx(2 * 1.0 / 5e-3)  # 2 ranks x 1 GB in 5 ms


def test_single_rank_is_the_identity():
    import bench
    assert bench.max_over_ranks(2.5, 1) == 2.5
    assert bench.job_throughput(10**9, 1, 1.0) == pytest.approx(1000.0)


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
