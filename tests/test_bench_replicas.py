"""The multi-GPU bench path on CPU: two ranks over gloo run independent
replicas, and the job's timing is the slowest rank's (max over ranks); the
whole-job throughput counts every rank's cycles.  No data-path collective
exists, so this timing reduction is the only one exercised."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r's replica took 100 + 10 r ms for its cycles and 2 + r s end to end
        got = bench.max_over_ranks([100.0 + 10 * rank, 2.0 + rank])
        out[rank] = (got, bench.replica_throughput(world, 50, got[0]))
    finally:
        dist.destroy_process_group()


def test_two_replicas_time_is_the_slowest_rank():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        got, value = res[r]
        assert got == [110.0, 3.0]
        assert value == pytest.approx(2 * 50 / 0.110)


def test_single_rank_needs_no_collective():
    import bench
    assert bench.max_over_ranks([7.0, 1.5]) == [7.0, 1.5]
    assert bench.replica_throughput(1, 3000, 1500.0) == pytest.approx(2000.0)


def test_window_options_size_the_state_and_bytes():
    """--ctx / --window: a ring of the window rounded to 128 cells, and K/V
    bytes for the attended positions only; the default workload unchanged."""
    import argparse
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    base = bench.workload_config(argparse.Namespace(weight_type=None, ctx=0, window=0))
    assert bench.state_capacity(base) == base.ctx + base.block
    full = bench.algorithmic_bytes(base, base.ctx, base.block, 8)
    assert full["step"] == 1884651520  # 1.792 GB draft + 92 MB fusion at 8192 positions, BF16
    win = bench.workload_config(argparse.Namespace(weight_type="q8_0", ctx=262144, window=32768))
    assert win.attn_window == 32768 and bench.state_capacity(win) == 32768
    b = bench.algorithmic_bytes(win, win.ctx, win.block, 8)
    nowin = bench.algorithmic_bytes(win.with_(attn_window=0), win.ctx, win.block, 8)
    kv_per_pos = win.n_layers * 2 * win.n_kv_heads * win.head_dim * 2
    assert nowin["draft"] - b["draft"] == kv_per_pos * (win.ctx + win.block - 32768)
    assert bench.state_capacity(win.with_(attn_window=100)) == 128
