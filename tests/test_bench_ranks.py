"""The benchmark's multi-rank bookkeeping on CPU ranks (gloo, world size 2): the job's
time is the slowest rank's, the job's rate counts every rank's rows, and the reference
arm runs on rank 0 only.  Replicas only: the timed work has no collective."""
import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks([1.0 + rank, 10.0 - rank, 0.5], dist, "cpu")
        out.put((rank, got, bench.whole_job_rate(4, world, got[0])))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_rate_on_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, rate in res:
        assert got == [2.0, 10.0, 0.5]          # every rank sees the slowest rank's times
        assert rate == pytest.approx(4 * 2 / 2.0e-3)  # 8 rows over 2 ms


def test_single_process_is_its_own_maximum():
    import bench
    assert bench.max_over_ranks([3.0, 4.5], None, "cpu") == [3.0, 4.5]
    assert bench.whole_job_rate(1, 1, 0.5) == pytest.approx(2000.0)


def test_reference_arm_runs_on_rank_zero_only():
    import bench

    class Args:
        workload = 0
        warmup = 1
        steps = 1

    assert bench.run_reference(Args(), 1, 2) is None  # returns before any work


def test_attention_flops_count_the_attended_keys():
    """The tensor roofline's FLOPs: per row and KV group, 8 query heads x (picked regions'
    tokens + own-region tokens) x 128 dims x 4 (Q K^T and P V, multiply and add).  Rows at
    7, 8, 4,100 and 40,000 attend 8, 9, 4,101 and 4,097 keys."""
    import bench
    import synthetic as S
    import block_sparse_attention_step5_gb300 as s5
    w = S.workload({"positions": [7, 8, 4100, 40000], "B": 4})
    assert bench.attention_flops(w, s5.STEP5_GEOMETRY) == (8 + 9 + 4101 + 4097) * 4 * 8 * 128 * 4
