"""Host logic of bench.py without a GPU: the multi-process path (gloo,
world size 2) -- barrier, max-over-ranks timing, rank 0 alone printing, the
whole-job rate -- and the command-line contract."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

from conftest import ROOT

sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(WORLD_SIZE=str(world), RANK=str(rank), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    r, w, barrier, reduce_max = bench.make_dist_ctx()
    barrier()
    t = reduce_max(1.5 + r)  # each rank's own "time"; the job takes the slowest
    out.put((r, w, t))
    barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r for r, _, _ in res] == [0, 1]
    assert all(w == world and t == 2.5 for _, w, t in res)


def test_single_process_context_needs_no_process_group():
    r, w, barrier, reduce_max = bench.make_dist_ctx()
    assert (r, w, barrier) == (0, 1, None) and reduce_max(3.25) == 3.25


def test_job_rate_is_weak_scaling_over_the_slowest_rank():
    # 10 MB per step, 1000 steps, slowest rank 2 ms, 4 replicas -> 4 x 10 GB / 2 ms
    assert bench.job_rate(10e6, 1000, 2e-3, 4) == pytest.approx(2e13)
    assert bench.job_rate(10e6, 1000, 2e-3, 1) * 4 == pytest.approx(bench.job_rate(10e6, 1000, 2e-3, 4))


def test_reference_arm_other_ranks_exit_without_work(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    assert bench.main(["--impl", "reference", "--steps", "5", "--warmup", "3"]) == 0


def test_warmup_below_three_is_rejected():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])


def test_step_units_match_the_workload():
    # decode step: the operation's inputs and output once each (bytes): X row, packed
    # codes, scales, zero points, A, B, Y; the intermediate T is not counted
    K = N = 4096
    want = K * 2 + N * K // 2 + N * (K // 32) * 2 + N * (K // 32) + K * 32 * 2 + N * 32 * 2 + N * 2
    assert bench.decode_bytes(1, K, N, 4, 32) == want
    assert bench.prefill_flops(1024, K, N, 32) == 2 * 1024 * N * K + 2 * 1024 * 32 * (K + N)
