"""The bench's multi-GPU host logic, on CPU with two gloo ranks.

The path has no exchange step, so `bench.py --gpus N` runs N independent replicas (weak scaling):
each rank draws its own seeded batch, and the ranks meet only in a barrier around the timed region
and in the max (time) / sum (bytes) reductions of the result. These tests run that logic as two
processes over gloo on 127.0.0.1 -- no GPU -- and check the reference arm's rank-0-only rule.
"""
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads as wl  # noqa: E402


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench as b
    import workloads as w
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        b.barrier(world)
        # per-rank step times and byte counts, as run_gpu reduces them
        t_max = b.all_reduce_max(1.5 + rank, world)
        total = b.all_reduce_sum(1000.0 * (rank + 1), world)
        # each rank's replica: its own seed and its own inputs of the same shapes
        cfg = w.CONFIGS["tiny"]
        case = w.make_case(cfg, device="cpu", seed=b.replica_seed(cfg, rank))
        q_sum = float(case.q.double().sum())
        b.barrier(world)
        out.put((rank, t_max, total, b.replica_seed(cfg, rank), q_sum, int(case.kv_bytes())))
    finally:
        dist.destroy_process_group()


def _run(world: int):
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    res = [out.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return sorted(res)


def test_two_gloo_ranks_reduce_and_draw_independent_replicas():
    res = _run(2)
    assert [r[0] for r in res] == [0, 1]
    for _, t_max, total, _, _, _ in res:
        assert t_max == 2.5        # the slowest rank's time, on every rank
        assert total == 3000.0     # every rank's bytes, on every rank
    seeds = [r[3] for r in res]
    assert seeds[0] != seeds[1]
    assert res[0][4] != res[1][4]  # different inputs ...
    assert res[0][5] == res[1][5]  # ... of the same shapes: the per-rank work is fixed (weak scaling)


def test_single_rank_needs_no_process_group():
    assert bench.all_reduce_max(3.0, 1) == 3.0
    assert bench.all_reduce_sum(4.0, 1) == 4.0
    bench.barrier(1)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    calls = []
    monkeypatch.setattr(bench, "run_reference", lambda args: calls.append(args.config))
    for rank, expect in (("1", []), ("0", ["tiny"])):
        calls.clear()
        monkeypatch.setenv("RANK", rank)
        monkeypatch.setenv("WORLD_SIZE", "2")
        monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--gpus", "2", "--config", "tiny"])
        bench.main()
        assert calls == expect
