"""Multi-rank host logic, run as gloo ranks on the CPU.

* bench.py: every rank gets the slowest rank's step time, and the reported
  value is the units all ranks processed over that time (independent
  sequences per rank, weak scaling: no collective touches the data).
* The sequence split: one sequence cut into per-rank segments needs one
  exchange, an all-gather of the segments' state transfers, after which each
  rank composes its own entering state."""
from __future__ import annotations

import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, step_ms, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.rank_barrier()
        slowest = bench.max_over_ranks(step_ms[rank], "cpu")
        rate = bench.whole_job_rate(32768, slowest, world)
        bench.rank_barrier()
        out.put((rank, slowest, rate))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_step():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    step_ms = [1.25, 2.5]
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, step_ms, out)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(out.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, rate in got:
        assert slowest == 2.5
        assert rate == pytest.approx(2 * 32768 / 2.5e-3)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.0, "cpu") == 3.0
    assert bench.whole_job_rate(100, 2.0, 1) == pytest.approx(50_000.0)


def test_several_gpus_without_torchrun_is_refused():
    env = dict(os.environ)
    env.pop("WORLD_SIZE", None)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2"],
                       capture_output=True, text=True, env=env, cwd=ROOT, timeout=120)
    assert r.returncode != 0
    assert "torchrun" in (r.stderr + r.stdout)


def _exchange_main(rank, world, port, Ms, Ss, h0, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    from chunkwise_gated_delta_gdn_gb300 import seqsplit

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        s_in = seqsplit.exchange_and_compose(Ms[rank], Ss[rank], h0,
                                             combine=lambda M, S, Sg: M @ S + Sg)
        out.put((rank, s_in))
    finally:
        dist.destroy_process_group()


def test_three_ranks_compose_the_state_transfers_in_rank_order():
    """Each rank's entering state is the composition of the transfers of the
    ranks before it (the sequence-split exchange), checked against a plain
    sequential fold."""
    import torch

    gen = torch.Generator().manual_seed(5)
    world = 3
    Ms = [torch.randn((1, 2, 4, 4), generator=gen, dtype=torch.float64) * 0.5 for _ in range(world)]
    Ss = [torch.randn((1, 2, 4, 3), generator=gen, dtype=torch.float64) for _ in range(world)]
    h0 = torch.randn((1, 2, 4, 3), generator=gen, dtype=torch.float64)
    expect, s = [], h0
    for p in range(world):
        expect.append(s)
        s = Ms[p] @ s + Ss[p]
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_exchange_main, args=(r, world, port, Ms, Ss, h0, out))
             for r in range(world)]
    for p in procs:
        p.start()
    got = dict(out.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(world):
        assert torch.allclose(got[r], expect[r], atol=1e-12), r
