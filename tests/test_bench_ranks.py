"""The bench's multi-process arithmetic, on CPU with two gloo ranks: the timed region
is the slowest rank's (max over ranks), the throughput counts every rank's tokens
(sum over ranks), and the shards are independent (weak scaling, no data-path
collective).  Also the choice of runner for the line the JSON leads with."""

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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench

        w, r, local = bench.dist_info()
        assert (w, r, local) == (world, rank, rank)
        ms = bench.max_over_ranks(10.0 + rank, world)  # rank 1 is the slow one
        tokens = bench.sum_over_ranks(64.0 * (rank + 1), world)
        bench.barrier(world)
        out[rank] = (ms, tokens)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_summed_tokens():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        ms, tokens = res[rank]
        assert ms == pytest.approx(11.0)
        assert tokens == pytest.approx(64.0 + 128.0)


def test_single_process_helpers_are_identity():
    import bench

    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.sum_over_ranks(7.0, 1) == 7.0
    bench.barrier(1)


@pytest.mark.parametrize("head", ["backward", "base_fused", "prefill"])
@pytest.mark.parametrize("cpu_seconds", [0.0, 2.0])
def test_head_line_runs_one_runner(monkeypatch, head, cpu_seconds):
    """The leading line runs exactly one runner for its workload, whatever --cpu-seconds is,
    and the backward and base-projection lines get their own oracle baseline only when asked."""
    import argparse

    import bench

    calls = []

    def runner(kind):
        def run(*a, **k):
            calls.append(kind)
            return {"value": 1.0}
        return run

    monkeypatch.setattr(bench, "run_backward_line", runner("backward"))
    monkeypatch.setattr(bench, "run_base_line", runner("base_fused"))
    monkeypatch.setattr(bench, "config_line", runner("config"))
    monkeypatch.setattr(bench, "cpu_baseline_line", lambda kind, s: {"kind": "oracle", "of": kind})
    args = argparse.Namespace(steps=3, warmup=3, soak_seconds=0.0, cpu_seconds=cpu_seconds)
    h = bench.head_line(head, args, 1, 0, 0)
    assert calls == [head if head in ("backward", "base_fused") else "config"]
    if head in ("backward", "base_fused") and cpu_seconds > 0:
        assert h["cpu_baseline"] == {"kind": "oracle", "of": head}
    else:
        assert "cpu_baseline" not in h
