"""The benchmark's multi-rank logic on CPU: two gloo ranks (the path bench.py
takes under torchrun with one process per GPU).  Each rank owns distinct
layers, the step time is the slowest rank's, the whole-job value is per
layer over all ranks, and the reference arm runs on rank 0 only."""
import os
import socket

import pytest

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local = [2.0, 3.5][rank]
    ms = bench.max_over_ranks(local, dist, "cpu")
    q.put((rank, ms, bench.job_value(ms, world), bench.rank_layer_ids(rank)))
    dist.destroy_process_group()


def test_two_gloo_ranks():
    torch = pytest.importorskip("torch")
    mp = torch.multiprocessing.get_context("spawn")
    q = mp.Queue()
    port = _free_port()
    procs = [mp.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [3.5, 3.5]          # slowest rank
    assert [r[2] for r in res] == [1.75, 1.75]        # ms per layer over the job
    assert not set(res[0][3]) & set(res[1][3])        # disjoint layers


def test_single_rank_needs_no_collective():
    assert bench.max_over_ranks(2.5) == 2.5
    assert bench.job_value(2.5, 1) == 2.5


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    bench.reference_arm(None)   # returns before touching its arguments
    assert capsys.readouterr().out == ""
