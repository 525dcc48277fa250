"""The benchmark's multi-rank host logic on CPU: two gloo ranks (no GPU).

With N ranks every rank runs its own request rows over replicated tables, so
the data path has no collective; the only cross-rank steps are the timing
contract's barrier and the max (and sum) over ranks.  These tests run those
steps as two spawned processes on 127.0.0.1.
"""
import argparse
import json
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import bench
from dspark_markov_draft_anchor_gb300 import workloads


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    d = bench.Dist()
    d.init("gloo")
    d.barrier()
    res = {
        "rank": d.rank,
        "max": d.max(10.0 + 5 * rank),
        "sum": d.sum(1.0 + rank),
    }
    # each rank draws its own rows: same shapes, different values
    wl = workloads.make("tiny", vocab=64, rows=2, steps=2, seed_salt=bench.rank_seed_salt(d.rank))
    res["base_sum"] = int(wl.base.astype(np.int64).sum())
    res["shape"] = wl.base.shape
    d.barrier()
    d.close()
    out.put(res)


def _run(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return sorted(res, key=lambda r: r["rank"])


def test_two_gloo_ranks_max_sum_and_distinct_rows():
    res = _run(2)
    assert [r["max"] for r in res] == [15.0, 15.0]  # the slowest rank's time is the job's
    assert [r["sum"] for r in res] == [3.0, 3.0]
    assert res[0]["shape"] == res[1]["shape"]
    assert res[0]["base_sum"] != res[1]["base_sum"]


def test_single_rank_needs_no_process_group(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    d = bench.Dist()
    d.init("gloo")
    assert d.pg is None and d.world == 1
    assert d.max(3.5) == 3.5 and d.sum(2.0) == 2.0
    d.barrier()
    d.close()


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = argparse.Namespace(steps=1, warmup=0, gpus=2)
    assert bench.run_reference(args, bench.Dist()) == 0
    assert capsys.readouterr().out == ""


def test_algorithmic_bytes_per_step():
    # w2 read + base read + cache write, BF16
    assert bench.algorithmic_bytes_per_step(163840, 16) == 163840 * 256 * 2 + 2 * 16 * 163840 * 2


def test_prob_verify_path_reference_arm_is_declared_unavailable(capsys):
    assert bench.main(["--path", "prob_verify", "--impl", "reference"]) == 0
    line = json.loads(capsys.readouterr().out.strip())
    assert line["impl"] == "reference" and "unavailable" in line


def test_prob_verify_traffic_lookup_is_keyed_by_its_own_sources():
    assert bench.PV_WORKLOAD == "prob_verify_256x5x129280"
    assert bench.source_digest(bench.PV_SOURCES) != bench.source_digest()


def test_algorithmic_bytes_per_step_with_fp8_w2():
    # E4M3 w2 (1 byte an entry) + FP16 row scales + base read + cache write
    assert bench.algorithmic_bytes_per_step(163840, 16, w2="fp8") == 163840 * 256 + 163840 * 2 + 2 * 16 * 163840 * 2
