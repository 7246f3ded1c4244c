"""The multi-rank host logic of bench.py on CPU (gloo, world size 2).

Every (sequence, head) is independent and the path has no exchange step, so an N-GPU job runs
N replicas of the workload: the job's step time is the slowest rank's, and its throughput
counts every rank's tokens.  The reference arm runs on rank 0 only.
"""
from __future__ import annotations

import json
import os
import socket
import types

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, step_ms, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench

        ms = bench.max_over_ranks(torch, dist, step_ms[rank], "cpu")
        value = bench.job_throughput(4096, world, ms)
        dist.barrier()
        q.put((rank, ms, value))
    finally:
        dist.destroy_process_group()


def test_two_replicas_report_the_slowest_step_and_every_ranks_tokens():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    step_ms = [2.0, 5.0]
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, step_ms, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
    assert [p.exitcode for p in procs] == [0, 0]
    for rank, ms, value in results:
        assert ms == 5.0
        assert value == pytest.approx(2 * 4096 / 5e-3)


def test_one_rank_is_its_own_maximum():
    import bench

    assert bench.max_over_ranks(torch, None, 3.5, "cpu") == 3.5
    assert bench.job_throughput(64, 1, 2.0) == pytest.approx(32000.0)


def test_reference_arm_runs_on_rank_zero_only(capsys):
    import bench

    args = types.SimpleNamespace(steps=1, warmup=1, gpus=2)
    assert bench.run_reference(args, rank=1) == 0
    assert capsys.readouterr().out == ""
    assert bench.run_reference(args, rank=0) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["metric"] == bench.METRIC and line["unit"] == "tokens/s" and line["higher_is_better"]
    assert all(line["config"][k] == v for k, v in bench.base_config().items())
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]


def test_traffic_digest_follows_included_headers(tmp_path):
    """A committed ncu traffic figure is reported only while the kernel is unchanged; an edit to
    a header the kernel includes (two levels down) must count as a change too."""
    import bench

    (tmp_path / "sub").mkdir()
    src, mid, leaf = tmp_path / "k.cu", tmp_path / "mid.cuh", tmp_path / "sub" / "leaf.cuh"
    src.write_text('#include <cuda.h>\n#include "mid.cuh"\n__global__ void k() {}\n')
    mid.write_text('#pragma once\n#include "sub/leaf.cuh"\n#include "k.cu"\n')   # a cycle ends
    leaf.write_text("#define TILE 32\n")
    d0 = bench.source_digest(str(src))
    assert bench.source_digest(str(src)) == d0
    leaf.write_text("#define TILE 64\n")
    d1 = bench.source_digest(str(src))
    assert d1 != d0
    mid.write_text('#pragma once\n#include "sub/leaf.cuh"\n#include "k.cu"\n// note\n')
    assert bench.source_digest(str(src)) != d1
