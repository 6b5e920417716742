"""Host-side logic of bench.py, on CPU: the max-over-ranks aggregation of a multi-rank
run (two gloo ranks on 127.0.0.1) and the reference arm (the CPU oracle) on the tiny
workload."""

import contextlib
import io
import json
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms_local = 2.0 if rank == 0 else 5.0      # rank 1 is the slow one
        ms_max, value = bench.aggregate(ms_local, 1000, world)
        out[rank] = (ms_max, value)
    finally:
        dist.destroy_process_group()


def test_aggregate_max_over_two_gloo_ranks():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        ms_max, value = res[rank]
        assert ms_max == pytest.approx(5.0)
        assert value == pytest.approx(world * 1000 / 5e-3)   # whole-job units per second


def test_aggregate_single_rank():
    ms, value = bench.aggregate(4.0, 500, 1)
    assert ms == 4.0 and value == pytest.approx(500 / 4e-3)


def test_reference_arm_json_line():
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "3",
                    "--warmup", "3"])
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["unit"] == bench.UNIT and line["value"] > 0
    assert line["config"]["workload"] == "tiny"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_profiled_traffic_requires_matching_source(tmp_path, monkeypatch):
    """The traffic figure is used only if the profile names this workload and size and was
    taken on the top-k source as it is now."""
    import hashlib
    with open(bench.TOPK_SOURCE, "rb") as f:
        sha = hashlib.sha256(f.read()).hexdigest()
    w = bench.wl.WORKLOADS["gemma_large"]
    prof = tmp_path / "p.json"
    monkeypatch.setattr(bench, "PROFILE_TOPK", str(prof))
    good = {"workload": "gemma_large", "R": 512, "source_sha256": sha,
            "traffic_bytes_per_launch": 123.0}
    prof.write_text(json.dumps(good))
    assert bench.profiled_traffic(w) == 123.0
    prof.write_text(json.dumps(dict(good, source_sha256="0" * 64)))
    assert bench.profiled_traffic(w) is None          # the top-k source has changed since
    prof.write_text(json.dumps(dict(good, R=32)))
    assert bench.profiled_traffic(w) is None          # another size
    assert bench.profiled_traffic(bench.wl.WORKLOADS["qwen_zipf"]) is None
