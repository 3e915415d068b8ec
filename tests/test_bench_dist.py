"""The benchmark's multi-rank logic on CPU (gloo, world size 2): the
timing reduction takes the slowest rank, and the reference arm runs on rank 0
only (other ranks exit without work)."""
import io
import json
import os
import contextlib

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks(10.0 + 5.0 * rank, world, "cpu")
        q.put(("max", rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert [r[2] for r in res] == [15.0, 15.0]


def test_reference_arm_rank_handling(monkeypatch):
    import argparse
    ns = argparse.Namespace(gpus=2, steps=1, warmup=0, impl="reference", config="tiny", fused=False,
                            unfused=False, tokens_per_slot=0, world=0, experts=0,
                            no_cpu_baseline=False, no_e2e=False)
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        assert bench.run_reference(ns) == 0
    assert buf.getvalue() == ""                      # non-zero ranks print nothing
    monkeypatch.setenv("RANK", "0")
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        assert bench.run_reference(ns) == 0
    line = json.loads(buf.getvalue())
    assert line["impl"] == "reference" and line["unit"] == "tokens/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0


def test_traffic_record_only_for_its_workload():
    """The committed DRAM-traffic record is reported only for the workload
    and shape it was captured on, and only while its sources are unchanged."""
    import json
    import moe_synth as ms
    rec = json.load(open(os.path.join(bench.ROOT, "profiles", "traffic.json")))
    name = rec["workload"]
    cfg = dict(ms.CONFIGS[name])
    expect = rec["traffic_bytes_per_step"] if rec["sources_code_sha256"] == bench.sources_code_sha256() else None
    assert bench.traffic_record(name, cfg) == expect
    other = next(k for k in ms.CONFIGS if k != name)
    assert bench.traffic_record(other, dict(ms.CONFIGS[other])) is None
    assert bench.traffic_record(name, dict(cfg, tokens_per_slot=cfg["tokens_per_slot"] // 2)) is None
