"""Host-side logic of bench.py without a GPU: argument defaults, the
max-over-ranks reduction over a real 2-rank gloo process group, the replica
aggregation, the reference arm's rank handling, and peak loading."""
from __future__ import annotations

import json
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.reduce_max(10.0 + rank * 5.0, world, torch.device("cpu"))
        bench.barrier(world)
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=10) for _ in range(2))
    assert res == {0: 15.0, 1: 15.0}


def test_args_defaults_and_warmup_floor():
    a = bench.parse_args([])
    assert a.gpus == 1 and a.steps > 0 and a.warmup >= 3 and a.impl == "ours"
    assert bench.parse_args(["--warmup", "1"]).warmup == 3


def test_reference_arm_nonzero_rank_exits_without_work(capsys):
    a = bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "0"])
    assert bench.run_reference(a, world=2, rank=1) == 0
    assert capsys.readouterr().out == ""


def test_reference_arm_prints_contract_line(capsys, monkeypatch):
    monkeypatch.setattr(bench, "CPU_SAMPLE_ROWS_A", 8)
    monkeypatch.setattr(bench, "CPU_SAMPLE_ROWS_W", 128)
    fake = [(torch.randn(64, 256).to(torch.bfloat16), (torch.randn(256, 256) * 0.02).to(torch.bfloat16))]
    import fp8_block_scaled_05_gb300.inputs as I

    class _C:
        def __init__(self, a, w):
            self.a, self.w = a, w
    monkeypatch.setattr(I, "llama8b_layers", lambda seed=0: [_C(a, w) for a, w in fake])
    a = bench.parse_args(["--impl", "reference", "--steps", "2", "--warmup", "0"])
    assert bench.run_reference(a, world=1, rank=0) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "cpu_baseline", "e2e", "impl"):
        assert k in line
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_peaks_fallback_and_measured(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    p = bench.load_peaks()
    assert p["source"] == "fallback" and p["hbm_gbs"] == 6800.0 and p["bf16_tflops"] == 1900.0
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 7100, "bf16_tflops": 2000}))
    p = bench.load_peaks()
    assert p["source"] == "measured" and p["hbm_gbs"] == 7100 and p["bf16_tflops"] == 2000
