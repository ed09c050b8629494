"""The N > 1 path of bench.py on the CPU: world-size-2 gloo ranks.

Each rank runs its own replica of the workload (weak scaling, no data-path
collective); the only exchange is the timing: the job's rate is the bytes all
ranks moved over the slowest rank's time, and only rank 0 prints.  No GPU.
"""
import json
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        # rank r: 2 + r ms for 1e9 * (r + 1) bytes
        gbs, ms = bench.whole_job_rate(torch, dist, 2.0 + rank, 1e9 * (rank + 1))
        m = bench.max_over_ranks(torch, dist, float(rank))
        sm = bench.sum_over_ranks(torch, dist, float(rank + 1))
        out[rank] = (gbs, ms, m, sm)
    finally:
        dist.destroy_process_group()


def test_whole_job_rate_over_two_gloo_ranks():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn",
                       join=True)
    for r in range(world):
        gbs, ms, m, sm = out[r]
        # (1e9 + 2e9) bytes over the slowest rank's 3 ms
        assert ms == pytest.approx(3.0)
        assert gbs == pytest.approx(3e9 / 3e-3 / 1e9)
        assert m == 1.0 and sm == 3.0


def test_single_process_rate_needs_no_process_group():
    import bench
    gbs, ms = bench.whole_job_rate(torch, None, 4.0, 2e9)
    assert ms == 4.0 and gbs == pytest.approx(2e9 / 4e-3 / 1e9)


def test_reference_arm_prints_on_rank_zero_only(capsys, monkeypatch):
    import bench

    class Args:
        steps, warmup, gpus, workload = 1, 0, 2, "gqa"

    # rank 1 returns without work and prints nothing
    assert bench.reference_arm(Args(), 1, 2) == 0
    assert capsys.readouterr().out == ""
    # rank 0 prints one JSON line (the oracle rate and the config are stubbed:
    # no timing here)
    monkeypatch.setattr(bench, "oracle_rate", lambda name, seconds: {
        "value": 1.5, "unit": "GB/s", "cores": 4, "kind": "oracle", "sample": "stub sample",
        "per_layer_ms": 2.0})
    monkeypatch.setattr(bench, "workload_config", lambda name: {"workload": name, "batch": 16})
    assert bench.reference_arm(Args(), 0, 2) == 0
    line = json.loads(capsys.readouterr().out.strip())
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] == 1.5
    assert line["cpu_baseline"]["cores"] == 4 and line["cpu_baseline"]["per_layer_ms"] == 2.0
    assert line["config"] == {"workload": "gqa", "batch": 16}
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_config_matches_the_gpu_arm_config():
    """Both arms print the same config block for a workload (built from host
    copies of the inputs here; from the device inputs in the GPU arm)."""
    import bench
    import workloads
    c = bench.workload_config("npuw")
    w = workloads.npuw(device="cpu", layers=1)
    assert c == bench.masked_config("npuw", w, 32, [int(x) for x in w.layers[0].lengths])
    assert c["layers"] == 32 and c["capacity"] == 1152 and c["q_heads"] == 32
    g = bench.workload_config("gqa")
    assert g["batch"] == 16 and g["kv_heads"] == 8 and g["layers"] == 32
    assert g["valid_len_step0"]["min"] >= 512 and g["valid_len_step0"]["max"] <= 8192
