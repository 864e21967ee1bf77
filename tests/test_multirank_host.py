"""bench.py's multi-rank host logic, on the CPU.

Runs past one GPU are replicas. Each rank times its own copy of the workload. The
job's time is the maximum over the ranks, taken after a barrier. The job's value counts
every rank's bytes. The reference arm runs on rank 0 only. Here the ranks are two
`gloo` processes.
"""
import contextlib
import importlib.util
import io
import os
import socket
import types

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _load_bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        b = _load_bench()
        # rank r is slower on the first figure and faster on the second
        vals = b.max_over_ranks(torch, dist, [1.0 + rank, 10.0 - rank], "cpu")
        q.put((rank, vals))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    try:
        res = dict(q.get(timeout=180) for _ in ps)
    finally:
        for p in ps:
            p.join(timeout=60)
    assert [p.exitcode for p in ps] == [0, 0]
    assert res[0] == res[1] == [2.0, 10.0]


def test_one_rank_passes_values_through():
    b = _load_bench()
    assert b.max_over_ranks(torch, None, [3.5, 4.0], "cpu") == [3.5, 4.0]


def test_job_value_counts_every_rank():
    b = _load_bench()
    assert b.job_gbs(2, 1e9, 1000.0) == pytest.approx(2.0)
    assert b.job_gbs(4, 1e9, 1000.0) == pytest.approx(4.0)
    assert b.job_gbs(1, 179306496, 0.0338) == pytest.approx(179306496 / 33.8e-6 / 1e9)


def test_reference_arm_runs_on_rank_zero_only():
    b = _load_bench()
    args = types.SimpleNamespace(steps=1, warmup=3)
    out = io.StringIO()
    with contextlib.redirect_stdout(out):
        assert b.run_reference(args, 1, 2) is None
    assert out.getvalue() == ""


def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` (the oracle on the host cores) prints one JSON line
    with the keys the driver reads."""
    import json
    import subprocess
    import sys
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 3
    assert d["value"] > 0 and d["unit"] == "GB/s" and d["higher_is_better"] is True
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
