"""Host side of bench.py under torchrun (no GPU): replicas only, so ranks exchange nothing but
timing. Two gloo ranks on 127.0.0.1 check the barrier and the max / sum over ranks that turn
per-rank times and units into the job's figures, and the reference arm's rank rule (rank 0
alone times the oracle and prints; the others exit without work)."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

RANK_SCRIPT = r"""
import json, os, sys, time
sys.path.insert(0, sys.argv[1])
import torch
import bench
rank, world, local = bench.dist_env()
bench.init_dist(world, "gloo")
cpu = torch.device("cpu")
if rank == 1:
    time.sleep(0.2)                      # the slower replica; the barrier must wait for it
t0 = time.time()
bench.barrier(world)
waited = time.time() - t0
job_s = bench.max_over_ranks(1.5 + rank, world, cpu)          # slowest replica sets the time
units = bench.sum_over_ranks(10.0 * (rank + 1), world, cpu)    # every replica's tokens count
print(json.dumps({"rank": rank, "world": world, "local": local, "job_s": job_s, "units": units,
                  "waited": waited}), flush=True)
torch.distributed.destroy_process_group()
"""


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_aggregate_time_and_units(tmp_path):
    script = tmp_path / "rank.py"
    script.write_text(RANK_SCRIPT)
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                   WORLD_SIZE="2", LOCAL_RANK=str(rank), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, str(script), ROOT], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        try:
            o, e = p.communicate(timeout=120)
        except subprocess.TimeoutExpired:
            for q in procs:
                q.kill()
            pytest.fail("gloo ranks did not finish")
        assert p.returncode == 0, e
        outs.append(json.loads(o.strip().splitlines()[-1]))
    for r in outs:
        assert r["world"] == 2 and r["local"] == r["rank"]
        assert r["job_s"] == 2.5            # max(1.5, 2.5)
        assert r["units"] == 30.0           # 10 + 20
    assert outs[0]["waited"] > 0.1          # rank 0 waited at the barrier for the late rank


def test_single_process_needs_no_process_group(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (0, 1, 0)
    bench.init_dist(1, "gloo")
    bench.barrier(1)
    assert bench.max_over_ranks(3.0, 1, None) == 3.0
    assert bench.sum_over_ranks(4.0, 1, None) == 4.0


def test_reference_arm_other_ranks_do_no_work(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("LOCAL_RANK", "1")
    bench.main(["--impl", "reference", "--config", "tiny_fp8_decode", "--steps", "2"])
    assert capsys.readouterr().out == ""


def test_reference_arm_line_on_rank0(monkeypatch, capsys):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    bench.main(["--impl", "reference", "--config", "tiny_fp8_decode", "--steps", "2", "--warmup", "3"])
    lines = [l for l in capsys.readouterr().out.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["steps"] == 2 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["cpu_baseline"]["value"] == d["value"] and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["config"]["workload"] == "tiny_fp8_decode"
