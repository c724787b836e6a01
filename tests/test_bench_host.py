"""Host-side checks of bench.py that need no GPU: the library drives one GPU, so a
multi-rank launch prints one "unavailable" line on rank 0 and no work runs on any
rank; the CPU-baseline record names the host's CPU and core count."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(env_extra, *args):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], env=env, capture_output=True,
                          text=True, timeout=120)


def test_multi_rank_launch_is_unavailable_on_rank0_and_silent_elsewhere():
    r0 = _run({"RANK": "0", "LOCAL_RANK": "0", "WORLD_SIZE": "2"}, "--gpus", "2")
    assert r0.returncode == 0
    lines = [l for l in r0.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert "unavailable" in rec and rec["n_gpus"] == 2
    r1 = _run({"RANK": "1", "LOCAL_RANK": "1", "WORLD_SIZE": "2"}, "--gpus", "2")
    assert r1.returncode == 0 and r1.stdout.strip() == ""


def test_gpus_flag_alone_is_unavailable():
    r = _run({"RANK": "0", "LOCAL_RANK": "0", "WORLD_SIZE": "1"}, "--gpus", "4")
    assert r.returncode == 0 and "unavailable" in json.loads(r.stdout.strip().splitlines()[-1])


def test_host_cpu_record():
    sys.path.insert(0, ROOT)
    import bench
    hc = bench.host_cpu()
    assert isinstance(hc["model"], str) and hc["model"]
    assert isinstance(hc["nproc"], int) and hc["nproc"] >= 1
