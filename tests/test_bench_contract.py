"""bench.py's reference arm on CPU: it runs the oracle on a bounded sample of the
chosen workload and prints one JSON line with the fields the throughput contract
needs (no GPU involved)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--config", "tiny",
                        "--steps", "3", "--warmup", "3"], cwd=ROOT, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["steps"] == 3 and d["warmup"] == 3
    assert d["value"] > 0 and d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["config"]["T"] == 64 and d["config"]["workload"].startswith("tiny")


def test_bench_refuses_fewer_than_three_warmup_steps():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--config", "tiny",
                        "--steps", "1", "--warmup", "2"], cwd=ROOT, capture_output=True,
                       text=True, timeout=120)
    assert r.returncode != 0
