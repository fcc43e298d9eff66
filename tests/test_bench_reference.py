"""The bench's reference arm runs on CPU (it times the oracle, as it stands, on
a bounded sample) and prints one JSON line with the contract's keys."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        *args], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    return json.loads(lines[0])


def test_reference_arm_decode_line():
    d = _run("--steps", "1", "--warmup", "0", "--workload", "long")
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["metric"].startswith("q8-KV decode attention")
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]


def test_reference_arm_prefill_line():
    d = _run("--steps", "1", "--warmup", "0", "--workload", "prefill")
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["cpu_baseline"]["value"] == d["value"]
