"""The bench's reference arm needs no GPU: `bench.py --impl reference` times the CPU oracle on a bounded token
sample and prints one JSON line with the fields of the bench contract (run here on the tiny chunk)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                        "--warmup", "1", "--config", "tiny"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    j = json.loads(lines[0])
    assert j["impl"] == "reference"
    assert j["metric"] == "routed token-expert pairs/s per MoE layer" and j["unit"] == "pairs/s"
    assert j["value"] > 0 and j["higher_is_better"] is True and j["n_gpus"] == 1
    assert j["steps"] == 2 and j["warmup"] == 1 and j["ms_per_step"] > 0
    assert j["config"]["workload"].startswith("tiny:")
    assert j["cpu_baseline"]["kind"] == "oracle" and j["cpu_baseline"]["cores"] >= 1
    assert j["cpu_baseline"]["value"] == j["value"]
    assert j["e2e"] == {"value": j["value"], "unit": "pairs/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    # a step is a token sample of the chunk, and the line says so
    assert j["step"]["kind"] == "bounded token sample of the chunk" and j["step"]["chunk_pairs"] == 64 * 2
