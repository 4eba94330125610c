"""bench.py's output contract, checked on the CPU through its reference arm (the oracle timed on
the host cores): one JSON line with the keys the round's bench line must carry, and a refusal of
fewer than 3 warm-up steps."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
        "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e")


def _bench(*args):
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                          timeout=900, cwd=ROOT)


def test_reference_arm_prints_one_contract_line():
    out = _bench("--impl", "reference", "--steps", "1", "--warmup", "3")
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    j = json.loads(lines[0])
    for k in KEYS:
        assert k in j, k
    assert j["impl"] == "reference" and j["steps"] == 1 and j["warmup"] == 3 and j["n_gpus"] == 1
    assert j["value"] > 0 and j["higher_is_better"] is True and j["unit"] == "tokens/s"
    assert j["cpu_baseline"]["kind"] == "oracle" and j["cpu_baseline"]["value"] == j["value"]
    assert j["cpu_baseline"]["cores"] >= 1 and j["cpu_baseline"]["sample"]
    assert j["e2e"] == {"value": j["value"], "unit": j["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert "workload" in j["config"] and "model" not in j["config"]


def test_fewer_than_three_warmup_steps_are_refused():
    out = _bench("--impl", "reference", "--steps", "1", "--warmup", "2")
    assert out.returncode != 0 and "warmup" in out.stderr
