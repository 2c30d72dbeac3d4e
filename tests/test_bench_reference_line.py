"""bench.py's reference arm (the oracle timed on the host cores) prints the
one JSON line the bench contract fixes, for every workload: the keys, the
"impl" tag, an e2e object with no host-device bytes, and a cpu_baseline that
describes the run. These run on the CPU in seconds (bounded samples)."""
import json
import subprocess
import sys
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]
KEYS = {"impl", "metric", "value", "unit", "n_gpus", "steps", "warmup",
        "ms_per_step", "higher_is_better", "scaling", "vs_baseline", "dtype",
        "data", "config", "e2e", "cpu_baseline"}


@pytest.mark.parametrize("workload", ["w1", "w4", "kda1", "bwd1", "bwd1f"])
def test_reference_line(workload):
    r = subprocess.run([sys.executable, str(ROOT / "bench.py"), "--impl",
                        "reference", "--workload", workload, "--steps", "1",
                        "--warmup", "0"], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert KEYS <= set(d), KEYS - set(d)
    assert d["impl"] == "reference" and d["n_gpus"] == 1
    assert d["warmup"] >= 3 and d["steps"] == 1 and d["value"] > 0
    assert d["higher_is_better"] is True and d["vs_baseline"] is None
    assert d["config"]["workload"]
    e2e = d["e2e"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"]
    assert cb["value"] == d["value"]
