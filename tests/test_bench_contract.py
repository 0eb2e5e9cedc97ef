"""bench.py's library arm prints one JSON line with every field of its
contract: throughput, roofline of the dominant kernel (with the recorded DRAM
traffic when it matches the source), end-to-end through host memory, clocks,
launch count, and the oracle baseline."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.gpu


def test_bench_line_has_the_contract_fields():
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "3", "--warmup", "3",
           "--no-fused", "--no-checkpoints"]
    res = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, res.stdout
    rec = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "e2e", "clocks", "gpu_launches", "cpu_baseline"):
        assert key in rec, key
    assert rec["n_gpus"] == 1 and rec["steps"] == 3 and rec["warmup"] == 3
    assert rec["value"] > 0 and rec["higher_is_better"] is True
    assert "workload" in rec["config"]
    roof = rec["roofline"]
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in roof, key
    assert 0 < roof["frac"] < 1.5
    e2e = rec["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert rec["gpu_launches"] >= 3  # at least one library kernel per timed step
    cpu = rec["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["value"] > 0
    assert rec["decode"]["roofline"]["frac"] > 0 and rec["decode_tokens"]["roofline"]["frac"] > 0
    assert rec["clocks"]["samples"] >= 10  # the soak keeps the sampler under load
    for leg in ("prefill_w2", "prefill_w3"):  # the long-context workloads, split across SMs
        r = rec[leg]
        assert r["value"] > 0 and "workload" in r
        assert 0 < r["roofline"]["frac"] < 1.5 and r["roofline"]["bound"] == "hbm"
        assert r["gpu_launches"] >= 3
    assert rec["prefill_w3"]["cpu_baseline"]["kind"] == "oracle"
