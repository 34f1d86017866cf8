"""bench.py --impl reference (the CPU oracle timed on the host cores) keeps
the JSON-line contract: one line with impl "reference", the metric, a
tokens/s value, a cpu_baseline describing the run (kind, cores, sample, its
value equal to the line's) and an e2e entry with no host-device bytes.  Run on
the small fp32 workload, where the sample is the whole batch."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny_fp32", "--steps", "2",
                          "--warmup", "3"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    j = json.loads(lines[0])
    assert j["impl"] == "reference" and j["unit"] == "tokens/s" and j["higher_is_better"] is True
    assert j["steps"] == 2 and j["warmup"] == 3 and j["n_gpus"] == 1
    assert j["value"] > 0 and j["ms_per_step"] > 0
    cb = j["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and "first 64 of 64 tokens" in cb["sample"]
    assert cb["value"] == j["value"]
    assert j["e2e"] == {"value": j["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert j["config"]["workload"] == "tiny_fp32" and j["vs_baseline"] is None
