"""The benchmark's reference arm (the oracle timed on the host cores) keeps its JSON
contract: the GPU arm's metric, unit and workload config, a cpu_baseline describing the
run, and an end-to-end block with no host-device traffic.  Each of its steps is the
oracle's repair of the whole declared chunk, so its time and token rate describe that
workload."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=600, check=True)
    line = json.loads(out.stdout.strip().splitlines()[-1])
    sys.path.insert(0, ROOT)
    import bench
    assert line["impl"] == "reference"
    assert line["metric"] == bench.METRIC and line["unit"] == "GB/s" and line["higher_is_better"] is True
    assert line["config"] == bench.repair_config(1)
    assert line["steps"] == 1 and line["warmup"] == 3 and line["value"] > 0
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1 and cb["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert cb["cpu_model"] and cb["nproc"] >= 1
    # the value, the step time and the token rate all describe the whole 32-layer chunk
    cfg = bench.synth.REPAIR_LLAMA8B
    by = bench.repair_bytes(cfg)
    sec = line["ms_per_step"] / 1e3
    assert abs(line["tokens_per_s"] - cfg.tokens / sec) <= 1e-3 * line["tokens_per_s"] + 1.0
    assert abs(line["value"] - by["corrected"] / sec / 1e9) <= 1e-3 * line["value"] + 1e-3
    assert "32 layers" in cb["sample"]
