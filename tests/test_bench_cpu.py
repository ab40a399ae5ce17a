"""bench.py's host-side bookkeeping, on the CPU: the ncu traffic figures
point at committed profile summaries, the per-step launch count follows the
library's own decode path choice, and the reference arm prints one JSON line
with the contract's keys without touching a GPU."""
import json
import os
import subprocess
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from synth import workloads as W  # noqa: E402


def test_traffic_figures_cite_committed_profiles():
    assert bench.NCU_TRAFFIC, "no traffic figures"
    for workload, (value, source) in bench.NCU_TRAFFIC.items():
        assert value is None or value > 0
        path = source.split(":")[0]
        assert os.path.isfile(os.path.join(ROOT, path)), (workload, path)
        text = open(os.path.join(ROOT, path)).read()
        if value is not None:
            # the summary states the figure bench.py reports
            assert ("%.3e" % value).replace("e+0", "e") in text or ("%.4g" % value) in text, (workload, value)
    assert bench.traffic_of("no such workload") == (None, None)


def test_launch_count_per_decode_step():
    # ssa_decode_step: route (+ plan), attend and merge on the 16-bit path
    assert bench.launches_per_decode_step(W.DECODE_1M) == 3
    # fp32 decode: route + attend rows
    w32 = W.DECODE_1M.with_(dtype=torch.float32)
    assert bench.launches_per_decode_step(w32) == 2


def test_job_throughput_is_the_whole_job():
    # units per rank x ranks / seconds
    assert bench.job_throughput(100, 2.0, 4) == 200.0
    assert bench.max_over_ranks(3.5, 1) == 3.5


def test_reference_arm_json_line_on_the_host():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    res = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"],
                         cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert res.returncode == 0, res.stderr[-2000:]
    line = json.loads(res.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    assert line["config"]["workload"] == "decode_1m"
