"""bench.py's JSON line on a GPU: one line with the contract's keys, run on small cases
(prefill-sized runs are the bench's own job)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

KEYS = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
        "vs_baseline", "dtype", "data", "config", "roofline", "gpu_launches", "e2e", "clocks")


def run(*args):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    r = subprocess.run([sys.executable, "bench.py", *args], cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    return lines[0]


@pytest.mark.parametrize("extra", [[], ["--graph", "10"], ["--op", "split", "--graph", "10"],
                                   ["--mxfp8", "ceil"], ["--op", "post_int8"]])
def test_bench_line_has_the_contract_keys(extra):
    d = run("--workload", "decode_verify", "--steps", "20", "--warmup", "3", "--no-cpu-baseline", *extra)
    for k in KEYS:
        assert k in d, k
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["gpu_launches"] > 0
    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["peak"] > 0 and 0 < rf["frac"] < 1.2
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert d["config"]["T"] == 6 and d["config"]["H"] == 7168
    sp = d["main_span_us"]
    assert sp["calls"] >= 3 and 0 < sp["p10"] <= sp["p50"] <= sp["p90"]


def test_bench_cpu_baseline_leg():
    d = run("--workload", "tiny", "--steps", "5", "--warmup", "3")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["cores"] >= 1 and cb["sample"]
