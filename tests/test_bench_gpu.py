"""bench.py on the GPU: one JSON line with every key of the benchmark contract, on the tiny workload."""
import json
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(*extra):
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "tiny", "--steps", "5", "--warmup", "3",
           "--e2e-steps", "2", "--cpu-seconds", "0.5", "--chain-steps", "2", *extra]
    out = subprocess.run(cmd, capture_output=True, text=True, cwd=ROOT, timeout=600)
    assert out.returncode == 0, out.stderr[-3000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout[-3000:]
    return json.loads(lines[0])


def check_contract(d, launches_per_step):
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 5 and d["warmup"] == 3 and d["higher_is_better"] is True
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["scaling"] == "weak" and d["vs_baseline"] is None
    assert d["config"]["workload"].startswith("tiny")
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    c = d["cpu_baseline"]
    assert c["kind"] == "oracle" and c["cores"] == 1 and c["value"] > 0 and c["sample"]
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] == 2 * 3 * 786_432 and e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] == 5 * launches_per_step
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(d["clocks"])


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def test_bench_line_pingpong():
    d = run_bench()
    check_contract(d, 1)
    assert d["inplace_step"]["launches_per_step"] == 2 and d["unfused_chain"]["ms_per_step"] > 0
    # a plan this small keeps register staging; the other staging is timed beside it
    assert d["staging"] == "registers" and d["other_staging"]["staging"] == "bulk"
    assert d["other_staging"]["ms_per_step"] > 0
    o = d["bucketed_overlap"]
    assert o["serial_ms"] > 0 and o["overlapped_ms"] > 0
    for cap in ("16", "152"):
        assert o["block_budget_sweep"][cap]["step_alone_ms"] > 0 and o["block_budget_sweep"][cap]["overlapped_ms"] > 0


def test_bench_line_second_workload():
    """The second workload (the default command's 1.3B key, here the GPT-2 shapes) is timed on its own buffers and
    reported under its own key, with its roofline, the other staging and the no-allocation step beside it."""
    d = run_bench("--second", "gpt2")
    check_contract(d, 1)
    s = d["workload_gpt2"]
    assert s["config"]["workload"].startswith("gpt2") and s["value"] > 0 and s["ms_per_step"] > 0
    assert s["config"]["staging"] == "bulk" and s["other_staging"]["staging"] == "registers"
    r = s["roofline"]
    assert r["bound"] == "hbm" and abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    assert s["noalloc_step"]["ms_per_step"] > 0 and s["noalloc_step"]["zr_step_ms_per_step"] > 0
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(s["clocks"])


def test_bench_line_in_place():
    d = run_bench("--inplace")
    check_contract(d, 2)
    assert "one set" in d["config"]["state_dtype"] and d["config"]["alg_bytes_per_param"] == 4 * 3 + 26
