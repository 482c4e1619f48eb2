"""bench.py end to end on the GPU: one short run of the default arm prints one
JSON line carrying every key of the benchmark contract, with consistent
values (the roofline fraction is achieved / peak, the kernel runs no faster
than its own launch allows, the end-to-end copies are counted)."""
import json
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _line(args):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                         timeout=900, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-3000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout[-3000:]
    return json.loads(lines[0])


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def test_default_arm_prints_the_contract_line():
    d = _line(["--workload", "llama1b_attn_out_swiglu", "--steps", "5", "--warmup", "3", "--sustained-s", "0.3",
               "--cpu-budget", "1"])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 5 and d["warmup"] == 3 and d["higher_is_better"] is True
    assert d["config"]["workload"] == "llama1b_attn_out_swiglu" and d["value"] > 0
    r = d["roofline"]
    for k in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert k in r, k
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    assert r["achieved"] >= d["value"] * 0.999  # one launch is the whole step here
    c = d["cpu_baseline"]
    assert c["kind"] == "oracle" and c["cores"] >= 1 and c["value"] > 0 and c["sample"]
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    w_bytes = 8192 * 2048 * 2  # X and R in, bf16
    assert e["h2d_bytes_per_step"] == 2 * w_bytes
    assert d["gpu_launches"] == d["steps"]  # one launch per step for this block
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]
