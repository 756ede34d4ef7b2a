"""bench.py's JSON line: the keys and types the measurement contract fixes,
for the reference arm (the oracle on the host cores, no GPU) and for the
CUDA arm (GPU)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, timeout):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                       timeout=timeout, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


BASE_KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
             "vs_baseline", "dtype", "data", "config", "e2e"}


def test_reference_arm_line():
    d = _run(["--impl", "reference", "--workload", "linear_4096", "--steps", "1", "--warmup", "3",
              "--ref-rows", "16"], timeout=600)
    assert BASE_KEYS <= set(d)
    assert d["impl"] == "reference" and d["warmup"] >= 3 and d["steps"] == 1
    assert d["value"] > 0 and d["higher_is_better"] is True and d["config"]["workload"] == "linear_4096"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


@pytest.mark.gpu
def test_cuda_arm_line():
    d = _run(["--workload", "linear_4096", "--steps", "2", "--warmup", "3", "--no-cpu-baseline"], timeout=900)
    assert BASE_KEYS <= set(d)
    assert d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] == 3 and d["value"] > 0
    assert d["config"]["workload"] == "linear_4096" and "l2" in d["config"]
    roof = d["roofline"]
    assert roof["bound"] in ("tensor", "hbm") and roof["unit"] in ("TFLOP/s", "GB/s")
    assert roof["achieved"] > 0 and roof["peak"] > 0 and abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 1e-3
    assert "traffic" in roof
    e2e = d["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] > 0
    # per layer and step: 5 forward kernels (the one-launch activation
    # quantization with the outliers on, subB, widening, plan, GEMM) and 2 of
    # the fused backward (the GEMM, which reduces grad_bias from the fp16
    # grad_output itself, and the grad_bias finalize)
    assert d["gpu_launches"] == d["steps"] * 7
    assert d["step_ms"]["best"] <= d["step_ms"]["median"] <= d["step_ms"]["worst"]
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(d["clocks"])
    assert d["per_layer"] and d["per_layer"][0]["fwd_tops"] > 0
    assert d["cuda_graph"]["ms_per_step"] > 0 and d["nf4_weight_only"]["value"] > 0


@pytest.mark.gpu
def test_token_sharded_mode_line():
    """--shard tokens at one rank: the colmax / all-reduce / from-colmax
    forward gives the unsharded forward's bits, and the line reports the
    exchange."""
    d = _run(["--shard", "tokens", "--workload", "linear_4096", "--steps", "3", "--warmup", "3"], timeout=600)
    assert {"metric", "value", "unit", "n_gpus", "steps", "ms_per_step", "scaling", "config"} <= set(d)
    assert d["scaling"] == "strong" and d["n_gpus"] == 1 and d["value"] > 0
    assert d["bit_identical_to_unsharded"] is True
    assert d["config"]["rows_per_rank"] == [2048]
    assert d["exchange"]["bytes_per_step"] == 4 * 4096 and 0 <= d["exchange"]["share"] < 0.05
