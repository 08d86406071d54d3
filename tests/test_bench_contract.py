"""bench.py prints one JSON line with the contract's keys: the reference arm
(the fp64 oracle on host cores) on CPU, the GPU arm on a small workload."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, timeout=600):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                         capture_output=True, text=True, timeout=timeout)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.strip().splitlines() if l.strip()]
    assert len(lines) == 1, out.stdout
    return json.loads(lines[0])


def test_reference_arm_json_line():
    d = _run(["--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "3",
              "--ref-step-s", "0.2"])
    assert d["impl"] == "reference"
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["value"] > 0 and d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]


def test_warmup_below_three_is_rejected():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--warmup", "2"], cwd=ROOT,
                         capture_output=True, text=True, timeout=120)
    assert out.returncode != 0


@pytest.mark.gpu
def test_gpu_arm_json_line():
    d = _run(["--workload", "tiny", "--steps", "3", "--warmup", "3"])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "roofline",
              "cpu_baseline", "clocks", "e2e", "gpu_launches"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3 and d["dtype"] == "bf16"
    assert d["value"] > 0 and d["gpu_launches"] >= 3 * 4
    r = d["roofline"]
    # bound by whichever of its algorithmic bytes and FLOPs takes longer at peak
    assert (r["bound"], r["unit"]) in (("tensor", "TFLOP/s"), ("hbm", "GB/s")) and r["peak"] > 0
    assert r["flops_per_launch"] > 0 and r["algorithmic_bytes_per_launch"] > 0
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"])
    assert d["e2e"]["h2d_bytes_per_step"] > 0 and d["e2e"]["d2h_bytes_per_step"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]


def test_algorithmic_bytes_follow_the_launch_decomposition():
    """The bytes bench.py's roofline charges each GEMM kind, on the 16K SFT
    step (one 4,096-row block x one slab per launch, the planner's dH
    k-splits): W read once per launch, D written / read once, h rows once per
    slab, dW written once per row block and read back on the later ones."""
    sys.path.insert(0, ROOT)
    import bench
    from chunked_lm_head_gb300 import _lib
    N, nv, H, V = 16384, 16380, 4096, 151936
    b = bench.algorithmic_bytes_step(N, nv, H, V, 4096, nv)
    splits = _lib.flce_backward_plan(N, H, V, 4096)["dh_splits"]
    assert splits > 1
    W, D, h = V * H * 2, nv * V * 2, nv * H * 2
    assert b["fwd_logits_lse"] == 4 * W + h
    assert b["bwd_dlogits"] == 4 * W + h + D
    assert b["bwd_dH"] == D + 4 * W + nv * H * 4 * splits  # k-splits of fp32 partials, one slab
    assert b["bwd_dW"] == D + h + 4 * V * H * 4 + 3 * V * H * 4
    # dW per launch: D + h + the fp32 write, plus the read on 3 of 4 blocks
    assert b["bwd_dW"] / 4 == pytest.approx(5.634e9, rel=1e-3)
