"""Host-side arithmetic of bench.py: the prefill roofline fractions against the
measured block-scaled rate, and the reference arm's line describing the same
workload (config dict) as the GPU arm."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
import synth  # noqa: E402


def test_tensor_roofline_fractions():
    roof = {"bound": "tensor", "achieved": 2000.0, "down_gemm": {"achieved": 1500.0}, "layer_tflops": 1600.0,
            "kernel_sm_mhz": 1500.0}
    peak = {"sustained_tflops": 3600.0, "sustained_sm_mhz": 1500.0, "burst_tflops": 4400.0, "burst_sm_mhz": 1800.0,
            "cycles_per_mma": 128.0}
    P = {"bf16_tflops": 1750.0}
    r = bench.tensor_roofline(roof, peak, P)
    assert r["peak"] == 3600.0 and r["frac"] == pytest.approx(2000 / 3600)
    assert r["frac_vs_burst_peak"] == pytest.approx(2000 / 4400)
    # the instruction's rate at the kernel's clock: burst rate scaled by clock
    assert r["peak_at_kernel_clock"] == pytest.approx(4400 * 1500 / 1800)
    assert r["frac_at_kernel_clock"] == pytest.approx(2000 / (4400 * 1500 / 1800))
    assert r["frac_vs_2x_bf16_burst"] == pytest.approx(2000 / 3500)
    assert r["down_gemm"]["frac"] == pytest.approx(1500 / 3600)
    assert r["layer_frac"] == pytest.approx(1600 / 3600)
    assert "kernel_sm_mhz" in r and "sustained" in r["peak_source"]


def test_headline_is_the_largest_workload_and_reference_arm_shares_its_config():
    args = type("A", (), dict(config="all", experts=None, tokens=None, act_scale="e8m0", weights="mxfp4"))()
    cfg = bench.headline_config(args)
    assert cfg.name == "pro-prefill-skew"
    biggest = max(synth.CONFIGS.values(), key=lambda c: c.T * c.H * c.I * c.E)
    assert cfg.name == biggest.name
    # the reference arm's line on a small workload carries exactly the GPU arm's config dict
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "toy",
                        "--steps", "1", "--warmup", "0", "--ref-budget", "0.5"], capture_output=True, text=True,
                       timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    args.config = "toy"
    assert line["config"] == bench.config_dict(synth.CONFIGS["toy"], args)
    assert line["impl"] == "reference" and line["e2e"]["value"] == line["value"]
