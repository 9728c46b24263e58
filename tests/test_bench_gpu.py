"""The benchmark's JSON line on a GPU: every key of its contract, with values
that agree with one another, from one short run of a small square shape."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*extra):
    r = subprocess.run([sys.executable, "bench.py", *extra], cwd=ROOT, capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-3000:]
    return json.loads(lines[0])


@pytest.mark.gpu
def test_bench_line_contract_small_square():
    B, H, N, d = 2, 8, 1000, 64
    line = _run("--shape", "%d,%d,%d,%d,1" % (B, H, N, d), "--steps", "3", "--warmup", "3",
                "--e2e-steps", "3", "--no-sweep", "--cpu-heads", "1")
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "clocks", "e2e", "gpu_launches", "roofline", "cpu_baseline"):
        assert key in line, key
    assert line["n_gpus"] == 1 and line["steps"] == 3 and line["warmup"] == 3
    assert line["higher_is_better"] is True and line["dtype"] == "bf16"
    assert line["config"]["N"] == N and line["config"]["causal"] is True
    assert line["value"] > 0 and line["ms_per_step"] > 0
    # fwd, prep, main, convert per step, plus whatever the L2 flush adds.
    assert line["gpu_launches"] >= 4 * line["steps"]

    rl = line["roofline"]
    assert rl["bound"] == "tensor" and rl["unit"] == "TFLOP/s" and rl["peak"] > 0
    assert rl["frac"] == pytest.approx(rl["achieved"] / rl["peak"], rel=1e-6)
    assert 0 < rl["frac"] < 1.3
    # The same achieved rate against the nominal peak at the sampled clock
    # and against the datasheet figure.
    assert rl["peak_datasheet"] == 2250.0
    assert rl["frac_datasheet"] == pytest.approx(rl["achieved"] / 2250.0, rel=1e-6)
    clk_mhz = line["clocks"]["sm_mhz"] or line["clocks"]["sm_max_mhz"]
    if clk_mhz:
        assert rl["peak_nominal_at_clock"] == pytest.approx(8192 * 152 * clk_mhz * 1e6 / 1e12,
                                                            rel=1e-6)
        assert rl["frac_nominal"] == pytest.approx(rl["achieved"] / rl["peak_nominal_at_clock"],
                                                   rel=1e-6)

    e2e = line["e2e"]
    elems = B * H * N * d
    assert e2e["h2d_bytes_per_step"] == 4 * elems * 2          # Q, K, V, dO (bf16)
    assert e2e["d2h_bytes_per_step"] == 4 * elems * 2 + B * H * N * 4  # O, dQ, dK, dV, lse
    assert 0 < e2e["value"] and e2e["unit"] == line["unit"]
    # The host link measured in the same run, and the bound it sets.
    cg = e2e["copy_gbs"]
    for k in ("h2d", "d2h", "h2d_concurrent", "d2h_concurrent"):
        assert cg[k] > 1.0, (k, cg)
    parts = e2e["bound_parts_ms"]
    assert e2e["bound_ms"] == pytest.approx(max(parts.values()), rel=1e-9)
    assert parts["h2d"] == pytest.approx(
        e2e["h2d_bytes_per_step"] / (cg["h2d_concurrent"] * 1e9) * 1e3, rel=1e-9)
    assert e2e["frac_of_bound"] == pytest.approx(e2e["bound_ms"] / e2e["ms_per_step"], rel=1e-9)

    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["cores"] >= 1 and cb["sample"]

    clk = line["clocks"]
    assert "sm_mhz" in clk and "reasons" in clk


@pytest.mark.gpu
def test_bench_decode_line_is_hbm_bound_and_plausible():
    from io_aware_exact_02_gb300 import synth
    wl = [g for g in synth.GQA_ALL if g.Nq <= 16][0]
    line = _run("--workload", wl.name, "--steps", "3", "--warmup", "3")
    assert line["unit"] == "GB/s" and line["config"]["Nkv"] == wl.Nkv
    rl = line["roofline"]
    assert rl["bound"] == "hbm" and rl["unit"] == "GB/s"
    assert rl["frac"] == pytest.approx(rl["achieved"] / rl["peak"], rel=1e-6)
    # A copy-rate denominator: a little above 1 is possible, far above is not.
    assert 0 < rl["frac"] < 1.3
    assert line["gpu_launches"] >= line["steps"]
