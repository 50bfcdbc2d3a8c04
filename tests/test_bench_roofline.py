"""The benchmark's roofline bookkeeping, on the CPU: the machine-readable
blocks of the committed ncu summaries parse, the DRAM traffic they give scales
with a launch's algorithmic bytes and goes null once the kernel code differs,
and the roofline fields are the stated ratios (algorithmic work over CUDA-event
time, over the peak of the bound)."""

import os
import re
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

PEAKS = {"hbm_gbs": 6000.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1600.0, "source": "measured"}


@pytest.fixture
def fixed_peaks(monkeypatch):
    monkeypatch.setattr(bench, "_PEAKS", dict(PEAKS))


def _block(name):
    text = open(os.path.join(ROOT, "profiles", name), encoding="utf-8").read()
    sha = re.search(r"^kernel_code_sha256: ([0-9a-f]{64})$", text, re.M).group(1)
    dram = int(re.search(r"^dram_bytes_per_launch: (\d+)$", text, re.M).group(1))
    alg = int(re.search(r"^alg_bytes_per_launch: (\d+)$", text, re.M).group(1))
    return sha, dram, alg


@pytest.mark.parametrize("workload", sorted(bench.TRAFFIC_PROFILES))
def test_profile_blocks_parse_and_are_plausible(workload):
    name = bench.TRAFFIC_PROFILES[workload]
    sha, dram, alg = _block(name)
    # ncu flushes the caches before a captured launch: every algorithmic byte
    # comes from DRAM at least once, and a capture far above it would be a
    # wrong kernel or a wrong algorithmic count.
    assert 1.0 <= dram / alg <= 1.2
    # the command in the summary runs the named workload
    text = open(os.path.join(ROOT, "profiles", name), encoding="utf-8").read()
    if workload != "s518":
        assert f"--workload {workload}" in text
    assert "--clock-control none" in text


@pytest.mark.parametrize("workload", sorted(bench.TRAFFIC_PROFILES))
def test_traffic_scales_with_algorithmic_bytes(workload, monkeypatch):
    sha, dram, alg = _block(bench.TRAFFIC_PROFILES[workload])
    monkeypatch.setattr(bench, "kernel_code_hash", lambda path: sha)
    assert bench.profiled_traffic(alg, workload) == pytest.approx(dram)
    assert bench.profiled_traffic(2 * alg, workload) == pytest.approx(2 * dram)


def test_traffic_is_null_for_stale_code_or_unknown_workload(monkeypatch):
    monkeypatch.setattr(bench, "kernel_code_hash", lambda path: "0" * 64)
    for workload in bench.TRAFFIC_PROFILES:
        assert bench.profiled_traffic(1e8, workload) is None
    assert bench.profiled_traffic(1e8, "no-such-workload") is None


def test_code_hash_ignores_comments_and_blank_lines(tmp_path):
    a = tmp_path / "a.cu"
    b = tmp_path / "b.cu"
    a.write_text("int f() {\n  return 1;\n}\n")
    b.write_text("// header\nint f() {  /* body\n spans */\n\n  return 1;  // one\n}\n")
    assert bench.kernel_code_hash(str(a)) == bench.kernel_code_hash(str(b))
    b.write_text("int f() {\n  return 2;\n}\n")
    assert bench.kernel_code_hash(str(a)) != bench.kernel_code_hash(str(b))


def test_bound_follows_the_ridge_point(fixed_peaks):
    ridge = PEAKS["bf16_tflops"] * 1e3 / PEAKS["hbm_gbs"]       # flop per byte
    assert bench.roof_bound(1.01 * ridge * 1e6, 1e6) == "tensor"
    assert bench.roof_bound(0.99 * ridge * 1e6, 1e6) == "hbm"
    # the two benchmark geometries at their late frames (visible K/V once + Q in + O out)
    def work(nq, nkv, H=16, D=64):
        return 4.0 * nq * nkv * H * D, 2.0 * nkv * H * D * 2 + 2.0 * nq * H * D * 2
    assert bench.roof_bound(*work(1005, 84216)) == "tensor"
    assert bench.roof_bound(*work(262, 19632)) == "hbm"


def test_roofline_fields_are_the_stated_ratios(fixed_peaks):
    flops, nbytes, ms, launches, step_ms = 4.0e12, 2.0e9, 4.0, 10, 5.0
    r = bench.attn_roofline("tensor", flops, nbytes, ms, launches, step_ms, "k", traffic=3.0e8)
    assert r["achieved"] == pytest.approx(flops / (ms / 1e3) / 1e12)
    assert r["frac"] == pytest.approx(r["achieved"] / PEAKS["bf16_tflops"])
    assert r["frac_sustained"] == pytest.approx(r["achieved"] / PEAKS["bf16_tflops_sustained"])
    roof_s = max(flops / (PEAKS["bf16_tflops"] * 1e12), nbytes / (PEAKS["hbm_gbs"] * 1e9))
    assert r["step_frac"] == pytest.approx(roof_s / (step_ms / 1e3))
    assert r["launch_ms"] == pytest.approx(ms / launches)
    assert r["flops_per_launch"] == pytest.approx(flops / launches)
    assert r["traffic"] == 3.0e8 and r["unit"] == "TFLOP/s"
    h = bench.attn_roofline("hbm", flops, nbytes, ms, launches, step_ms, "k")
    assert h["unit"] == "GB/s" and h["traffic"] is None
    assert h["achieved"] == pytest.approx(nbytes / (ms / 1e3) / 1e9)
    assert h["frac"] == pytest.approx(h["achieved"] / PEAKS["hbm_gbs"])
    assert h["frac_sustained"] is None


def test_compact_line_keeps_the_roofline_headline(fixed_peaks):
    roof = bench.attn_roofline("hbm", 1e12, 1e9, 2.0, 4, 3.0, "k", traffic=1.03e9)
    roof["outside_attn_ms_per_step"] = 0.1
    roof["launch_shape"] = {"q_tiles": 1, "splits": 3}
    line = {"metric": "m", "value": 1.0, "unit": "frames/s", "steps": 2, "ms_per_step": 1.5,
            "config": {"workload": "w"}, "roofline": roof, "gpu_launches": 12, "clocks": None}
    c = bench.compact(line)
    for k in ("bound", "achieved", "peak", "unit", "frac", "traffic", "launch_ms", "launch_shape"):
        assert c["roofline"][k] == roof[k]
    assert c["workload"] == "w" and c["gpu_launches"] == 12
