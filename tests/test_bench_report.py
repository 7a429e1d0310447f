"""Host logic of the benchmark's roofline report (no GPU): the dominant
kernel's fraction is algorithmic bytes per launch over the measured launch
time against the measured HBM copy rate; an FP64 sweep also carries its FP64
issue-rate fraction against the measured probe rate, and ``binding`` names
the larger; the blocked FP32 row's modelled DRAM traffic follows its tiling."""
from __future__ import annotations

import math

import bench


def test_roofline_is_hbm_fraction_with_fp64_beside_it():
    r = bench.rows()["diffuse_fp64"]
    r["launches"] = bench.DIFF_STEPS
    sweep = {"ms": 0.5 * bench.DIFF_STEPS}          # 0.5 ms per launch
    roof = bench.roofline(r, "diffuse_fp64", sweep, 6800.0, "measured", {"fp64_fma": 0.5})
    bytes_per_launch = 2 * bench.DIFF_N ** 2 * 8
    assert roof["bound"] == "hbm" and roof["unit"] == "GB/s"
    assert math.isclose(roof["achieved"], bytes_per_launch / 0.5e-3 / 1e9, rel_tol=1e-4)
    assert math.isclose(roof["frac"], roof["achieved"] / 6800.0, rel_tol=1e-3)
    fp = roof["fp64"]
    cells = (bench.DIFF_N - 2) ** 2
    ops = bench.FP64_INSTR["diffuse_fp64"] * cells / 0.5e-3 / 1e12
    assert math.isclose(fp["achieved"], ops, rel_tol=1e-3)
    assert math.isclose(fp["frac"], ops / 0.5, rel_tol=1e-3)
    assert roof["binding"] == ("fp64" if fp["frac"] > roof["frac"] else "hbm")


def test_roofline_without_probe_rate_keeps_hbm_only():
    r = bench.rows()["pack_x"]
    roof = bench.roofline(r, "pack_x", {"ms": 0.2}, 6800.0, "measured", {})
    assert "fp64" not in roof and roof["binding"] == "hbm"
    assert math.isclose(roof["frac"], r["bytes"] / 0.2e-3 / 1e9 / 6800.0, rel_tol=1e-3)


def test_blocked_traffic_model():
    t = bench.blocked_traffic(10.0, 6800.0)
    tiles = math.ceil(8192 / 112) * math.ceil(8192 / 64)
    # 199 steps in blocks of 8: 25 launches (odd, as the 200-step parity needs)
    expect = 25 * tiles * (128 * 80 + 112 * 64) * 4 + 2 * 8192 * 8192 * 4
    assert t["dram_bytes_model"] == expect
    assert math.isclose(t["frac_hbm_dram_model"], expect / 10e-3 / 1e9 / 6800.0, rel_tol=1e-3)
