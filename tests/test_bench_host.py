"""Host logic of bench.py, checked against hand-worked values: which kernel
each workload's default plans launch (the names its HBM / ALU rooflines and
DRAM traffic are filed under), the algorithmic bytes of the spreading and
interpolation kernels (minimum traffic per launch), and the multiply-add
count of the ALU roofline."""
import json
import os
import re

import pytest

import bench
import nonuniform_fft_gb300 as nf
from nonuniform_fft_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "nonuniform_fft_gb300", "csrc")

# default plans: (type 1 method, type 2 method, tile3d, igroup) -> kernels
DEFAULTS = {
    "2d_t1_f32_N64_M1e4": ((nf.METHOD_REGTILE, 0, 1, 0), {"spread": "spread_regtile2d_kernel"}),
    "2d_f32_N1024_M1e7": ((nf.METHOD_REGTILE, nf.METHOD_SM, 1, 0),
                          {"spread": "spread_regtile2d_kernel", "interp": "interp_sm_kernel"}),
    "2d_t1_f32_N1024_M1e7_cluster": ((nf.METHOD_REGTILE, 0, 1, 0), {"spread": "spread_regtile2d_kernel"}),
    "3d_f32_N128_M3.2e7": ((nf.METHOD_REGTILE, nf.METHOD_SM, 2, 2),
                           {"spread": "spread_slab3d_kernel", "interp": "interp_group3d_kernel"}),
    "3d_f64_N64_M1e7_mix": ((nf.METHOD_REGTILE, nf.METHOD_SM, 1, 0),
                            {"spread": "spread_plane3d_df_kernel", "interp": "interp_sm3d_df_kernel"}),
    "1d_f64_N1e6_M1e7": ((nf.METHOD_REGTILE, nf.METHOD_SM, 1, 0),
                         {"spread": "spread_reg1d_df_kernel", "interp": "interp_sm1d_df_kernel"}),
}


def _kernel_names_in_sources():
    names = set()
    for f in os.listdir(CSRC):
        if f.endswith((".cu", ".cuh")):
            text = open(os.path.join(CSRC, f)).read()
            for m in re.finditer(r"__global__\s+void\s+(?:__launch_bounds__\([^)]*\)\s+)?(\w+)\s*\(", text):
                names.add(m.group(1))
    return names


@pytest.mark.parametrize("name", sorted(DEFAULTS))
def test_kernel_names_of_default_plans(name):
    (m1, m2, tile3d, igroup), want = DEFAULTS[name]
    wl = W.WORKLOADS[name]
    got = bench.kernel_names(wl, m1, m2, tile3d, igroup)
    for key, kernel in want.items():
        assert got[key] == kernel
        assert kernel in _kernel_names_in_sources(), kernel


def test_traffic_entries_name_kernels_the_plans_launch():
    """profiles/traffic.json files DRAM bytes under the kernels of each
    workload's default plans (the names the bench line looks up)."""
    traffic = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    assert set(traffic) == set(DEFAULTS)
    for name, entries in traffic.items():
        assert set(entries) == set(DEFAULTS[name][1].values()), name


def test_algorithmic_bytes_hand_worked():
    # 2D bench workload: M = 1e7 float points (2 coordinates + a 4-byte index),
    # complex64 strengths / results, fine grid 2048^2 complex64
    wl = W.WORKLOADS["2d_f32_N1024_M1e7"]
    b = bench.algorithmic_bytes(wl, (2048, 2048))
    assert b["spread"] == 10_000_000 * (8 + 4) + 10_000_000 * 8 + 2 * 2048 * 2048 * 8 == 267_108_864
    assert b["interp"] == 10_000_000 * (8 + 4) + 2048 * 2048 * 8 + 10_000_000 * 8 == 233_554_432
    # 3D single precision: M = 3.2e7, fine grid 256^3
    wl = W.WORKLOADS["3d_f32_N128_M3.2e7"]
    b = bench.algorithmic_bytes(wl, (256, 256, 256))
    assert b["spread"] == 32_000_000 * 16 + 32_000_000 * 8 + 2 * 256 ** 3 * 8 == 1_036_435_456
    assert b["interp"] == 32_000_000 * 16 + 256 ** 3 * 8 + 32_000_000 * 8 == 902_217_728
    # batched launch of 4 vectors: the points once, strengths and grid per vector
    wl = W.WORKLOADS["2d_f32_N1024_M1e7"]
    b4 = bench.algorithmic_bytes(wl, (2048, 2048), 4)
    assert b4["spread"] == 10_000_000 * 12 + 4 * (10_000_000 * 8 + 2 * 2048 * 2048 * 8)


def test_alu_roofline_counts():
    # 2 w^d real multiply-adds per point: 3D single precision w = 7, M = 3.2e7
    wl = W.WORKLOADS["3d_f32_N128_M3.2e7"]
    r = bench.alu_roofline(wl, 7, 1.0)
    assert r["algorithmic_fma_per_launch"] == 2 * 7 ** 3 * 32_000_000
    assert r["peak"] == pytest.approx(128 * 152 * 2.07e9 / 1e12)
    assert r["achieved"] == pytest.approx(2 * 343 * 32e6 / 1e-3 / 1e12)
    # double precision is measured against the nominal FP64 multiply-add rate
    r = bench.alu_roofline(W.WORKLOADS["3d_f64_N64_M1e7_mix"], 13, 1.0)
    assert r["peak"] == pytest.approx(0.625)
