"""bench.py's roofline arithmetic on the host: each bound's achieved rate,
peak and fraction against values worked out by hand from the same inputs."""
import os
import sys
from types import SimpleNamespace

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402

PEAKS = {"hbm_gbs": 6780.7, "sm_max_mhz": 2070.0, "tf32_measured": 1000.0,
         "fma_measured": {"scalar": 68.0, "packed": 76.0}}


def case(**kw):
    base = dict(bytes=143_258_816, flops=1_417_052_160, bound="hbm", tensor_passes=0,
                precision=0)
    base.update(kw)
    return SimpleNamespace(**base)


def test_hbm_bound_fraction_is_bytes_over_time_over_peak():
    t = 44.0e-6
    r = bench.roofline_for(case(), t, PEAKS, "measured", 2070.0)
    gbs = 143_258_816 / t / 1e9                     # 3255.9 GB/s
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(gbs)
    assert r["frac"] == pytest.approx(gbs / 6780.7)
    assert "tensor_tflops" not in r                 # no tensor work on this path


@pytest.mark.parametrize("passes", [1, 3])
def test_tensor_work_counts_every_mma_pass(passes):
    t = 44.0e-6
    r = bench.roofline_for(case(tensor_passes=passes), t, PEAKS, "measured", 2070.0)
    work = 1_417_052_160 * passes / t / 1e12        # 3xTF32: three products per FLOP pair
    assert r["tensor_tflops"] == pytest.approx(work)
    assert r["tensor_frac_of_ceiling"] == pytest.approx(work / 1000.0)
    assert r["frac"] == pytest.approx(143_258_816 / t / 1e9 / 6780.7)   # still HBM


def test_alu_bound_against_unit_count_peak_and_measured_ceiling():
    t = 1.7e-3
    flops = 85_899_345_920
    r = bench.roofline_for(case(bound="alu", flops=flops), t, PEAKS, "measured", 2070.0)
    peak = 152 * 128 * 2 * 2070e6 / 1e12            # 80.55 TFLOP/s
    assert r["unit"] == "TFLOP/s"
    assert r["peak"] == pytest.approx(peak)
    assert r["frac"] == pytest.approx(flops / t / 1e12 / peak)
    assert r["frac_of_measured_ceiling"] == pytest.approx(flops / t / 1e12 / 76.0)


def test_mixed_bound_takes_the_larger_floor():
    t = 50.0e-6
    hbm_floor = 143_258_816 / 6780.7e9
    # FLOPs chosen so that the FP32 floor is the larger one
    flops = int(1.5 * hbm_floor * 80.5e12)
    r = bench.roofline_for(case(bound="hbm+alu", flops=flops), t, PEAKS, "measured", 2070.0)
    fp32_floor = flops / (152 * 128 * 2 * 2070e6)
    assert fp32_floor > hbm_floor
    assert r["bound"] == "alu"
    assert r["frac"] == pytest.approx(fp32_floor / t)


def test_profile_traffic_is_used_only_for_the_profiled_source(tmp_path, monkeypatch):
    """bench.py quotes a kernel's DRAM traffic per workload from its profile summary only
    while the kernel's source still has the hash recorded beside it."""
    import hashlib
    csrc = tmp_path / "average_pooling_stencil_gb300" / "csrc"
    prof = tmp_path / "profiles"
    csrc.mkdir(parents=True)
    prof.mkdir()
    src = csrc / "k.cu"
    src.write_text("__global__ void k() {}\n")
    sha = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    (prof / "k.md").write_text(f"source_sha256_16: {sha}\n"
                               "traffic_bytes_per_launch[wa]: 1.25e+09\n"
                               "traffic_bytes_per_launch[wb]: 3.5e8\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_from_profile("k.cu", "k.md", "wa") == pytest.approx(1.25e9)
    assert bench.traffic_from_profile("k.cu", "k.md", "wb") == pytest.approx(3.5e8)
    assert bench.traffic_from_profile("k.cu", "k.md", "wc") is None
    src.write_text("__global__ void k() { }\n")            # the kernel changed
    assert bench.traffic_from_profile("k.cu", "k.md", "wa") == "stale"
    assert bench.traffic_from_profile("k.cu", "missing.md", "wa") is None


def test_every_measured_workload_names_a_kernel_source_and_profile():
    csrc = os.path.join(ROOT, "average_pooling_stencil_gb300", "csrc")
    for key, cfg, prec, mode in bench.PER_CONFIG:
        if mode == "graph":
            continue                      # launch-latency bound: no traffic figure
        src, _ = bench.PROFILE_OF[key]
        assert os.path.exists(os.path.join(csrc, src)), key


def test_compact_json_round_trips_and_keeps_the_per_config_block_short():
    import json
    v = {"a": 442600000000.0, "b": [1610000000.0, 2.5], "c": 1234567.0, "d": 12345678.9,
         "e": 8589934592, "f": 194987777516.0, "g": None, "h": "x1.0,2"}
    s = bench.compact_json(v)
    assert json.loads(s) == v
    assert "4.426e11" in s and " " not in s.replace("x1.0,2", "")
    per = {}
    for key, cfg, prec, mode in bench.PER_CONFIG:
        c = SimpleNamespace(bytes=1_611_000_000, flops=85_899_345_920, outputs=134_234_112,
                            bound="alu" if prec == 3 else "hbm",
                            tensor_passes={0: 3, 1: 1, 2: 3, 3: 0}[prec])
        per[key] = bench.per_config_entry(key, c, 303.3e-6, PEAKS, "measured", 2.1e7)
    per["_cols"] = bench.PER_CONFIG_COLS
    per["_peaks"] = {"hbm_GB_s": 6780.7, "fp32_TF_s": 80.55, "fp32_meas_TF_s": 75.9,
                     "tf32_gemm_TF_s": 1066.0}
    per["_cpu"] = {"model": "Neoverse-V2", "threads": 16, "fused_tiny_1thread_s": 0.006503,
                   "fused_tiny_1thread_out_s": 7750000.0}
    per["_fused_us_after_flush"] = 42.63
    # the driver keeps the last 1500 characters of the output; the whole block, and the
    # line's closing braces, must fit in it
    assert len(bench.compact_json({"per_config": per})) < 1450
    assert all(len(v) == len(bench.PER_CONFIG_COLS) for k, v in per.items() if k[0] != "_")


def test_both_arms_print_the_same_config():
    from average_pooling_stencil_gb300 import workloads
    wl = workloads.get(bench.HEADLINE_CFG)
    a, b = bench.line_config(wl, 1), bench.line_config(wl, 1)
    assert a == b and set(a) == {"workload", "seed", "l2", "parallelism"}
    assert a["workload"] == "avgpool3d k3 s2 p1 count_include_pad x[16x32x128x128x256] fp32"
    assert "avgpool3d k2 s2 p0 count_include_pad x" in bench.workload_desc(workloads.get(9))
    assert "count_include_pad=False" in bench.workload_desc(workloads.get(8))
