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
    """bench.py quotes a kernel's DRAM traffic from its profile summary only while the
    kernel's source still has the hash recorded beside it."""
    import hashlib
    csrc = tmp_path / "average_pooling_stencil_gb300" / "csrc"
    prof = tmp_path / "profiles"
    csrc.mkdir(parents=True)
    prof.mkdir()
    src = csrc / "k.cu"
    src.write_text("__global__ void k() {}\n")
    sha = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    (prof / "k.md").write_text(f"source_sha256_16: {sha}\ntraffic_bytes_per_launch: 1.25e+09\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_from_profile("k.cu", "k.md") == pytest.approx(1.25e9)
    src.write_text("__global__ void k() { }\n")            # the kernel changed
    assert bench.traffic_from_profile("k.cu", "k.md") is None
    assert bench.traffic_from_profile("k.cu", "missing.md") is None
