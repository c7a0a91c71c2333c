"""The benchmark's host-side reporting without a GPU: the roofline fractions
(against the measured peak, the larger of that peak and a same-run library
figure, and the nominal ~8 TB/s for the HBM-bound workloads), the config
naming of each kernel mode, and the CPU-oracle baseline entry."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
import gemm_inputs  # noqa: E402

PEAKS = {"hbm_gbs": 6684.5, "bf16_tflops": 1932.6, "bf16_tflops_sustained": 1749.0, "source": "measured"}


def test_tensor_roofline_fractions():
    w = gemm_inputs.WORKLOADS["square8192_bf16"]
    ms = w.flops / 2000e12 * 1e3                       # 2000 TFLOP/s
    r = bench.roofline_of(w, ms, PEAKS, None)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["achieved"] == pytest.approx(2000.0)
    assert r["frac"] == pytest.approx(2000.0 / 1932.6)
    assert "frac_conservative" not in r                # no library figure given
    lib = {"impl": "torch.matmul (cuBLAS)", "value": 2100.0}
    r = bench.roofline_of(w, ms, PEAKS, None, lib)     # the library beats the measured peak
    assert r["frac_conservative"] == pytest.approx(2000.0 / 2100.0)
    assert "library" in r["frac_conservative_of"]
    lib = {"impl": "torch.matmul (cuBLAS)", "value": 1800.0}
    r = bench.roofline_of(w, ms, PEAKS, None, lib)     # the measured peak is the larger
    assert r["frac_conservative"] == pytest.approx(2000.0 / 1932.6)


def test_fp8_peak_is_twice_bf16():
    w = gemm_inputs.WORKLOADS["square8192_e4m3"]
    r = bench.roofline_of(w, w.flops / 3600e12 * 1e3, PEAKS, None)
    assert r["peak"] == pytest.approx(2 * 1932.6)
    assert "nominal FP8" in r["peak_source"]


def test_hbm_roofline_fractions():
    w = gemm_inputs.WORKLOADS["swin4k_proj_f16"]
    ms = w.algorithmic_bytes / 5600e9 * 1e3            # 5.6 TB/s
    r = bench.roofline_of(w, ms, PEAKS, 12345)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["traffic"] == 12345
    assert r["achieved"] == pytest.approx(5600.0)
    assert r["frac"] == pytest.approx(5600.0 / 6684.5)
    assert r["frac_of_nominal_8tbs"] == pytest.approx(5600.0 / 8000.0)
    assert r["algorithmic_bytes_per_launch"] == 99_532_800 + 73_728 + 1_536 + 398_131_200


@pytest.mark.parametrize("mode,pair,bn,tile,name", [
    (1, 0, 128, "128x128x64", "single CTA"),
    (3, 1, 256, "256x256x64", "paired MMA"),
    (6, 1, 512, "256x512x64", "256x512 tiles"),
    (4, 0, 128, "128x128x64", "resident B"),
])
def test_config_names_each_mode(mode, pair, bn, tile, name):
    w = gemm_inputs.WORKLOADS["square8192_bf16"]
    plan = {"block_m": 128, "block_n": bn, "block_k": 64, "stages": 4, "grid": 152, "pair_mma": pair, "mode": mode,
            "group_m": 12}
    c = bench.config_of(w, plan)
    assert c["tile"] == tile and name in c["kernel_mode"]
    assert c["workload"] == "square8192_bf16" and "256 MiB write then a 256 MiB read" in c["l2"]
    assert "a 256 MiB write," in bench.config_of(w, plan, "write")["l2"]


def test_cpu_baseline_entry_small_workload(oracle_mod):
    w = gemm_inputs.WORKLOADS["square256_f16"]
    e = bench.cpu_baseline_entry(w, 0.5)
    assert e["kind"] == "oracle" and e["unit"] == "TFLOP/s" and e["cores"] >= 1
    assert e["extrapolated"] is False                  # 256 rows: the whole product
    assert e["value"] > 0 and "rows 0..255" in e["sample"]
    assert "gbs" not in e


def test_cpu_baseline_entry_hbm_workload_has_bandwidth(oracle_mod):
    w = gemm_inputs.WORKLOADS["swin4k_proj_f16"]
    e = bench.cpu_baseline_entry(w, 0.2)
    assert e["extrapolated"] is True and e["gbs"] > 0
