"""The bench's flop and byte accounting, pinned by the arithmetic the pages
print (HipKittens "L2" detail page, §4 "Roofline placement" and "% peak
derivation"; values in tests/golden/pages_figures.json with citations)."""
import json
import os

import bench

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "pages_figures.json")


def fig():
    with open(GOLDEN) as f:
        return json.load(f)


def test_arithmetic_intensity_8192():
    g = fig()["ai_bf16_gemm_8192"]
    ai = bench.gemm_flops(g["M"], g["N"], g["K"]) / bench.gemm_bytes(g["M"], g["N"], g["K"])
    assert round(ai) == g["flop_per_byte"]


def test_flops_per_k_step():
    g = fig()["flops_per_k_step_256x256x64"]
    f = bench.gemm_flops(g["tile_m"], g["tile_n"], g["k_step"])
    assert abs(f - g["flops"]) / g["flops"] < 1e-3


def test_percent_of_peak_and_knee():
    g = fig()["pct_peak_hk_bf16_8192"]
    assert round(100 * g["tflops"] / g["peak_tflops"], 1) == g["pct"]
    k = fig()["roofline_knee_mi355x"]
    assert round(k["peak_tflops"] / k["hbm_tbs"]) == k["knee_flop_per_byte"]


def test_workload_config_names_the_shape():
    import synth
    c = bench.workload_config(synth.WORKLOADS["gemm_8192"])
    assert c["workload"] == "gemm_8192" and (c["M"], c["N"], c["K"]) == (8192, 8192, 8192)
    assert "larger than L2" in c["l2"]
