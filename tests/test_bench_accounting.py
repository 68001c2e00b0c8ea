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


def test_both_arms_build_config_from_the_workload_alone():
    """The GPU arm and the reference arm print one `config` for one workload:
    every line's config comes from the workload builders, which hold no
    kernel choice (tile, stages, grid, raster group)."""
    import re
    import synth
    src = open(bench.__file__).read()
    configs = re.findall(r'"config":\s*([^\n]*)', src)
    assert len(configs) >= 6
    for c in configs:
        assert re.match(r'(workload_config|mx_config|attn_config)\(w(, world(, (args\.epilogue|"none"), args\.cold_l2)?)?\),?$',
                        c.strip()), c
    kernel_keys = {"tile", "stages", "grid_ctas", "group_m"}
    built = [bench.workload_config(w, 1) for w in synth.WORKLOADS.values()]
    built += [bench.workload_config(w, 1) for w in synth.FP8_WORKLOADS.values()]
    built += [bench.mx_config(w, 1) for w in synth.MX_WORKLOADS.values()]
    built += [bench.attn_config(w, 1) for w in synth.ATTN_WORKLOADS.values()]
    assert len(built) >= 14
    for c in built:
        assert not kernel_keys & set(c), c["workload"]
        assert c["parallelism"] == "single GPU", c["workload"]


def test_reference_arm_names_the_cold_l2_protocol():
    """--cold-l2 changes the workload's `l2` entry in both arms alike."""
    import json
    import subprocess
    import sys
    import synth
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "gemm_256", "--cold-l2",
                        "--steps", "1", "--warmup", "0"], cwd=os.path.dirname(os.path.abspath(bench.__file__)),
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads([l for l in r.stdout.splitlines() if l.startswith("{")][-1])
    assert d["config"] == bench.workload_config(synth.WORKLOADS["gemm_256"], 1, "none", True)
    assert d["config"]["l2"].startswith("flushed: 256 MiB")


def test_tensor_peak_burst_or_sustained_by_timed_length():
    peaks = {"bf16_tflops": 1937.8, "bf16_tflops_sustained": 1734.0, "hbm_gbs": 6773.9}
    short, src_short = bench.tensor_peak(peaks, "measured", 0.06)
    long_, src_long = bench.tensor_peak(peaks, "measured", 0.66)
    assert short == 1937.8 and "burst" in src_short
    assert long_ == 1734.0 and "sustained" in src_long
    fp8, src_fp8 = bench.tensor_peak(peaks, "measured", 0.06, fp8=True)
    assert fp8 == 2 * 1937.8 and "fp8/bf16" in src_fp8
    only_burst = {"bf16_tflops": 1900.0, "hbm_gbs": 6800.0}   # no sustained figure: burst
    assert bench.tensor_peak(only_burst, "fallback", 5.0)[0] == 1900.0


def test_decode_workloads_are_hbm_bound_and_larger_than_l2():
    import synth
    peaks = dict(bench.FALLBACK_PEAKS)
    knee = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)   # flop per byte
    for name in ("decode_1x28672x8192", "decode_64x8192x28672", "decode_256x8192x8192"):
        w = synth.WORKLOADS[name]
        ai = bench.gemm_flops(w.M, w.N, w.K) / bench.gemm_bytes(w.M, w.N, w.K)
        assert ai < knee, name
        assert "larger than L2" in bench.workload_config(w)["l2"], name


def test_source_digest_sees_code_not_comments():
    """Stored ncu traffic stays valid across comment and layout edits of the
    kernel sources, and only those: any change of code (a string literal
    included) changes the text the digest is taken over."""
    src = 'int f(int x) {  // add one\n    /* the sum */ return x + 1;\n}\nconst char* s = "a";\n'
    same = 'int f(int x) {\n  return x + 1;   // different comment\n}\n/* block */ const char* s = "a";\n'
    assert bench._code_only(src) == bench._code_only(same)
    assert bench._code_only(src) != bench._code_only(src.replace("x + 1", "x + 2"))
    assert bench._code_only(src) != bench._code_only(src.replace('"a"', '"b"'))
    for kind in ("gemm", "attention"):
        d = bench.kernel_source_digest(kind)
        assert len(d) == 16 and d == bench.kernel_source_digest(kind)


def test_calibration_mode_names_resolve():
    """Every global name the calibration functions use exists in the module
    (they only run on a GPU, so a broken name would otherwise go unseen)."""
    import ast
    import builtins
    tree = ast.parse(open(bench.__file__).read())
    for fn in (n for n in tree.body if isinstance(n, ast.FunctionDef) and n.name in ("sweep_plans", "l2_latency",
                                                                                      "_calib_warm_us")):
        local = {a.arg for a in ast.walk(fn) if isinstance(a, ast.arg)}
        local |= {t.id for t in ast.walk(fn) if isinstance(t, ast.Name) and isinstance(t.ctx, ast.Store)}
        local |= {n.name for n in ast.walk(fn) if isinstance(n, (ast.FunctionDef, ast.Lambda)) and hasattr(n, "name")}
        local |= {a.asname or a.name.split(".")[0] for n in ast.walk(fn) if isinstance(n, (ast.Import, ast.ImportFrom))
                  for a in n.names}
        for name in {t.id for t in ast.walk(fn) if isinstance(t, ast.Name) and isinstance(t.ctx, ast.Load)}:
            assert name in local or hasattr(bench, name) or hasattr(builtins, name), (fn.name, name)
