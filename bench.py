"""Benchmark of the GB300 BF16 GEMM (C = A·Bᵀ, bf16 in, fp32 accumulate, bf16 out).

One step = one GEMM of the workload (default: the 8192³ headline shape of the
HipKittens "L2" detail page, §2 Q3 and §5 Tab. 2) through the C-ABI
``hk_gemm_bf16``. Prints ONE JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl hk|reference]
                    [--workload NAME] [--no-cpu-baseline]
    python bench.py --calibrate plans [--shapes MxNxK ...]   # plan sweep
    python bench.py --calibrate l2                           # L2 latency probe

With N > 1 (launched by torchrun) every rank runs an independent replica of
the workload on its own GPU (the GEMM has no exchange step); the reported
value is the sum of all ranks' work over the slowest rank's time.

``--impl reference`` times the CPU oracle (the only reference this method has)
on a bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "BF16 GEMM TFLOPS at 1 GB300 and % of dense-BF16 tensor peak"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}

# DRAM traffic of one launch of the GEMM kernel from an ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum), valid only for the kernel
# sources whose digest is given (the code of those sources, comments and
# layout excluded).
MEASURED_TRAFFIC = {
    "gemm_8192": {"source_digest": "cb16790c5d83d15d", "bytes_per_launch": 1069123584 + 126451968},
    # inputs smaller than L2 (warm): DRAM traffic is below the algorithmic bytes
    "gemm_4096": {"source_digest": "cb16790c5d83d15d", "bytes_per_launch": 81972736 + 13856256},
    "skinny_128x28672x8192": {"source_digest": "cb16790c5d83d15d", "bytes_per_launch": 471965184 + 3204864},
    "fp8_gemm_8192": {"source_digest": "cb16790c5d83d15d", "bytes_per_launch": 344409600 + 115722240},
    # the block-scaled GEMM kernel alone (the scale arrangement kernel moves ~8 MB more)
    "mxfp8_gemm_8192": {"source_digest": "cb16790c5d83d15d", "bytes_per_launch": 359903744 + 117093888},
    # the GEMM kernel alone (the split-K reduction reads the fp32 partials and writes C)
    "decode_64x8192x28672": {"source_digest": "cb16790c5d83d15d", "bytes_per_launch": 473511680 + 3490560},
    # one launch, no K split (the 256x112 pair): B read once, A and C
    "decode_256x8192x8192": {"source_digest": "cb16790c5d83d15d", "bytes_per_launch": 138511360 + 3212288},
    # attention: captured at B2 (one launch); the B16 figure scales it by 8 (traffic grows with B)
    "attn_gqa_b2_s4096_d128": {"source_digest": "89f7a7a6da310d8d", "bytes_per_launch": 199923456 + 110883584},
    "attn_gqa_b16_s4096_d128": {"source_digest": "89f7a7a6da310d8d", "bytes_per_launch": 8 * (199923456 + 110883584)},
    # D = 64 captured at the bench's own size (one launch)
    "attn_gqa_b16_s4096_d64": {"source_digest": "89f7a7a6da310d8d", "bytes_per_launch": 2865444352 + 548965888},
}


KERNEL_SOURCES = {
    "gemm": ("gemm_kernel.cuh", "ptx.cuh", "hk_gemm.cu"),
    "attention": ("attn_kernel.cuh", "ptx.cuh", "hk_attention.cu", "host_internal.h"),
}


def _code_only(text: str) -> str:
    """C/C++ source without comments and with whitespace runs collapsed: two
    sources that differ only in comments or layout compile to the same code."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_digest(kind: str = "gemm") -> str:
    """Digest of the code of the sources one kernel is built from, comments
    and layout excluded (a stored ncu traffic figure is valid only while that
    code is unchanged)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "dense_bf16_gemm_02_gb300", "csrc")
    for f in KERNEL_SOURCES[kind]:
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            h.update(f.encode() + b"\0" + _code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def gemm_flops(M: int, N: int, K: int) -> float:
    """Algorithmic flops of one GEMM: one multiply and one add per (i, j, k)."""
    return 2.0 * M * N * K


def gemm_bytes(M: int, N: int, K: int) -> float:
    """Algorithmic bytes: read A and B once, write C once, bf16."""
    return 2.0 * (M * K + N * K + M * N)


SUSTAINED_AFTER_S = 0.5   # timed regions at least this long run under the power cap


def tensor_peak(peaks: dict, src: str, timed_s: float, fp8: bool = False) -> tuple[float, str]:
    """The dense tensor peak a kernel is compared with: the measured burst
    figure for a short timed region, the sustained (power-capped) one once
    back-to-back launches run for SUSTAINED_AFTER_S or longer. FP8 takes the
    bf16 figure times the nominal FP8/BF16 ratio of 2."""
    key = "bf16_tflops_sustained" if timed_s >= SUSTAINED_AFTER_S and "bf16_tflops_sustained" in peaks else "bf16_tflops"
    kind = "sustained" if key.endswith("sustained") else "burst"
    scale, note = (2.0, " × 2 (nominal fp8/bf16 ratio)") if fp8 else (1.0, "")
    return float(peaks[key]) * scale, f"{key} ({kind}, timed region {timed_s:.2f} s) of {src}{note}"


def load_peaks() -> tuple[dict, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            peaks = json.load(f)
        if "bf16_tflops" in peaks:
            return peaks, "measured"
    except (OSError, ValueError):
        pass
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------- clocks --

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons in a side process;
    each line is stamped with the host time it arrived."""

    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_index: int, interval_ms: int = 20):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={','.join(self.FIELDS)}",
                 "--format=csv,noheader,nounits", "-lms", str(interval_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == len(self.FIELDS):
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float) -> dict:
        inside = [s for t, s in self.samples if t0 <= t <= t1]
        window = "timed"
        if not inside:
            # timed region shorter than the sampling interval: nearest samples
            inside = [s for t, s in self.samples if t0 - 0.5 <= t <= t1 + 0.5]
            window = "timed±0.5s"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(s[0]) for s in inside if num(s[0]) is not None]
        smax = [num(s[1]) for s in inside if num(s[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for s in inside for n, v in zip(names, s[4:8]) if v.lower() == "active"})
        power = [num(s[2]) for s in inside if num(s[2]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(inside), "window": window,
                "power_w_max": max(power) if power else None}


# ------------------------------------------------------- distributed --

def dist_setup(gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def replica_value(flops_per_step: float, steps: int, world: int, elapsed_ms_max: float) -> float:
    """Whole-job TFLOP/s of `world` independent replicas that each ran `steps`
    GEMMs: the flops of all ranks over the slowest rank's time."""
    return flops_per_step * steps * world / (elapsed_ms_max / 1e3) / 1e12


def max_over_ranks(world, x: float) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------- CPU oracle --

ALL_WORKLOADS = {**synth.WORKLOADS, **synth.FP8_WORKLOADS}


def is_fp8(w) -> bool:
    return w.name in synth.FP8_WORKLOADS


def operands_of(w):
    return synth.operands_fp8(w) if is_fp8(w) else synth.operands(w)


def oracle_rows_timed(A, B, rows, with_values: bool = False):
    """Time the oracle on full rows of C; returns (seconds, threads used[, the rows' bf16 bits])."""
    import oracle
    t0 = time.perf_counter()
    if A.dtype == np.uint8:      # FP8 operands: full rows as entries
        N = B.shape[0]
        rr = np.repeat(np.asarray(rows, dtype=np.int64), N)
        cc = np.tile(np.arange(N, dtype=np.int64), len(rows))
        sa, sb = synth.FP8_SCALES
        vals = oracle.gemm_fp8_entries(A, B, rr, cc, sa, sb).reshape(len(rows), N)
        used = os.cpu_count() or 1
    else:
        vals, used = oracle.gemm_rows(A, B, rows)
    dt = time.perf_counter() - t0
    return (dt, used, vals) if with_values else (dt, used)


def oracle_entries_timed(A, B, rows, cols):
    """Time the oracle on single entries of C; returns (seconds, the entries' bf16 bits)."""
    import oracle
    t0 = time.perf_counter()
    if A.dtype == np.uint8:
        sa, sb = synth.FP8_SCALES
        vals = oracle.gemm_fp8_entries(A, B, rows, cols, sa, sb)
    else:
        vals, _ = oracle.gemm_entries(A, B, rows, cols)
    return time.perf_counter() - t0, vals


def parity_tolerance(ref_bits: np.ndarray, K: int, sigma_ab: float) -> np.ndarray:
    """Per-entry bound |C_gpu − C_ref| ≤ 2⁻⁷·|C_ref| + 2⁻¹²·√K·σ_A·σ_B
    (σ_A·σ_B = ``sigma_ab``, the generator's nominal standard deviations, times
    the FP8 scales where they apply): one bf16 ulp of the value for a
    rounding-boundary flip, plus fp32 cancellation near 0."""
    ref = synth.bf16_bits_to_f32(ref_bits).astype(np.float64)
    return 2.0 ** -7 * np.abs(ref) + 2.0 ** -12 * np.sqrt(max(K, 1)) * sigma_ab


def cpu_baseline(w, A, B, C_gpu=None, budget_s: float = 15.0):
    """The oracle, as it stands, on full rows of this workload's C plus 1024
    seeded single entries (tile edges included). The rows and entries it
    computes are then compared with the GPU's C of the timed run (``C_gpu``,
    host bf16 bits), entry by entry within the parity tolerance: a miss fails
    the bench. Returns (the baseline, the check or None)."""
    probe = np.arange(min(64, w.M), dtype=np.int64)   # enough rows to occupy every host core
    t, _ = oracle_rows_timed(A, B, probe)
    per_row = max(t / len(probe), 1e-6)
    nrows = int(max(1, min(w.M, budget_s / per_row)))
    rows = np.arange(nrows, dtype=np.int64)
    t, used, row_vals = oracle_rows_timed(A, B, rows, with_values=True)
    er, ec = synth.sample_positions(w.M, w.N, 3000 + w.wid, count=1024)
    te, ent_vals = oracle_entries_timed(A, B, er, ec)
    tflops = (gemm_flops(nrows, w.N, w.K) + gemm_flops(len(er), 1, w.K)) / (t + te) / 1e12
    base = {"value": tflops, "unit": UNIT, "cores": used, "kind": "oracle",
            "sample": f"rows 0..{nrows - 1} of C ({nrows}x{w.N}x{w.K}) and {len(er)} seeded entries "
                      f"(tile edges included), fp64 C oracle, {t + te:.1f} s"}
    if C_gpu is None:
        return base, None
    got = np.concatenate([C_gpu[:nrows].ravel(), C_gpu[er, ec]])
    ref = np.concatenate([row_vals.ravel(), ent_vals])
    sigma_ab = float(np.prod(synth.FP8_SCALES)) if is_fp8(w) else w.scale * w.scale
    err = np.abs(synth.bf16_bits_to_f32(got).astype(np.float64) - synth.bf16_bits_to_f32(ref).astype(np.float64))
    tol = parity_tolerance(ref, w.K, sigma_ab)
    bad = ~(err <= tol)
    check = {"entries": int(got.size), "full_rows": nrows, "sampled_entries": int(len(er)), "misses": int(bad.sum()),
             "max_err_over_tol": float(np.max(err / tol)),
             "tolerance": "2^-7·|C_ref| + 2^-12·sqrt(K)·σ_A·σ_B per entry, against the fp64 oracle"}
    if bad.any():
        raise RuntimeError(f"parity check of the timed run's C against the oracle failed: {check}")
    return base, check


def run_reference(args, w):
    """Reference arm: the CPU oracle on a bounded sample per step."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    A, B = operands_of(w)
    probe = np.arange(min(64, w.M), dtype=np.int64)
    t, _ = oracle_rows_timed(A, B, probe)
    per_row = max(t / len(probe), 1e-6)
    rows_per_step = int(max(1, min(64, 120.0 / (args.steps + args.warmup) / per_row)))
    rows = np.arange(rows_per_step, dtype=np.int64)
    for _ in range(args.warmup):
        oracle_rows_timed(A, B, rows)
    total = 0.0
    used = 0
    for _ in range(args.steps):
        dt, used = oracle_rows_timed(A, B, rows)
        total += dt
    value = gemm_flops(rows_per_step, w.N, w.K) * args.steps / total / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(w, world, "none", args.cold_l2),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": used, "kind": "oracle",
                         "sample": f"{rows_per_step} full rows of C per step ({rows_per_step}x{w.N}x{w.K})"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def parallelism(world: int) -> str:
    return "replicas" if world > 1 else "single GPU"


L2_FLUSH_BYTES = 256 << 20   # written before each timed launch with --cold-l2 (GB300 L2: 126 MiB)


def workload_config(w, world: int = 1, epilogue: str = "none", cold_l2: bool = False) -> dict:
    """The workload as both arms name it (the kernel's own choices go under
    the line's `kernel_config`, so that the two arms' configs are equal)."""
    elem = 1 if is_fp8(w) else 2
    cfg = {"workload": w.name, "M": w.M, "N": w.N, "K": w.K,
           "layout": "A MxK row-major, B NxK row-major, C MxN row-major (C = A·Bᵀ)",
           "values": f"N(0,1)·{w.scale} rounded to {'E4M3' if elem == 1 else 'bf16'}, "
                     f"seeds {1000 + w.wid}/{2000 + w.wid}",
           "l2": ("flushed: %d MiB written before each timed launch, outside its two events"
                  % (L2_FLUSH_BYTES >> 20)) if cold_l2 else
                 "no flush: inputs larger than L2 (A+B = %d MiB > 126 MiB)" % ((w.M + w.N) * w.K * elem >> 20)
                 if (w.M + w.N) * w.K * elem > 126 << 20 else "inputs smaller than L2 (warm L2)",
           "accumulate": "fp32", "output": "bf16", "parallelism": parallelism(world), "epilogue": epilogue}
    if elem == 1:
        cfg["scales"] = list(synth.FP8_SCALES)
    return cfg


# Pause before a timed block. The GPU's clock depends on its recent load (it
# runs faster for a while after a pause than under continuous work; measured
# at 8192^3: whichever of two kernels is timed first after a 2 s pause reads
# 10-15 % higher), so our timed region and the library's context block both
# start after the same warm-up and the same pause.
TIMED_PAUSE_S = 0.3


def time_library(call, dev, warmup: int, n: int) -> float:
    """Mean ms per call of `call`, under the protocol of our timed region:
    `warmup` calls, a TIMED_PAUSE_S pause, then `n` back-to-back calls
    between CUDA events on the current stream."""
    import torch
    for _ in range(max(3, warmup)):
        call()
    torch.cuda.synchronize(dev)
    time.sleep(TIMED_PAUSE_S)
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0.record()
    for _ in range(n):
        call()
    c1.record()
    torch.cuda.synchronize(dev)
    return c0.elapsed_time(c1) / n


def time_cold(call, flush, stream, n: int) -> list:
    """Durations (ms) of `n` calls of `call` on `stream`, each after `flush`
    (a buffer larger than L2) is overwritten and timed alone between its own
    two CUDA events, so that no call finds its operands in L2."""
    import torch
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * n)]
    with torch.cuda.stream(stream):
        for i in range(n):
            flush.fill_(i & 0x7F)
            ev[2 * i].record(stream)
            call()
            ev[2 * i + 1].record(stream)
    torch.cuda.synchronize()
    return [ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(n)]


def launch_spread(call, stream, n: int) -> list:
    """Durations (ms) of `n` launches of `call` with an event between each, for
    the spread (p10/p90) of launch times. Taken after the timed region, not in
    it: an event between two launches keeps the second from starting early as
    a programmatic dependent of the first, which slows back-to-back steps."""
    import torch
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
    with torch.cuda.stream(stream):
        ev[0].record(stream)
        for i in range(n):
            call()
            ev[i + 1].record(stream)
    torch.cuda.synchronize()
    return [ev[i].elapsed_time(ev[i + 1]) for i in range(n)]


# ---------------------------------------------------------------- GPU arm --

def run_hk(args, w):
    import torch

    world, rank, local = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import dense_bf16_gemm_02_gb300 as hk

    fp8 = is_fp8(w)
    A_bits, B_bits = operands_of(w)
    if fp8:
        A = torch.from_numpy(A_bits).to(dev)
        B = torch.from_numpy(B_bits).to(dev)
    else:
        A = torch.from_numpy(A_bits.view(np.int16)).to(dev).view(torch.bfloat16)
        B = torch.from_numpy(B_bits.view(np.int16)).to(dev).view(torch.bfloat16)
    C = torch.empty((w.M, w.N), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.Stream(device=dev)
    sh = int(stream.cuda_stream)
    sa, sb = synth.FP8_SCALES
    # decode-regime workloads run through a plan that may split K (with a workspace);
    # the others through the one-shot call, which never splits
    decode = w.name.startswith("decode_")
    plan = hk.Plan(w.M, w.N, w.K, device=local, group_m=args.group_m, split_k=0 if decode else 1,
                   input_type=hk.HK_INPUT_E4M3 if fp8 else hk.HK_INPUT_BF16, alpha=sa * sb if fp8 else 0.0)
    info = plan.info()
    ws_bytes = plan.workspace_size
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev) if decode else None
    flops = gemm_flops(w.M, w.N, w.K)

    act = {"none": 0, "bias": 0, "bias_relu": 1, "bias_gelu": 2, "bias_silu": 3}[args.epilogue]
    bias_t = None
    if args.epilogue != "none":
        bias_bits = synth.normal_bf16(1, w.N, 4000 + w.wid, 1.0)[0]
        bias_t = torch.from_numpy(bias_bits.view(np.int16)).to(dev)

    def step():
        if fp8:
            st = hk.hk_gemm_fp8_e4m3(A.data_ptr(), B.data_ptr(), C.data_ptr(), w.M, w.N, w.K, w.K, w.K, w.N, sa, sb,
                                     sh)
            if st != hk.HK_OK:
                raise hk.HKError(st, "hk_gemm_fp8_e4m3")
            return
        if bias_t is not None:
            st = hk.hk_gemm_bf16_epilogue(A.data_ptr(), B.data_ptr(), C.data_ptr(), bias_t.data_ptr(), w.M, w.N,
                                          w.K, w.K, w.K, w.N, act, sh)
            if st != hk.HK_OK:
                raise hk.HKError(st, "hk_gemm_bf16_epilogue")
            return
        if decode:
            st = plan.run_raw(A.data_ptr(), B.data_ptr(), C.data_ptr(), ws.data_ptr(), ws_bytes, sh)
            where = "hk_gemm_plan_run"
        elif args.group_m:
            # an explicit schedule goes through a plan (hk_gemm_plan_run)
            st = plan.run_raw(A.data_ptr(), B.data_ptr(), C.data_ptr(), 0, 0, sh)
            where = "hk_gemm_plan_run"
        else:
            st = hk.hk_gemm_bf16(A.data_ptr(), B.data_ptr(), C.data_ptr(), w.M, w.N, w.K, w.K, w.K, w.N, sh)
            where = "hk_gemm_bf16"
        if st != hk.HK_OK:
            raise hk.HKError(st, where)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize(dev)
    if hk.hk_gemm_last_device_status(local) != hk.HK_OK:
        raise RuntimeError("device status after warm-up: " + hk.hk_gemm_last_error_string())

    # ---- device-resident timed region: K back-to-back launches between two events
    # (--cold-l2: each launch after a write of a buffer larger than L2, timed alone)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev) if args.cold_l2 else None
    events = [torch.cuda.Event(enable_timing=True) for _ in range(2)]   # the timed region's two ends
    sampler = ClockSampler(local) if rank == 0 else None
    time.sleep(TIMED_PAUSE_S)   # (also lets the clock sampler start)
    barrier(world)
    torch.cuda.synchronize(dev)
    t_host0 = time.time()
    cold_ms = None
    if flush is not None:
        cold_ms = time_cold(step, flush, stream, args.steps)
    else:
        with torch.cuda.stream(stream):
            events[0].record(stream)
            for i in range(args.steps):
                step()
            events[1].record(stream)
    torch.cuda.synchronize(dev)
    t_host1 = time.time()
    barrier(world)
    elapsed_ms = sum(cold_ms) if cold_ms is not None else events[0].elapsed_time(events[1])
    if hk.hk_gemm_last_device_status(local) != hk.HK_OK:
        raise RuntimeError("device status after timing: " + hk.hk_gemm_last_error_string())
    clocks = None
    if sampler:
        time.sleep(0.15)
        sampler.stop()
        clocks = sampler.summary(t_host0, t_host1)
    # per-launch spread, outside the timed region (cold: the timed launches themselves)
    per_launch = cold_ms if cold_ms is not None else launch_spread(step, stream, min(args.steps, 20))
    elapsed_max = max_over_ranks(world, elapsed_ms)

    # ---- end to end: pinned host inputs -> device -> GEMM -> host result.
    # Steps are independent GEMMs, so they are pipelined on three streams:
    # the H2D copy of step i+1 and the D2H copy of step i-1 overlap the GEMM
    # of step i; device operands are double-buffered.
    if fp8:
        A_h = torch.from_numpy(A_bits).pin_memory()
        B_h = torch.from_numpy(B_bits).pin_memory()
    else:
        A_h = torch.from_numpy(A_bits.view(np.int16)).view(torch.bfloat16).pin_memory()
        B_h = torch.from_numpy(B_bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    C_h = [torch.empty((w.M, w.N), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    A_d = [A, torch.empty_like(A)]
    B_d = [B, torch.empty_like(B)]
    C_d = [C, torch.empty_like(C)]
    s_h2d, s_d2h = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    # steady state: the pipeline's fill and drain (one H2D and one D2H not overlapped) amortised over
    # at least 50 steps whatever K is (at 8192^3: 741 TFLOP/s over 20 steps, 764 over 100)
    e2e_steps = min(max(args.steps, 50), 100)

    def e2e_run(n):
        h2d_done = [torch.cuda.Event() for _ in range(2)]
        comp_done = [None, None]
        d2h_done = [None, None]
        for i in range(n):
            k = i & 1
            if comp_done[k] is not None:
                s_h2d.wait_event(comp_done[k])      # the GEMM that read slot k is finished
            with torch.cuda.stream(s_h2d):
                A_d[k].copy_(A_h, non_blocking=True)
                B_d[k].copy_(B_h, non_blocking=True)
                h2d_done[k].record(s_h2d)
            stream.wait_event(h2d_done[k])
            if d2h_done[k] is not None:
                stream.wait_event(d2h_done[k])      # C of slot k has been copied out
            if fp8:
                st = hk.hk_gemm_fp8_e4m3(A_d[k].data_ptr(), B_d[k].data_ptr(), C_d[k].data_ptr(), w.M, w.N, w.K,
                                         w.K, w.K, w.N, sa, sb, sh)
            elif decode:
                st = plan.run_raw(A_d[k].data_ptr(), B_d[k].data_ptr(), C_d[k].data_ptr(), ws.data_ptr(), ws_bytes, sh)
            else:
                st = hk.hk_gemm_bf16(A_d[k].data_ptr(), B_d[k].data_ptr(), C_d[k].data_ptr(), w.M, w.N, w.K, w.K,
                                     w.K, w.N, sh)
            if st != hk.HK_OK:
                raise hk.HKError(st, "GEMM")
            comp_done[k] = torch.cuda.Event()
            comp_done[k].record(stream)
            s_d2h.wait_event(comp_done[k])
            with torch.cuda.stream(s_d2h):
                C_h[k].copy_(C_d[k], non_blocking=True)
                d2h_done[k] = torch.cuda.Event()
                d2h_done[k].record(s_d2h)

    e2e_run(2)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    e0.record(s_h2d)
    e2e_run(e2e_steps)
    e1.record(s_d2h)
    torch.cuda.synchronize(dev)
    barrier(world)
    e2e_ms = max_over_ranks(world, e0.elapsed_time(e1))
    if not np.array_equal(C_h[(e2e_steps - 1) & 1].view(torch.int16).numpy()[0, :16].view(np.uint16),
                          C.view(torch.int16).cpu().numpy()[0, :16].view(np.uint16)):
        raise RuntimeError("end-to-end result differs from the device result")
    if hk.hk_gemm_last_device_status(local) != hk.HK_OK:
        raise RuntimeError("device status after the end-to-end run: " + hk.hk_gemm_last_error_string())

    # ---- context only: the vendor library on the same GPU and inputs (outside the timed region)
    cublas = None
    if rank == 0 and not args.no_cublas_context:
        try:
            if fp8:
                A8, B8 = A.view(torch.float8_e4m3fn), B.view(torch.float8_e4m3fn)
                s_a = torch.tensor(sa, dtype=torch.float32, device=dev)
                s_b = torch.tensor(sb, dtype=torch.float32, device=dev)
                lib_call = lambda: torch._scaled_mm(A8, B8.t(), scale_a=s_a, scale_b=s_b, out_dtype=torch.bfloat16)
                what = ("torch._scaled_mm (cuBLASLt FP8) on the same GPU and inputs, timed after ours with the same "
                        "warm-up and pause; context only")
            else:
                lib_call = lambda: torch.matmul(A, B.t(), out=C)
                what = ("torch.matmul (cuBLAS) on the same GPU and inputs, timed after ours with the same warm-up "
                        "and pause; context only")
            n_ctx = max(5, args.steps)   # as many back-to-back calls as our timed region
            if flush is not None:
                for _ in range(max(3, args.warmup)):
                    lib_call()
                torch.cuda.synchronize(dev)
                time.sleep(TIMED_PAUSE_S)
                ms = sum(time_cold(lib_call, flush, torch.cuda.current_stream(dev), n_ctx)) / n_ctx
                what += "; each call after the same L2 flush, timed alone"
            else:
                ms = time_library(lib_call, dev, args.warmup, n_ctx)
            cublas = {"value": flops / (ms / 1e3) / 1e12, "unit": UNIT, "ms_per_gemm": ms, "launches": n_ctx,
                      "what": what}
        except Exception as exc:   # context only: never fails the bench
            cublas = {"unavailable": str(exc)[:200]}

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return 0

    peaks, peaks_src = load_peaks()
    peak, tensor_src = tensor_peak(peaks, peaks_src, elapsed_max / 1e3, fp8)
    value = replica_value(flops, args.steps, world, elapsed_max)
    mean_launch_ms = elapsed_ms / args.steps   # the timed region's mean, back to back
    nbytes = gemm_bytes(w.M, w.N, w.K) if not fp8 else float(w.M * w.K + w.N * w.K + 2 * w.M * w.N)
    hbm_bound = flops / nbytes < peak * 1e12 / (float(peaks["hbm_gbs"]) * 1e9)   # below the roofline knee
    if hbm_bound:
        bound, rf_unit, rf_peak = "hbm", "GB/s", float(peaks["hbm_gbs"])
        achieved = nbytes / (mean_launch_ms / 1e3) / 1e9
        peak_source = f"hbm_gbs of {peaks_src}"
    else:
        bound, rf_unit, rf_peak = "tensor", UNIT, peak
        achieved = flops / (mean_launch_ms / 1e3) / 1e12
        peak_source = tensor_src
    digest = kernel_source_digest()
    traffic = None
    tr = MEASURED_TRAFFIC.get(w.name)
    if tr and tr.get("source_digest") == digest and not args.cold_l2:   # (captured without a flush)
        traffic = tr["bytes_per_launch"]
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3" if fp8 else "bf16", "data": "synthetic",
        "config": workload_config(w, world, args.epilogue, args.cold_l2),
        "kernel_config": {"tile": f"{info['tile_m']}x{info['tile_n']}x{info['tile_k']} per "
                                  f"{'CTA pair' if info['ctas_per_unit'] == 2 else 'CTA'}",
                          "stages": info["stages"], "grid_ctas": info["grid_ctas"], "group_m": info["group_m"]},
        "pct_of_peak": 100.0 * value / world / peak,
        "roofline": {"bound": bound, "achieved": achieved, "peak": rf_peak, "unit": rf_unit,
                     "frac": achieved / rf_peak, "traffic": traffic,
                     "peak_source": peak_source,
                     "algorithmic_flops_per_launch": flops,
                     "algorithmic_bytes_per_launch": nbytes,
                     "mean_launch_ms": mean_launch_ms, "p10_launch_ms": float(np.percentile(per_launch, 10)),
                     "p90_launch_ms": float(np.percentile(per_launch, 90)),
                     "spread_source": "p10/p90: the timed launches, each after an L2 flush" if args.cold_l2 else
                                      "p10/p90: launches timed one by one after the timed region",
                     "kernel": f"gemm_bf16_kernel ({info['tile_m']}x{info['tile_n']}, "
                               f"{info['ctas_per_unit']} CTA(s) per tile)",
                     "source_digest": digest},
        "e2e": {"value": replica_value(flops, e2e_steps, world, e2e_ms), "unit": UNIT,
                "h2d_bytes_per_step": int(A_h.numel() * A_h.element_size() + B_h.numel() * B_h.element_size()),
                "d2h_bytes_per_step": int(C_h[0].numel() * 2), "steps": e2e_steps,
                "pipelined": "H2D(i+1) | GEMM(i) | D2H(i-1) on three streams"},
        "gpu_launches": args.steps * int(info["kernels_per_run"]),
        "clocks": clocks,
        "context_cublas": cublas,
    }
    if not args.no_cpu_baseline:
        C_host = C.view(torch.int16).cpu().numpy().view(np.uint16)   # the device C of the timed steps
        line["cpu_baseline"], line["parity_check"] = cpu_baseline(
            w, A_bits, B_bits, C_host if args.epilogue == "none" else None)
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


# ------------------------------------------------------------- MXFP8 GEMM --

MX_METRIC = "MXFP8 GEMM TFLOPS at 1 GB300 and % of dense-FP8 tensor peak"


def mx_config(w, world: int = 1) -> dict:
    return {"workload": w.name, "M": w.M, "N": w.N, "K": w.K,
            "layout": "A MxK, B NxK E4M3 row-major; SFA Mx(K/32), SFB Nx(K/32) UE8M0; C MxN bf16 (C = A·Bᵀ)",
            "values": f"E4M3 of N(0,1), seeds {1000 + w.wid}/{2000 + w.wid}; scales uniform 2^-3..2^3, "
                      f"seeds {3100 + w.wid}/{3200 + w.wid}",
            "l2": "no flush: inputs larger than L2 (A+B = %d MiB > 126 MiB)" % ((w.M + w.N) * w.K >> 20)
            if (w.M + w.N) * w.K > 126 << 20 else "inputs smaller than L2 (warm L2)",
            "block": 32, "accumulate": "fp32", "output": "bf16", "parallelism": parallelism(world)}


def oracle_mx_rows_timed(A, B, SA, SB, rows, with_values: bool = False):
    import oracle
    N = B.shape[0]
    rr = np.repeat(np.asarray(rows, dtype=np.int64), N)
    cc = np.tile(np.arange(N, dtype=np.int64), len(rows))
    t0 = time.perf_counter()
    vals = oracle.gemm_mxfp8_entries(A, B, SA, SB, rr, cc).reshape(len(rows), N)
    dt = time.perf_counter() - t0
    return (dt, os.cpu_count() or 1, vals) if with_values else (dt, os.cpu_count() or 1)


def mx_parity_check(A, B, SA, SB, rows_ref, C_gpu) -> dict:
    """Rows 0..r-1 of the timed run's C against the oracle's, per entry within
    2^-7·|C_ref| + 2^-16·Σ_b 2^(SA+SB-254)·Σ_{k in b} |A·B| (one bf16 rounding
    plus fp32 accumulation with margin); a miss fails the bench."""
    r = rows_ref.shape[0]
    import torch
    dec = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    dec = np.where(np.isnan(dec), 0.0, dec)
    a = np.abs(dec[A[:r]]) * np.repeat(np.exp2(SA[:r].astype(np.float64) - 127), 32, axis=1)
    b = np.abs(dec[B]) * np.repeat(np.exp2(SB.astype(np.float64) - 127), 32, axis=1)
    mag = a @ b.T
    ref = synth.bf16_bits_to_f32(rows_ref).astype(np.float64)
    got = synth.bf16_bits_to_f32(C_gpu[:r]).astype(np.float64)
    tol = 2.0 ** -7 * np.abs(ref) + 2.0 ** -16 * mag
    err = np.abs(got - ref)
    bad = ~(err <= tol)
    check = {"entries": int(ref.size), "full_rows": r, "misses": int(bad.sum()),
             "max_err_over_tol": float(np.max(err / np.maximum(tol, 1e-300))),
             "tolerance": "2^-7·|C_ref| + 2^-16·Σ_b scale_a·scale_b·Σ|A·B| per entry, against the fp64 oracle"}
    if bad.any():
        raise RuntimeError(f"parity check of the timed run's C against the oracle failed: {check}")
    return check


def run_reference_mx(args, w):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if int(os.environ.get("RANK", "0")) != 0:
        return 0
    A, B, SA, SB = synth.operands_mx(w)
    t, _ = oracle_mx_rows_timed(A, B, SA, SB, [0])
    rows_per_step = int(max(1, min(64, 120.0 / (args.steps + args.warmup) / max(t, 1e-6))))
    rows = np.arange(rows_per_step, dtype=np.int64)
    for _ in range(args.warmup):
        oracle_mx_rows_timed(A, B, SA, SB, rows)
    total, used = 0.0, 0
    for _ in range(args.steps):
        dt, used = oracle_mx_rows_timed(A, B, SA, SB, rows)
        total += dt
    value = gemm_flops(rows_per_step, w.N, w.K) * args.steps / total / 1e12
    print(json.dumps({
        "impl": "reference", "metric": MX_METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": mx_config(w, world),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": used, "kind": "oracle",
                         "sample": f"{rows_per_step} full rows of C per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}), flush=True)
    return 0


def run_mx(args, w):
    import torch

    world, rank, local = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import dense_bf16_gemm_02_gb300 as hk

    Ab, Bb, SAb, SBb = synth.operands_mx(w)
    A, B, SA, SB = (torch.from_numpy(x).to(dev) for x in (Ab, Bb, SAb, SBb))
    C = torch.empty((w.M, w.N), dtype=torch.bfloat16, device=dev)
    nbytes = hk.hk_gemm_mxfp8_workspace_size(w.M, w.N, w.K)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)
    sh = int(stream.cuda_stream)
    flops = gemm_flops(w.M, w.N, w.K)
    kb = w.K // 32

    def launch(a, b, sa, sb, c):
        st = hk.hk_gemm_mxfp8(a.data_ptr(), b.data_ptr(), sa.data_ptr(), sb.data_ptr(), c.data_ptr(), w.M, w.N, w.K,
                              w.K, w.K, kb, kb, w.N, ws.data_ptr(), nbytes, sh)
        if st != hk.HK_OK:
            raise hk.HKError(st, "hk_gemm_mxfp8")

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            launch(A, B, SA, SB, C)
    torch.cuda.synchronize(dev)
    events = [torch.cuda.Event(enable_timing=True) for _ in range(2)]   # the timed region's two ends
    sampler = ClockSampler(local) if rank == 0 else None
    time.sleep(TIMED_PAUSE_S)   # (also lets the clock sampler start)
    barrier(world)
    torch.cuda.synchronize(dev)
    t_host0 = time.time()
    with torch.cuda.stream(stream):
        events[0].record(stream)
        for i in range(args.steps):
            launch(A, B, SA, SB, C)
        events[1].record(stream)
    torch.cuda.synchronize(dev)
    t_host1 = time.time()
    barrier(world)
    elapsed_ms = events[0].elapsed_time(events[1])
    if hk.hk_gemm_last_device_status(local) != hk.HK_OK:
        raise RuntimeError("device status after timing: " + hk.hk_gemm_last_error_string())
    clocks = None
    if sampler:
        time.sleep(0.15)
        sampler.stop()
        clocks = sampler.summary(t_host0, t_host1)
    # per-launch spread, outside the timed region
    per_launch = launch_spread(lambda: launch(A, B, SA, SB, C), stream, min(args.steps, 20))
    elapsed_max = max_over_ranks(world, elapsed_ms)

    # end to end: pinned host A, B, scales -> device -> GEMM -> C to pinned host (three streams)
    hosts = [torch.from_numpy(x).pin_memory() for x in (Ab, Bb, SAb, SBb)]
    devs = [[A, torch.empty_like(A)], [B, torch.empty_like(B)], [SA, torch.empty_like(SA)], [SB, torch.empty_like(SB)]]
    C_d = [C, torch.empty_like(C)]
    C_h = [torch.empty((w.M, w.N), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    s_h2d, s_d2h = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    e2e_steps = max(4, min(args.steps, 30))

    def e2e_run(n):
        h2d_done = [torch.cuda.Event() for _ in range(2)]
        comp_done, d2h_done = [None, None], [None, None]
        for i in range(n):
            k = i & 1
            if comp_done[k] is not None:
                s_h2d.wait_event(comp_done[k])
            with torch.cuda.stream(s_h2d):
                for h, d in zip(hosts, devs):
                    d[k].copy_(h, non_blocking=True)
                h2d_done[k].record(s_h2d)
            stream.wait_event(h2d_done[k])
            if d2h_done[k] is not None:
                stream.wait_event(d2h_done[k])
            launch(devs[0][k], devs[1][k], devs[2][k], devs[3][k], C_d[k])
            comp_done[k] = torch.cuda.Event()
            comp_done[k].record(stream)
            s_d2h.wait_event(comp_done[k])
            with torch.cuda.stream(s_d2h):
                C_h[k].copy_(C_d[k], non_blocking=True)
                d2h_done[k] = torch.cuda.Event()
                d2h_done[k].record(s_d2h)

    e2e_run(2)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    e0.record(s_h2d)
    e2e_run(e2e_steps)
    e1.record(s_d2h)
    torch.cuda.synchronize(dev)
    barrier(world)
    e2e_ms = max_over_ranks(world, e0.elapsed_time(e1))

    ctx = None
    if rank == 0 and not args.no_cublas_context:
        try:   # cuBLASLt block-scaled FP8 through torch, if this torch exposes it
            a8, b8 = A.view(torch.float8_e4m3fn), B.view(torch.float8_e4m3fn)
            sa8, sb8 = SA.view(torch.float8_e8m0fnu), SB.view(torch.float8_e8m0fnu)
            call = lambda: torch._scaled_mm(a8, b8.t(), scale_a=sa8, scale_b=sb8, out_dtype=torch.bfloat16)
            n_ctx = max(5, args.steps)   # as many back-to-back calls as our timed region
            ms = time_library(call, dev, args.warmup, n_ctx)
            ctx = {"value": flops / (ms / 1e3) / 1e12, "unit": UNIT, "ms_per_gemm": ms, "launches": n_ctx,
                   "what": "torch._scaled_mm with e8m0 block scales (cuBLASLt) on the same GPU and inputs, timed after "
                           "ours with the same warm-up and pause; context only"}
        except Exception as exc:
            ctx = {"unavailable": str(exc)[:200]}

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return 0
    peaks, peaks_src = load_peaks()
    peak, peak_source = tensor_peak(peaks, peaks_src, elapsed_max / 1e3, fp8=True)
    value = replica_value(flops, args.steps, world, elapsed_max)
    mean_launch_ms = elapsed_ms / args.steps   # the timed region's mean, back to back
    achieved = flops / (mean_launch_ms / 1e3) / 1e12
    digest = kernel_source_digest("gemm")
    tr = MEASURED_TRAFFIC.get(w.name)
    traffic = tr["bytes_per_launch"] if tr and tr.get("source_digest") == digest else None
    line = {
        "metric": MX_METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed_max / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3 (mx)", "data": "synthetic",
        "config": mx_config(w, world),
        "kernel_config": {"tile": "256x256 per CTA pair (M > 128; 128x192 per CTA otherwise)"},
        "pct_of_peak": 100.0 * value / world / peak,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT, "frac": achieved / peak,
                     "traffic": traffic,
                     "peak_source": peak_source,
                     "algorithmic_flops_per_launch": flops,
                     "algorithmic_bytes_per_launch": float(w.M * w.K + w.N * w.K + (w.M + w.N) * kb + 2 * w.M * w.N),
                     "mean_launch_ms": mean_launch_ms, "p10_launch_ms": float(np.percentile(per_launch, 10)),
                     "p90_launch_ms": float(np.percentile(per_launch, 90)),
                     "spread_source": "p10/p90: launches timed one by one after the timed region",
                     "kernel": ("mx_scale_blocks_kernel + gemm_bf16_kernel<2, 256, fp8, mx>" if w.M > 128 else "mx_scale_blocks_kernel + gemm_bf16_kernel<1, 192, fp8, mx>"), "source_digest": digest},
        "e2e": {"value": replica_value(flops, e2e_steps, world, e2e_ms), "unit": UNIT,
                "h2d_bytes_per_step": int(sum(h.numel() for h in hosts)), "d2h_bytes_per_step": int(C_h[0].numel() * 2),
                "steps": e2e_steps, "pipelined": "H2D(i+1) | GEMM(i) | D2H(i-1) on three streams"},
        "gpu_launches": args.steps * 2,
        "clocks": clocks,
        "context_cublaslt": ctx,
    }
    if not args.no_cpu_baseline:
        t, used = oracle_mx_rows_timed(Ab, Bb, SAb, SBb, np.arange(2))
        rows = int(max(1, min(w.M, 15.0 / max(t / 2, 1e-6))))
        t, used, ref_rows = oracle_mx_rows_timed(Ab, Bb, SAb, SBb, np.arange(rows), with_values=True)
        line["cpu_baseline"] = {"value": gemm_flops(rows, w.N, w.K) / t / 1e12, "unit": UNIT, "cores": used,
                                "kind": "oracle", "sample": f"rows 0..{rows - 1} of C (fp64 C oracle, {t:.1f} s)"}
        line["parity_check"] = mx_parity_check(Ab, Bb, SAb, SBb, ref_rows,
                                               C.view(torch.int16).cpu().numpy().view(np.uint16))
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


# ------------------------------------------------- attention forward --

ATTN_METRIC = "GQA attention forward TFLOPS at 1 GB300 and % of dense-BF16 tensor peak"


def attn_flops(w) -> float:
    """Algorithmic flops of one attention forward: Q·Kᵀ and P·V, 2·D flops
    each per visible (query, key) pair; S² pairs per head, S(S+1)/2 causal."""
    pairs = w.S * (w.S + 1) / 2 if w.causal else float(w.S) * w.S
    return 4.0 * w.B * w.Hq * w.D * pairs


def attn_bytes(w) -> float:
    """Algorithmic bytes: read Q, K, V once, write O once (bf16)."""
    return 2.0 * w.D * w.S * w.B * (2 * w.Hq + 2 * w.Hkv)


def attn_config(w, world: int = 1) -> dict:
    return {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "S": w.S, "D": w.D, "causal": w.causal,
            "layout": "Q, O [B, Hq, S, D]; K, V [B, Hkv, S, D]; bf16 row-major",
            "values": f"N(0,1) rounded to bf16, seeds {4000 + w.wid}/{5000 + w.wid}/{6000 + w.wid}",
            "l2": "no flush: Q alone is %d MiB > 126 MiB" % (w.B * w.Hq * w.S * w.D * 2 >> 20)
            if w.B * w.Hq * w.S * w.D * 2 > 126 << 20 else "inputs smaller than L2 (warm L2)",
            "softmax_scale": "1/sqrt(D)", "accumulate": "fp32", "output": "bf16", "parallelism": parallelism(world)}


def oracle_attn_rows_timed(Q, K, V, w, rows, with_values: bool = False):
    """The oracle on `rows` (query rows of head (0, 0)); returns (seconds, threads[, O rows as bf16 bits])."""
    import oracle
    q1, k1, v1 = (np.ascontiguousarray(x[:1, :1]) for x in (Q, K, V))
    t0 = time.perf_counter()
    O = oracle.attention_fwd(q1, k1, v1, causal=w.causal, rows=(0, rows))
    dt = time.perf_counter() - t0
    used = min(os.cpu_count() or 1, rows)
    return (dt, used, O[0, 0, :rows]) if with_values else (dt, used)


def attn_row_flops(w, rows: int) -> float:
    pairs = rows * (rows + 1) / 2 if w.causal else float(rows) * w.S
    return 4.0 * w.D * pairs


def attn_cpu_sample(w, Q, K, V, budget_s: float):
    """(oracle TFLOP/s, threads, query rows, seconds, those rows of O) on head (0, 0)."""
    rows = min(w.S, 64)
    t, _ = oracle_attn_rows_timed(Q, K, V, w, rows)
    rate = attn_row_flops(w, rows) / max(t, 1e-6)
    while rows < w.S and attn_row_flops(w, min(w.S, rows * 2)) / rate < budget_s:
        rows = min(w.S, rows * 2)
    t, used, O_ref = oracle_attn_rows_timed(Q, K, V, w, rows, with_values=True)
    return attn_row_flops(w, rows) / t / 1e12, used, rows, t, O_ref


def attn_parity_check(w, V, O_ref, O_gpu) -> dict:
    """Query rows 0..r-1 of head (0, 0) of the timed run's O against the
    oracle's, per entry within (2^-7 + S·2^-24)·max|V| + 2^-8·|O_ref| (bf16
    rounding of P, fp32 scores and accumulation, the output rounding; the
    weighted |V| of a row is at most max|V|); a miss fails the bench."""
    r = O_ref.shape[0]
    vmax = float(np.max(np.abs(synth.bf16_bits_to_f32(V[0, 0]).astype(np.float64))))
    ref = synth.bf16_bits_to_f32(O_ref).astype(np.float64)
    got = synth.bf16_bits_to_f32(O_gpu[0, 0, :r]).astype(np.float64)
    tol = (2.0 ** -7 + w.S * 2.0 ** -24) * vmax + 2.0 ** -8 * np.abs(ref)
    err = np.abs(got - ref)
    bad = ~(err <= tol)
    check = {"entries": int(ref.size), "query_rows": r, "misses": int(bad.sum()),
             "max_err_over_tol": float(np.max(err / tol)),
             "tolerance": "(2^-7 + S·2^-24)·max|V| + 2^-8·|O_ref| per entry, against the fp64 oracle"}
    if bad.any():
        raise RuntimeError(f"parity check of the timed run's O against the oracle failed: {check}")
    return check


def run_reference_attn(args, w):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if int(os.environ.get("RANK", "0")) != 0:
        return 0
    Q, K, V = synth.attn_operands(w)
    per_step = 120.0 / (args.steps + args.warmup)
    _, _, rows, _, _ = attn_cpu_sample(w, Q, K, V, per_step)
    for _ in range(args.warmup):
        oracle_attn_rows_timed(Q, K, V, w, rows)
    total, used = 0.0, 0
    for _ in range(args.steps):
        dt, used = oracle_attn_rows_timed(Q, K, V, w, rows)
        total += dt
    value = attn_row_flops(w, rows) * args.steps / total / 1e12
    line = {
        "impl": "reference", "metric": ATTN_METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": attn_config(w, world),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": used, "kind": "oracle",
                         "sample": f"query rows 0..{rows - 1} of head (0,0) per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_attn(args, w):
    import torch

    world, rank, local = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import dense_bf16_gemm_02_gb300 as hk

    Qb, Kb, Vb = synth.attn_operands(w)
    to_dev = lambda x: torch.from_numpy(x.view(np.int16)).to(dev).view(torch.bfloat16)
    Q, K, V = to_dev(Qb), to_dev(Kb), to_dev(Vb)
    O = torch.empty_like(Q)
    lse = torch.empty((w.B, w.Hq, w.S), dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    sh = int(stream.cuda_stream)
    flops = attn_flops(w)

    def launch(q, k, v, o):
        st = hk.hk_attention_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), w.B, w.Hq,
                                 w.Hkv, w.S, w.D, int(w.causal), sh)
        if st != hk.HK_OK:
            raise hk.HKError(st, "hk_attention_fwd")

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            launch(Q, K, V, O)
    torch.cuda.synchronize(dev)
    if hk.hk_gemm_last_device_status(local) != hk.HK_OK:
        raise RuntimeError("device status after warm-up: " + hk.hk_gemm_last_error_string())

    events = [torch.cuda.Event(enable_timing=True) for _ in range(2)]   # the timed region's two ends
    sampler = ClockSampler(local) if rank == 0 else None
    time.sleep(TIMED_PAUSE_S)   # (also lets the clock sampler start)
    barrier(world)
    torch.cuda.synchronize(dev)
    t_host0 = time.time()
    with torch.cuda.stream(stream):
        events[0].record(stream)
        for i in range(args.steps):
            launch(Q, K, V, O)
        events[1].record(stream)
    torch.cuda.synchronize(dev)
    t_host1 = time.time()
    barrier(world)
    elapsed_ms = events[0].elapsed_time(events[1])
    if hk.hk_gemm_last_device_status(local) != hk.HK_OK:
        raise RuntimeError("device status after timing: " + hk.hk_gemm_last_error_string())
    clocks = None
    if sampler:
        time.sleep(0.15)
        sampler.stop()
        clocks = sampler.summary(t_host0, t_host1)
    # per-launch spread, outside the timed region
    per_launch = launch_spread(lambda: launch(Q, K, V, O), stream, min(args.steps, 20))
    elapsed_max = max_over_ranks(world, elapsed_ms)

    # ---- end to end: pinned host Q, K, V -> device -> attention -> O to pinned host,
    # pipelined on three streams with double-buffered device tensors
    Q_h, K_h, V_h = (torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory() for x in (Qb, Kb, Vb))
    O_h = [torch.empty(Q.shape, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    Q_d, K_d, V_d, O_d = [Q, torch.empty_like(Q)], [K, torch.empty_like(K)], [V, torch.empty_like(V)], \
        [O, torch.empty_like(O)]
    s_h2d, s_d2h = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    e2e_steps = max(4, min(args.steps, 12))

    def e2e_run(n):
        h2d_done = [torch.cuda.Event() for _ in range(2)]
        comp_done, d2h_done = [None, None], [None, None]
        for i in range(n):
            k = i & 1
            if comp_done[k] is not None:
                s_h2d.wait_event(comp_done[k])
            with torch.cuda.stream(s_h2d):
                Q_d[k].copy_(Q_h, non_blocking=True)
                K_d[k].copy_(K_h, non_blocking=True)
                V_d[k].copy_(V_h, non_blocking=True)
                h2d_done[k].record(s_h2d)
            stream.wait_event(h2d_done[k])
            if d2h_done[k] is not None:
                stream.wait_event(d2h_done[k])
            launch(Q_d[k], K_d[k], V_d[k], O_d[k])
            comp_done[k] = torch.cuda.Event()
            comp_done[k].record(stream)
            s_d2h.wait_event(comp_done[k])
            with torch.cuda.stream(s_d2h):
                O_h[k].copy_(O_d[k], non_blocking=True)
                d2h_done[k] = torch.cuda.Event()
                d2h_done[k].record(s_d2h)

    e2e_run(2)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    e0.record(s_h2d)
    e2e_run(e2e_steps)
    e1.record(s_d2h)
    torch.cuda.synchronize(dev)
    barrier(world)
    e2e_ms = max_over_ranks(world, e0.elapsed_time(e1))
    if not np.array_equal(O_h[(e2e_steps - 1) & 1].view(torch.int16).numpy()[0, 0, :4],
                          O.view(torch.int16).cpu().numpy()[0, 0, :4]):
        raise RuntimeError("end-to-end result differs from the device result")

    # ---- context only: PyTorch's fused attention on the same GPU and inputs
    sdpa = None
    if rank == 0 and not args.no_cublas_context:
        try:
            import torch.nn.functional as F
            call = lambda: F.scaled_dot_product_attention(Q, K, V, is_causal=w.causal, enable_gqa=True)
            n_ctx = max(3, args.steps)   # as many back-to-back calls as our timed region
            ms = time_library(call, dev, args.warmup, n_ctx)
            sdpa = {"value": flops / (ms / 1e3) / 1e12, "unit": UNIT, "ms_per_call": ms, "launches": n_ctx,
                    "what": "torch scaled_dot_product_attention (enable_gqa) on the same GPU and inputs, "
                            "timed after ours with the same warm-up and pause; context only"}
        except Exception as exc:
            sdpa = {"unavailable": str(exc)[:200]}

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return 0
    peaks, peaks_src = load_peaks()
    peak, peak_source = tensor_peak(peaks, peaks_src, elapsed_max / 1e3)
    value = replica_value(flops, args.steps, world, elapsed_max)
    mean_launch_ms = elapsed_ms / args.steps   # the timed region's mean, back to back
    achieved = flops / (mean_launch_ms / 1e3) / 1e12
    digest = kernel_source_digest("attention")
    tr = MEASURED_TRAFFIC.get(w.name)
    traffic = tr["bytes_per_launch"] if tr and tr.get("source_digest") == digest else None
    h2d = int(sum(x.numel() * 2 for x in (Q_h, K_h, V_h)))
    line = {
        "metric": ATTN_METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": attn_config(w, world),
        "kernel_config": {"tile": "2x128 query rows per CTA, 128-key blocks"},
        "pct_of_peak": 100.0 * value / world / peak,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT,
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_source": peak_source,
                     "algorithmic_flops_per_launch": flops, "algorithmic_bytes_per_launch": attn_bytes(w),
                     "mean_launch_ms": mean_launch_ms, "p10_launch_ms": float(np.percentile(per_launch, 10)),
                     "p90_launch_ms": float(np.percentile(per_launch, 90)),
                     "spread_source": "p10/p90: launches timed one by one after the timed region",
                     "kernel": f"attn_fwd_kernel<{w.D}>", "source_digest": digest},
        "e2e": {"value": replica_value(flops, e2e_steps, world, e2e_ms), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": int(O_h[0].numel() * 2), "steps": e2e_steps,
                "pipelined": "H2D(i+1) | attention(i) | D2H(i-1) on three streams"},
        "gpu_launches": args.steps,
        "clocks": clocks,
        "context_sdpa": sdpa,
    }
    if not args.no_cpu_baseline:
        v, used, rows, t, O_ref = attn_cpu_sample(w, Qb, Kb, Vb, 15.0)
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": used, "kind": "oracle",
                                "sample": f"query rows 0..{rows - 1} of head (0,0) (fp64 C oracle, {t:.1f} s)"}
        line["parity_check"] = attn_parity_check(w, Vb, O_ref, O.view(torch.int16).cpu().numpy().view(np.uint16))
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0

# ---------------------------------------------------------------- calibration

CALIBRATE_SHAPES = [(1, 8192, 8192), (16, 8192, 8192), (64, 8192, 8192), (128, 8192, 8192), (192, 8192, 8192),
                  (256, 8192, 8192), (384, 8192, 8192), (512, 8192, 8192), (128, 28672, 8192), (1, 1024, 8192),
                  (1, 4096, 8192), (1, 8192, 28672), (1, 28672, 8192), (64, 8192, 28672), (256, 28672, 8192),
                  (128, 4096, 4096), (256, 4096, 16384), (2048, 2048, 8192), (1024, 8192, 8192), (64, 2048, 8192)]


def _calib_warm_us(fn, reps: int = 25) -> float:
    import torch
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / reps


def sweep_plans(shapes) -> None:
    """Every plan a shape can be forced to (every kernel id, K splits 1, 2, 3, 4,
    6, 8, 12), warm back-to-back calls between CUDA events, next to
    torch.matmul (cuBLAS) on the same inputs; per shape the automatic plan's
    time and every candidate sorted by time. The plan's time model
    (``estimate_us`` in the package's ``csrc/hk_gemm.cu``) is fitted to these."""
    import torch
    from dense_bf16_gemm_02_gb300 import hk_gemm as hk
    dev = torch.device("cuda", 0)
    for (M, N, K) in shapes:
        A = torch.randn(M, K, device=dev).to(torch.bfloat16)
        B = torch.randn(N, K, device=dev).to(torch.bfloat16)
        C = torch.empty(M, N, device=dev, dtype=torch.bfloat16)
        ref = A.float() @ B.float().T
        st = int(torch.cuda.current_stream().cuda_stream)

        def timed(plan):
            ws = torch.empty(max(plan.workspace_size, 256), dtype=torch.uint8, device=dev)
            run = lambda: plan.run_raw(A.data_ptr(), B.data_ptr(), C.data_ptr(), ws.data_ptr(), plan.workspace_size, st)
            if run() != hk.HK_OK:
                raise hk.HKError(run(), "hk_gemm_plan_run")
            torch.cuda.synchronize()
            err = (C.float() - ref).abs().max().item() / max(ref.abs().max().item(), 1e-30)
            if err > 0.02:
                raise AssertionError(f"{M}x{N}x{K} plan {plan.info()}: relative error {err}")
            return _calib_warm_us(run)

        auto = hk.Plan(M, N, K)
        ai = auto.info()
        t_auto = timed(auto)
        auto.close()
        t_lib = _calib_warm_us(lambda: torch.matmul(A, B.t()))
        res = []
        for kernel in hk.KERNELS:
            for split in (1, 2, 3, 4, 6, 8, 12):
                try:
                    plan = hk.Plan(M, N, K, kernel=kernel, split_k=split)
                except hk.HKError:
                    continue
                inf = plan.info()
                res.append((timed(plan), kernel, split, inf["tile_n"], inf["grid_ctas"], inf["stages"]))
                plan.close()
        res.sort()
        print(f"{M}x{N}x{K}: cuBLAS {t_lib:.1f} us; auto kernel {ai['kernel']} split {ai['split_k']} -> {t_auto:.1f} us; "
              "best: " + "; ".join(f"k{k} n{tn} s{s} g{g} st{stg}: {t:.1f}" for t, k, s, tn, g, stg in res), flush=True)


def l2_latency() -> None:
    """Builds and runs the package's ``csrc/diag_l2_latency.cu``: L2-hit latency
    by SM and by address region (the die question of the grid schedule)."""
    from dense_bf16_gemm_02_gb300.build import ARCH_FLAGS, BUILD_DIR, nvcc_path
    src = os.path.join(ROOT, "dense_bf16_gemm_02_gb300", "csrc", "diag_l2_latency.cu")
    exe = os.path.join(BUILD_DIR, "diag_l2_latency")
    os.makedirs(BUILD_DIR, exist_ok=True)
    subprocess.run([nvcc_path(), *ARCH_FLAGS, "-O3", "-std=c++17", "-o", exe, src], check=True)
    subprocess.run([exe], check=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["hk", "reference"], default="hk")
    ap.add_argument("--workload", default="gemm_8192",
                    choices=sorted(ALL_WORKLOADS) + sorted(synth.ATTN_WORKLOADS) + sorted(synth.MX_WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-cublas-context", action="store_true")
    ap.add_argument("--cold-l2", action="store_true",
                    help="GEMM workloads: write a %d MiB buffer before each timed launch and time each launch "
                         "alone (operands never in L2)" % (L2_FLUSH_BYTES >> 20))
    ap.add_argument("--epilogue", default="none", choices=["none", "bias", "bias_relu", "bias_gelu", "bias_silu"],
                    help="fused epilogue of each step (hk_gemm_bf16_epilogue)")
    ap.add_argument("--group-m", type=int, default=0,
                    help="raster group height in tile rows (0: the library default via hk_gemm_bf16)")
    ap.add_argument("--calibrate", choices=["plans", "l2"],
                    help="instead of a bench line: 'plans' times every forced plan of --shapes next to "
                         "cuBLAS (the data the plan time model is fitted to); 'l2' runs the L2 latency probe")
    ap.add_argument("--shapes", nargs="*", default=[], help="MxNxK shapes for --calibrate plans")
    args = ap.parse_args(argv)
    if args.calibrate == "plans":
        sweep_plans([tuple(map(int, s.split("x"))) for s in args.shapes] or CALIBRATE_SHAPES)
        return 0
    if args.calibrate == "l2":
        l2_latency()
        return 0
    args.warmup = max(args.warmup, 3)   # at least 3 untimed warm-up steps
    if args.cold_l2 and (args.workload in synth.MX_WORKLOADS or args.workload in synth.ATTN_WORKLOADS):
        ap.error("--cold-l2 applies to the bf16 and E4M3 GEMM workloads")
    if args.workload in synth.MX_WORKLOADS:
        w = synth.MX_WORKLOADS[args.workload]
        return run_reference_mx(args, w) if args.impl == "reference" else run_mx(args, w)
    if args.workload in synth.ATTN_WORKLOADS:
        w = synth.ATTN_WORKLOADS[args.workload]
        return run_reference_attn(args, w) if args.impl == "reference" else run_attn(args, w)
    w = ALL_WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)
    return run_hk(args, w)


if __name__ == "__main__":
    sys.exit(main())
