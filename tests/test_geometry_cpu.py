"""Compile-time geometry of every GEMM kernel variant, read on the CPU.

A small host program (built with nvcc, no GPU needed) includes the kernel
header and prints each variant's ring depth, shared memory, TMEM columns,
accumulator layout and tail-split flag. The checks pin the layout rules the
kernels rely on: shared memory within the 227 KB a CTA may have, TMEM
within 512 columns, epilogue chunks covering the tile, and half-width tail
units only where N / 2 is a valid MMA width with whole 8-row swizzle atoms
of B per CTA. They also pin the ring depths that were chosen by measurement.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "dense_bf16_gemm_02_gb300", "csrc")

# (CTAs per tile, tile N, FP8, MXFP8, A rows per stage, K atoms per stage): the library's variants
VARIANTS = [
    (1, 256, 0, 0, 16, 1), (1, 192, 0, 0, 16, 1), (1, 128, 0, 0, 16, 1), (1, 64, 0, 0, 16, 1),
    (1, 256, 0, 0, 64, 1), (1, 192, 0, 0, 64, 1), (1, 128, 0, 0, 64, 1), (1, 64, 0, 0, 64, 1),
    (2, 256, 0, 0, 128, 1), (2, 128, 0, 0, 128, 1), (2, 112, 0, 0, 128, 1),
    (1, 256, 0, 0, 128, 1), (1, 192, 0, 0, 128, 1), (1, 128, 0, 0, 128, 1), (1, 64, 0, 0, 128, 1),
    (2, 256, 1, 0, 128, 1), (1, 256, 1, 0, 128, 1), (1, 192, 1, 0, 128, 1), (1, 128, 1, 0, 128, 1),
    (1, 64, 1, 0, 128, 1), (1, 192, 1, 1, 128, 1), (2, 256, 1, 1, 128, 1),
]
FIELDS = ["stages", "smem", "tmem", "acc_bufs", "acc_cols", "halves", "chunks", "last_cols", "b_rows", "sf_slots",
          "sf_cols"]


@pytest.fixture(scope="module")
def geometry(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    d = tmp_path_factory.mktemp("geometry")
    lines = ['#include "gemm_kernel.cuh"', "#include <cstdio>", "template <class G> void row() {",
             '    std::printf("%d %d %d %d %d %d %d %d %d %d %d\\n", G::kStages, G::kSmemBytes, G::kTmemCols,',
             "                G::kAccBufs, G::kAccCols, G::kHalves ? 1 : 0, G::kEpiChunks, G::kLastChunkCols,",
             "                G::kBRows, G::kSfSlots, G::kSfCols);", "}", "int main() {"]
    for cg, n, fp8, mx, arows, atoms in VARIANTS:
        lines.append(f"    row<hk::Geometry<{cg}, {n}, {'true' if fp8 else 'false'}, {'true' if mx else 'false'}, "
                     f"{arows}, {atoms}>>();")
    lines.append("}")
    src = d / "geometry.cu"
    src.write_text("\n".join(lines) + "\n")
    exe = d / "geometry"
    subprocess.run([nvcc, "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a", "-I", CSRC, "-o", str(exe),
                    str(src)], check=True, capture_output=True, timeout=600)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True, timeout=60).stdout.split("\n")
    rows = [dict(zip(FIELDS, map(int, l.split()))) for l in out if l.strip()]
    assert len(rows) == len(VARIANTS)
    return dict(zip(VARIANTS, rows))


def test_every_variant_fits_shared_memory_and_tmem(geometry):
    for v, g in geometry.items():
        assert g["smem"] <= 232448, v                       # dynamic shared memory a CTA may have on sm_103
        assert g["stages"] >= 3, v
        assert 32 <= g["tmem"] <= 512 and g["tmem"] & (g["tmem"] - 1) == 0, v   # a power-of-2 allocation
        assert g["acc_bufs"] * g["acc_cols"] + g["sf_slots"] * g["sf_cols"] <= g["tmem"], v
        assert g["b_rows"] % 8 == 0 and g["b_rows"] * v[0] == v[1], v   # whole swizzle atoms of B per CTA


def test_epilogue_chunks_cover_the_tile(geometry):
    for v, g in geometry.items():
        n = v[1]
        assert g["acc_cols"] == 32 * g["chunks"] and g["acc_cols"] >= n, v   # 32-column TMEM reads stay inside
        assert g["last_cols"] == n - 32 * (g["chunks"] - 1) and g["last_cols"] in (16, 32), v


def test_half_width_units_only_where_the_half_is_a_valid_tile(geometry):
    for v, g in geometry.items():
        cg, n = v[0], v[1]
        valid = n % (16 * cg) == 0 and (n // cg // 2) % 8 == 0
        assert g["halves"] == int(valid), v
    assert geometry[(2, 112, 0, 0, 128, 1)]["halves"] == 0      # N / 2 = 56: no cta_group::2 MMA of that width
    assert geometry[(2, 128, 0, 0, 128, 1)]["halves"] == 1
    assert geometry[(2, 256, 0, 0, 128, 1)]["halves"] == 1


def test_ring_depths_chosen_by_measurement(geometry):
    assert geometry[(2, 256, 0, 0, 128, 1)]["stages"] == 6      # 32 KB stages of the 256-wide pair
    assert geometry[(2, 128, 0, 0, 128, 1)]["stages"] == 8      # capped at 8
    assert geometry[(2, 112, 0, 0, 128, 1)]["stages"] == 9      # 23 KB stages: a ninth fits (bytes in flight)
    assert geometry[(2, 112, 0, 0, 128, 1)]["acc_cols"] == 128  # 112 columns at a 128-column stride
    for n in (256, 192, 128, 64):                               # short A stages hold more of B in flight
        assert (geometry[(1, n, 0, 0, 16, 1)]["stages"] >= geometry[(1, n, 0, 0, 64, 1)]["stages"]
                >= geometry[(1, n, 0, 0, 128, 1)]["stages"]), n
    assert geometry[(2, 256, 1, 1, 128, 1)]["acc_bufs"] == 1    # block-scaled pair: one accumulator beside the scale ring
