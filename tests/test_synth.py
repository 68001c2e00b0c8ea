"""The seeded input generator: determinism, chunk independence, rounding."""
import numpy as np
import torch

import synth


def test_f32_to_bf16_matches_torch_rne():
    g = np.random.Generator(np.random.PCG64(1))
    x = (g.standard_normal(1 << 16) * np.exp2(g.integers(-30, 30, 1 << 16))).astype(np.float32)
    x[:4] = [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 0.0]
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(synth.f32_to_bf16_bits(x), want)
    assert np.array_equal(synth.bf16_bits_to_f32(want), torch.from_numpy(want.view(np.int16)).view(
        torch.bfloat16).float().numpy())


def test_chunked_generation_is_one_stream(monkeypatch):
    full = synth.normal_bf16(64, 1000, 7, 0.5)
    monkeypatch.setattr(synth, "_CHUNK", 777)
    assert np.array_equal(synth.normal_bf16(64, 1000, 7, 0.5), full)


def test_deterministic_and_scaled():
    a = synth.normal_bf16(128, 128, 1001)
    assert np.array_equal(a, synth.normal_bf16(128, 128, 1001))
    v = synth.bf16_bits_to_f32(synth.normal_bf16(512, 512, 3, 0.02))
    assert abs(float(v.std()) - 0.02) < 0.001 and abs(float(v.mean())) < 0.001


def test_integer_variant_range():
    a = synth.bf16_bits_to_f32(synth.int_bf16(100, 100, 1101))
    assert set(np.unique(a).tolist()) == set(range(-4, 5))


def test_positions_cover_edges():
    r, c = synth.sample_positions(300, 700, 3003, count=100)
    assert r.min() >= 0 and r.max() == 299 and c.min() == 0 and c.max() == 699
    assert ((r == 0) & (c == 0)).any() and ((r == 299) & (c == 699)).any()
    rows = synth.full_rows(8192, 3003)
    assert len(rows) == 8 and rows[0] == 0 and rows[-1] == 8191


def test_workload_table():
    w = synth.WORKLOADS["gemm_8192"]
    assert (w.M, w.N, w.K, w.scale) == (8192, 8192, 8192, 0.5)
    assert synth.WORKLOADS["skinny_128x28672x8192"].M == 128
