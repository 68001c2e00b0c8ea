"""Pins for the attention-forward oracle, against things other than itself.

The operation (HipKittens "L2" detail page, §3 "Target operation" table, rows
"MHA fwd" and "GQA fwd"; §5 "Numerical considerations", online softmax with
temperature sqrt(1/D)): for every batch b, query head h and query row i,

    O[b,h,i,:] = bf16_rne( Σ_j softmax_j(Q[b,h,i,:]·K[b,g,j,:] / √D) V[b,g,j,:] ),
    g = h // (Hq / Hkv),  j ≤ i when causal,

plus the log-sum-exp ln Σ_j exp(Q·K/√D) of every row (§9.3, epilogue). The
pages print no element values, so the pins are closed forms (a zero query
averages the visible value rows; a dominant key selects its value row; two
keys give the logistic function), exact rational arithmetic for the
averages, and structural identities (GQA equals MHA over repeated K/V heads,
a batched call equals per-head calls, a causal row equals the full softmax
over its prefix). ``test_attention_mutants_fail_pins`` plants plausible
mistakes into a copy of the oracle's C source and checks that the pins catch
every one of them.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from fractions import Fraction

import numpy as np
import pytest

import synth
from exact_bf16 import bits_to_fraction, round_fraction

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


class _AttnLib:
    """Driver for a compiled copy of the oracle's C source (attention only)."""

    def __init__(self, path):
        lib = ctypes.CDLL(path)
        P, I = ctypes.c_void_p, ctypes.c_int64
        lib.oracle_attention_fwd.argtypes = [P, P, P, P, P, I, I, I, I, I, ctypes.c_int, I, I, ctypes.c_int]
        lib.oracle_attention_fwd.restype = ctypes.c_int
        self.lib = lib

    def attention_fwd(self, Q, K, V, causal=False, rows=None, threads=1, with_lse=False):
        Q, K, V = (np.ascontiguousarray(x, dtype=np.uint16) for x in (Q, K, V))
        B, Hq, S, D = Q.shape
        Hkv = K.shape[1]
        O = np.zeros_like(Q)
        lse = np.full((B, Hq, S), np.nan)
        r0, r1 = (0, B * Hq * S) if rows is None else rows
        self.lib.oracle_attention_fwd(Q.ctypes.data, K.ctypes.data, V.ctypes.data, O.ctypes.data,
                                      lse.ctypes.data, B, Hq, Hkv, S, D, int(causal), r0, r1, threads)
        return (O, lse) if with_lse else O


class _Packaged:
    """The packaged oracle with the same call shape as ``_AttnLib``."""

    def __init__(self, oracle):
        self.o = oracle

    def attention_fwd(self, Q, K, V, causal=False, rows=None, threads=1, with_lse=False):
        return self.o.attention_fwd(Q, K, V, causal=causal, rows=rows, threads=threads, with_lse=with_lse)


def _f(bits):
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


def _bits(x: float) -> int:
    """bf16 bits of a value that is exactly representable."""
    b = round_fraction(Fraction(x))
    assert bits_to_fraction(b) == Fraction(x)
    return b


def _near(ref: float, got_bits: int, eps: float = 1e-12) -> bool:
    """``got`` is the RNE rounding of a value within relative eps of ``ref``
    (the reference is a binary64 evaluation; only a rounding boundary closer
    than eps could make the two roundings differ)."""
    lo, hi = sorted((ref * (1 - eps), ref * (1 + eps)))
    cands = {round_fraction(Fraction(lo)), round_fraction(Fraction(hi)), round_fraction(Fraction(ref))}
    return int(got_bits) in cands


# ---------------------------------------------------------------- the pins --

def pin_zero_query_averages(o):
    """Q = 0: every visible score is 0, so each output row is the plain mean
    of the visible value rows (exact rational, rounded once), and the
    log-sum-exp is ln(number of visible keys)."""
    B, Hq, Hkv, S, D = 2, 4, 2, 12, 8
    Q = np.zeros((B, Hq, S, D), dtype=np.uint16)
    K = synth.normal_bf16(B * Hkv * S, D, 11).reshape(B, Hkv, S, D)
    V = synth.int_bf16(B * Hkv * S, D, 12).reshape(B, Hkv, S, D)
    for causal in (False, True):
        O, lse = o.attention_fwd(Q, K, V, causal=causal, with_lse=True)
        for b in range(B):
            for h in range(Hq):
                g = h // (Hq // Hkv)
                for i in range(S):
                    n = i + 1 if causal else S
                    for t in range(D):
                        mean = sum(bits_to_fraction(int(V[b, g, j, t])) for j in range(n)) / n
                        if int(O[b, h, i, t]) != round_fraction(mean):
                            return f"zero query: O[{b},{h},{i},{t}] causal={causal}"
                    if abs(lse[b, h, i] - math.log(n)) > 1e-12:
                        return f"zero query: lse[{b},{h},{i}] = {lse[b, h, i]}, want ln {n}"
    return None


def _one_hot_keys(S, D, mag=64.0):
    """Key j = mag · e_j (needs S <= D)."""
    K = np.zeros((S, D), dtype=np.uint16)
    for j in range(S):
        K[j, j] = _bits(mag)
    return K


def pin_dominant_key(o):
    """Query i = 64·e_π(i) against keys 64·e_j (D = S = 16): the matching key
    scores 64·64/√16 = 1024 and every other key 0, so exp(-1024) vanishes in
    binary64 and O = V[π(i)] exactly, with log-sum-exp 1024. Causal: a query
    that points at a future key sees only zero scores, so it averages the
    value rows up to its own position."""
    S = D = 16
    Kh = _one_hot_keys(S, D)
    V = synth.int_bf16(S, D, 21).reshape(1, 1, S, D)
    perm = np.random.Generator(np.random.PCG64(22)).permutation(S)
    Q = np.zeros((1, 1, S, D), dtype=np.uint16)
    for i in range(S):
        Q[0, 0, i, perm[i]] = _bits(64.0)
    O, lse = o.attention_fwd(Q, Kh.reshape(1, 1, S, D), V, with_lse=True)
    for i in range(S):
        if not np.array_equal(O[0, 0, i], V[0, 0, perm[i]]):
            return f"dominant key: row {i} is not V[{perm[i]}]"
        if lse[0, 0, i] != 1024.0:
            return f"dominant key: lse[{i}] = {lse[0, 0, i]}"
    # causal: query i points at key i+1 (masked) except the last, which points at key 0
    Qc = np.zeros((1, 1, S, D), dtype=np.uint16)
    for i in range(S):
        Qc[0, 0, i, (i + 1) % S] = _bits(64.0)
    Oc = o.attention_fwd(Qc, Kh.reshape(1, 1, S, D), V, causal=True)
    for i in range(S - 1):
        for t in range(D):
            mean = sum(bits_to_fraction(int(V[0, 0, j, t])) for j in range(i + 1)) / (i + 1)
            if int(Oc[0, 0, i, t]) != round_fraction(mean):
                return f"dominant key, causal: row {i} col {t} is not the prefix mean"
    if not np.array_equal(Oc[0, 0, S - 1], V[0, 0, 0]):
        return "dominant key, causal: last row is not V[0]"
    return None


def pin_two_keys_logistic(o):
    """Two keys: the weights are σ(Δ) and σ(-Δ) with Δ = q·(k1 - k0)/√D, the
    logistic function (scipy.special.expit), so O = σ(Δ)·v1 + σ(-Δ)·v0."""
    from scipy.special import expit
    for D, seed in ((16, 31), (64, 32), (128, 33)):
        Hq = 3
        Q = synth.int_bf16(Hq * 2, D, seed, -2, 2).reshape(1, Hq, 2, D)
        K = synth.int_bf16(2, D, seed + 100, -2, 2).reshape(1, 1, 2, D)
        V = synth.normal_bf16(2, D, seed + 200).reshape(1, 1, 2, D)
        O, lse = o.attention_fwd(Q, K, V, with_lse=True)
        q, k, v = _f(Q[0]), _f(K[0, 0]), _f(V[0, 0])
        for h in range(Hq):
            for i in range(2):
                s0, s1 = (q[h, i] @ k[0]) / math.sqrt(D), (q[h, i] @ k[1]) / math.sqrt(D)
                w1 = expit(s1 - s0)
                w0 = expit(s0 - s1)
                for t in range(D):
                    ref = w1 * v[1, t] + w0 * v[0, t]
                    if not _near(ref, O[0, h, i, t]):
                        return f"two keys D={D}: O[{h},{i},{t}]"
                want_lse = max(s0, s1) + math.log1p(math.exp(-abs(s1 - s0)))
                if abs(lse[0, h, i] - want_lse) > 1e-12 * max(1.0, abs(want_lse)):
                    return f"two keys D={D}: lse[{h},{i}]"
    return None


def pin_gqa_is_repeated_mha(o):
    """GQA with Hq/Hkv query heads per KV head equals MHA whose K and V heads
    are the GQA heads each repeated Hq/Hkv times, consecutively."""
    B, Hq, Hkv, S, D = 2, 6, 2, 9, 16
    Q = synth.normal_bf16(B * Hq * S, D, 41).reshape(B, Hq, S, D)
    K = synth.normal_bf16(B * Hkv * S, D, 42).reshape(B, Hkv, S, D)
    V = synth.normal_bf16(B * Hkv * S, D, 43).reshape(B, Hkv, S, D)
    Kr = np.ascontiguousarray(np.repeat(K, Hq // Hkv, axis=1))
    Vr = np.ascontiguousarray(np.repeat(V, Hq // Hkv, axis=1))
    for causal in (False, True):
        a, la = o.attention_fwd(Q, K, V, causal=causal, with_lse=True)
        m, lm = o.attention_fwd(Q, Kr, Vr, causal=causal, with_lse=True)
        if not (np.array_equal(a, m) and np.array_equal(la, lm)):
            return f"GQA differs from repeated-head MHA (causal={causal})"
    return None


def pin_batched_equals_per_head(o):
    """A batched call equals one single-head call per (b, h) on that head's
    query and its KV group's keys and values."""
    B, Hq, Hkv, S, D = 2, 4, 2, 7, 8
    Q = synth.normal_bf16(B * Hq * S, D, 51).reshape(B, Hq, S, D)
    K = synth.normal_bf16(B * Hkv * S, D, 52).reshape(B, Hkv, S, D)
    V = synth.normal_bf16(B * Hkv * S, D, 53).reshape(B, Hkv, S, D)
    for causal in (False, True):
        O = o.attention_fwd(Q, K, V, causal=causal)
        for b in range(B):
            for h in range(Hq):
                g = h // (Hq // Hkv)
                one = o.attention_fwd(np.ascontiguousarray(Q[b:b + 1, h:h + 1]),
                                      np.ascontiguousarray(K[b:b + 1, g:g + 1]),
                                      np.ascontiguousarray(V[b:b + 1, g:g + 1]), causal=causal)
                if not np.array_equal(one[0, 0], O[b, h]):
                    return f"batched call differs from the per-head call at b={b} h={h} (causal={causal})"
    return None


def pin_causal_is_prefix(o):
    """Causal row i equals row i of the full (non-causal) softmax over the
    first i+1 keys, and does not move when later keys and values change."""
    S, D = 10, 8
    Q = synth.normal_bf16(S, D, 61).reshape(1, 1, S, D)
    K = synth.normal_bf16(S, D, 62).reshape(1, 1, S, D)
    V = synth.normal_bf16(S, D, 63).reshape(1, 1, S, D)
    O = o.attention_fwd(Q, K, V, causal=True)
    for i in range(S):
        n = i + 1
        pre = o.attention_fwd(np.ascontiguousarray(Q[:, :, :n]), np.ascontiguousarray(K[:, :, :n]),
                              np.ascontiguousarray(V[:, :, :n]))
        if not np.array_equal(pre[0, 0, i], O[0, 0, i]):
            return f"causal row {i} differs from the full softmax over its prefix"
    K2, V2 = K.copy(), V.copy()
    K2[0, 0, 5:] = synth.normal_bf16(S - 5, D, 64)
    V2[0, 0, 5:] = synth.normal_bf16(S - 5, D, 65)
    O2 = o.attention_fwd(Q, K2, V2, causal=True)
    if not np.array_equal(O2[0, 0, :5], O[0, 0, :5]):
        return "causal rows depend on later keys"
    return None


def pin_rows_subset(o):
    """Computing a range of rows gives those rows of the full result."""
    B, Hq, Hkv, S, D = 1, 2, 1, 8, 8
    Q = synth.normal_bf16(B * Hq * S, D, 71).reshape(B, Hq, S, D)
    K = synth.normal_bf16(B * Hkv * S, D, 72).reshape(B, Hkv, S, D)
    V = synth.normal_bf16(B * Hkv * S, D, 73).reshape(B, Hkv, S, D)
    full = o.attention_fwd(Q, K, V, causal=True).reshape(-1, D)
    part = o.attention_fwd(Q, K, V, causal=True, rows=(5, 13)).reshape(-1, D)
    if not (np.array_equal(part[5:13], full[5:13]) and not part[:5].any() and not part[13:].any()):
        return "row range differs from the full result"
    return None


PINS = [pin_zero_query_averages, pin_dominant_key, pin_two_keys_logistic, pin_gqa_is_repeated_mha,
        pin_batched_equals_per_head, pin_causal_is_prefix, pin_rows_subset]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_attention_oracle_pin(oracle_lib, pin):
    assert pin(_Packaged(oracle_lib)) is None


def test_attention_threads_agree(oracle_lib):
    B, Hq, Hkv, S, D = 1, 4, 1, 33, 64
    Q = synth.normal_bf16(B * Hq * S, D, 81).reshape(B, Hq, S, D)
    K = synth.normal_bf16(B * Hkv * S, D, 82).reshape(B, Hkv, S, D)
    V = synth.normal_bf16(B * Hkv * S, D, 83).reshape(B, Hkv, S, D)
    a = oracle_lib.attention_fwd(Q, K, V, causal=True, threads=1)
    b = oracle_lib.attention_fwd(Q, K, V, causal=True, threads=7)
    assert np.array_equal(a, b)


def test_attention_rejects_bad_shapes(oracle_lib):
    Q = np.zeros((1, 3, 4, 8), dtype=np.uint16)
    K = np.zeros((1, 2, 4, 8), dtype=np.uint16)
    with pytest.raises(ValueError):
        oracle_lib.attention_fwd(Q, K, K)


# ------------------------------------------------------------- mutations --

ATTN_MUTANTS = {
    "no_scale": ("const double scale = 1.0 / sqrt((double)w->D);", "const double scale = 1.0;"),
    "scale_by_d": ("const double scale = 1.0 / sqrt((double)w->D);", "const double scale = 1.0 / (double)w->D;"),
    "group_modulo": ("g = h / group;", "g = h % w->Hkv;"),
    "causal_off_by_one": ("const int64_t n = w->causal ? i + 1 : w->S;", "const int64_t n = w->causal ? i : w->S;"),
    "causal_ignored": ("const int64_t n = w->causal ? i + 1 : w->S;", "const int64_t n = w->S;"),
    "not_normalised": ("out[t] = oracle_round_bf16(o[t] / sum);", "out[t] = oracle_round_bf16(o[t]);"),
    "values_from_keys": ("const uint16_t* vb = w->V +", "const uint16_t* vb = w->K +"),
    "no_max_shift": ("s[j] = exp(s[j] - mx);", "s[j] = exp(s[j]);"),
    "batch_ignored": ("const uint16_t* kb = w->K + (b * w->Hkv + g) * w->S * w->D;",
                      "const uint16_t* kb = w->K + g * w->S * w->D;"),
    "row_order": ("const int64_t i = r % w->S, h = (r / w->S) % w->Hq,",
                  "const int64_t h = r % w->Hq, i = (r / w->Hq) % w->S,"),
    "value_columns_reversed": ("o[t] += s[j] * bf16_bits_to_double(vb[j * w->D + t]);",
                               "o[t] += s[j] * bf16_bits_to_double(vb[j * w->D + (w->D - 1 - t)]);"),
    "lse_without_max": ("if (w->lse) w->lse[r] = mx + log(sum);", "if (w->lse) w->lse[r] = log(sum);"),
}


@pytest.mark.parametrize("name", sorted(ATTN_MUTANTS))
def test_attention_mutants_fail_pins(tmp_path, name):
    src = open(os.path.join(ROOT, "oracle", "gemm_ref.c")).read()
    old, new = ATTN_MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    path_c = tmp_path / f"{name}.c"
    path_so = tmp_path / f"{name}.so"
    path_c.write_text(src.replace(old, new))
    subprocess.run(["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
                    "-D_GNU_SOURCE", str(path_c), "-o", str(path_so), "-lm"], check=True)
    mutant = _AttnLib(str(path_so))
    with np.errstate(all="ignore"):
        failures = [p.__name__ for p in PINS if p(mutant) is not None]
    assert failures, f"mutant {name} passed every attention pin"
