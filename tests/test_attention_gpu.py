"""GPU parity of the attention forward (hk_attention_fwd) against the oracle.

Every case runs the CUDA kernel through the C-ABI and compares each output
element with the fp64 oracle on the same seeded inputs. The tolerance is
derived from the kernel's arithmetic (written out in ``attn_tolerance``).
Sizes span several K/V blocks and query tiles with ragged tails; the
workloads of the pages' Figure 7 (batch 16, 64 query heads, 8 KV heads,
S 4096, D 64 / 128, causal and not) are checked on sampled heads and rows.
"""
from __future__ import annotations

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def hk():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("no CUDA device")
    import dense_bf16_gemm_02_gb300 as pkg
    pkg.load()
    return pkg


@pytest.fixture(scope="module")
def oracle():
    import oracle as o
    o.build()
    return o


def _dev(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to("cuda").view(torch.bfloat16)


def _host(t):
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def run_attention(hk, Q, K, V, causal, flags=0, timeout_ns=0):
    """(O bits, lse) from the CUDA kernel through the C-ABI."""
    import torch
    B, Hq, S, D = Q.shape
    Hkv = K.shape[1]
    q, k, v = _dev(Q), _dev(K), _dev(V)
    o = torch.full(Q.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, Hq, S), float("nan"), dtype=torch.float32, device="cuda")
    stream = int(torch.cuda.current_stream().cuda_stream)
    st = hk.hk_attention_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                B, Hq, Hkv, S, D, int(causal), flags, timeout_ns, stream)
    assert st == hk.HK_OK, hk.hk_gemm_last_error_string()
    torch.cuda.synchronize()
    return _host(o), lse.cpu().numpy().astype(np.float64)


def attn_tolerance(Q, K, V, causal, want_bits):
    """Per-element bound on |O_gpu - O_oracle| for one head's rows:

        (2^-7 + S·2^-24) · W  +  2^-8 · |O_oracle|,   W = Σ_j P_ij |V_jt|.

    The kernel rounds P to bf16 (≤ 2^-9 relative per weight) while the row
    sum uses the fp32 P (another ≤ 2^-9 on the normalisation); exp2 and the
    fp32 scores add well under 2^-12; the margin doubles the 2^-8 these give.
    The fp32 accumulation of P·V over S keys is bounded by S·2^-24·W, and
    the two bf16 roundings of the outputs by 2^-8·|O|. Q, K, V here are one
    head's [S, D] float64 arrays; W is formed in float64."""
    S, D = Q.shape
    s = (Q @ K.T) / np.sqrt(D)
    if causal:
        s = np.where(np.tril(np.ones((s.shape[0], S), dtype=bool)), s, -np.inf)
    s -= s.max(axis=1, keepdims=True)
    P = np.exp(s)
    P /= P.sum(axis=1, keepdims=True)
    W = P @ np.abs(V)
    want = synth.bf16_bits_to_f32(want_bits).astype(np.float64)
    return (2.0 ** -7 + S * 2.0 ** -24) * W + 2.0 ** -8 * np.abs(want) + 1e-30


def _f64(bits):
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


def check_heads(got, want, Q, K, V, causal, heads=None, rows=None, what=""):
    """Element-wise comparison per (b, h) head (all heads unless given)."""
    B, Hq, S, D = Q.shape
    Hkv = K.shape[1]
    heads = heads if heads is not None else [(b, h) for b in range(B) for h in range(Hq)]
    for b, h in heads:
        g = h // (Hq // Hkv)
        r = np.arange(S) if rows is None else np.asarray(rows)
        q = _f64(Q[b, h])
        tol = attn_tolerance(q[r], _f64(K[b, g]), _f64(V[b, g]), False, want[b, h][r])
        if causal:   # mask per row: recompute with the rows' own prefixes
            tol = np.stack([attn_tolerance(q[i:i + 1], _f64(K[b, g, :i + 1]), _f64(V[b, g, :i + 1]), False,
                                           want[b, h][i:i + 1])[0] for i in r])
        g_ = _f64(got[b, h][r])
        w_ = _f64(want[b, h][r])
        assert np.all(np.isfinite(g_)), f"{what}: non-finite output at head ({b},{h})"
        err = np.abs(g_ - w_)
        bad = err > tol
        if bad.any():
            idx = np.argwhere(bad)[:5]
            raise AssertionError(f"{what}: head ({b},{h}): {int(bad.sum())} of {bad.size} outside tolerance; "
                                 f"first (row,col) {[(int(r[i]), int(j)) for i, j in idx]} got {g_[bad][:5]} "
                                 f"want {w_[bad][:5]} tol {tol[bad][:5]}")


def check_lse(got, want, what=""):
    ok = np.abs(got - want) <= 1e-4 + 1e-5 * np.abs(want)
    assert ok.all(), f"{what}: lse differs at {np.argwhere(~ok)[:5].tolist()}: got {got[~ok][:5]} want {want[~ok][:5]}"


def _inputs(B, Hq, Hkv, S, D, seed, q_scale=1.0):
    Q = synth.normal_bf16(B * Hq * S, D, seed, q_scale).reshape(B, Hq, S, D)
    K = synth.normal_bf16(B * Hkv * S, D, seed + 1).reshape(B, Hkv, S, D)
    V = synth.normal_bf16(B * Hkv * S, D, seed + 2).reshape(B, Hkv, S, D)
    return Q, K, V


SHAPES = [
    # B, Hq, Hkv, S, D
    (1, 1, 1, 128, 128),     # one K/V block, one query tile (the second tile is empty)
    (1, 2, 1, 256, 128),     # both query tiles, two K/V blocks
    (2, 8, 2, 300, 128),     # GQA, ragged S (three blocks, last one 44 keys)
    (1, 4, 1, 520, 64),      # D = 64, ragged, 3 query pairs
    (1, 2, 2, 1, 128),       # a single key and query
    (1, 3, 1, 129, 64),      # one key past a block boundary
    (1, 2, 1, 1000, 128),    # eight blocks
]


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_attention_matches_oracle(hk, oracle, shape, causal):
    B, Hq, Hkv, S, D = shape
    Q, K, V = _inputs(B, Hq, Hkv, S, D, 100 + S + D)
    got, lse = run_attention(hk, Q, K, V, causal)
    want, want_lse = oracle.attention_fwd(Q, K, V, causal=causal, with_lse=True)
    check_heads(got, want, Q, K, V, causal, what=f"{shape} causal={causal}")
    check_lse(lse, want_lse, f"{shape} causal={causal}")


# Many more work items (256 query rows of one head) than CTAs (one per SM), so
# each CTA walks several items back to back: ragged S makes the last item of
# every head end with an empty second tile (S = 300: rows 256..299 only) or a
# short one (S = 520), and causal items differ in length; every element is
# checked against the oracle.
MULTI_ITEM_SHAPES = [
    (8, 32, 8, 300, 128),    # 512 items, every second one with an empty second tile
    (4, 32, 4, 520, 64),     # 384 items of three lengths
    (16, 16, 4, 1, 128),     # 256 items of a single row
]


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("shape", MULTI_ITEM_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_attention_many_items_per_cta(hk, oracle, shape, causal):
    B, Hq, Hkv, S, D = shape
    Q, K, V = _inputs(B, Hq, Hkv, S, D, 700 + S + D)
    got, lse = run_attention(hk, Q, K, V, causal)
    want, want_lse = oracle.attention_fwd(Q, K, V, causal=causal, with_lse=True)
    check_heads(got, want, Q, K, V, causal, what=f"{shape} causal={causal}")
    check_lse(lse, want_lse, f"{shape} causal={causal}")


def test_attention_growing_scores_rescale(hk, oracle):
    """Keys whose norm grows along the sequence make every row's maximum
    jump by more than 2^8 between blocks, exercising the output rescale."""
    B, Hq, Hkv, S, D = 1, 2, 1, 640, 128
    Q, K, V = _inputs(B, Hq, Hkv, S, D, 900, q_scale=2.0)
    ramp = (1.0 + np.arange(S) / 32.0).astype(np.float32)[None, None, :, None]
    K = synth.f32_to_bf16_bits(synth.bf16_bits_to_f32(K) * ramp).reshape(K.shape)
    for causal in (False, True):
        got, lse = run_attention(hk, Q, K, V, causal)
        want, want_lse = oracle.attention_fwd(Q, K, V, causal=causal, with_lse=True)
        check_heads(got, want, Q, K, V, causal, what=f"growing scores causal={causal}")
        check_lse(lse, want_lse, f"growing scores causal={causal}")


def test_attention_one_hot_selects_value_rows(hk):
    """Query i = 64·e_π(i), key j = 64·e_j (S = D = 128): the matching key's
    score (64·64/√128 ≈ 362) dwarfs the rest, so O = V[π(i)] to bf16."""
    S = D = 128
    perm = np.random.Generator(np.random.PCG64(5)).permutation(S)
    Q = np.zeros((1, 1, S, D), dtype=np.uint16)
    K = np.zeros((1, 1, S, D), dtype=np.uint16)
    Q[0, 0, np.arange(S), perm] = 0x4280   # 64.0
    K[0, 0, np.arange(S), np.arange(S)] = 0x4280
    V = synth.normal_bf16(S, D, 6).reshape(1, 1, S, D)
    got, _ = run_attention(hk, Q, K, V, False)
    assert np.array_equal(got[0, 0], V[0, 0, perm])


def test_attention_is_deterministic(hk):
    Q, K, V = _inputs(1, 8, 2, 777, 128, 31)
    a, la = run_attention(hk, Q, K, V, True)
    b, lb = run_attention(hk, Q, K, V, True)
    assert np.array_equal(a, b) and np.array_equal(la, lb)


@pytest.mark.parametrize("name", sorted(synth.ATTN_WORKLOADS))
def test_attention_workloads(hk, oracle, name):
    """The benchmarked workloads at full size: sampled heads (first, last and
    seeded ones), each checked on sampled rows including the first and last
    row and both sides of query-tile and K/V-block boundaries."""
    w = synth.ATTN_WORKLOADS[name]
    Q, K, V = synth.attn_operands(w)
    got, lse = run_attention(hk, Q, K, V, w.causal)
    g = np.random.Generator(np.random.PCG64(7000 + w.wid))
    heads = {(0, 0), (w.B - 1, w.Hq - 1)}
    while len(heads) < (4 if w.sampled else w.B * w.Hq):
        heads.add((int(g.integers(0, w.B)), int(g.integers(0, w.Hq))))
    edge = {0, w.S - 1} | {x for t in range(0, w.S, 128) for x in (t, t + 127) if x < w.S}
    rows = sorted(edge | set(int(x) for x in g.integers(0, w.S, size=24))) if w.sampled else None
    for b, h in sorted(heads):
        kvh = h // (w.Hq // w.Hkv)
        q1 = np.ascontiguousarray(Q[b:b + 1, h:h + 1])
        k1 = np.ascontiguousarray(K[b:b + 1, kvh:kvh + 1])
        v1 = np.ascontiguousarray(V[b:b + 1, kvh:kvh + 1])
        if rows is None:
            want, want_lse = oracle.attention_fwd(q1, k1, v1, causal=w.causal, with_lse=True)
            sel = np.arange(w.S)
        else:
            want = np.zeros_like(q1)
            want_lse = np.full((1, 1, w.S), np.nan)
            for r in rows:
                o1, l1 = oracle.attention_fwd(q1, k1, v1, causal=w.causal, rows=(r, r + 1), with_lse=True)
                want[0, 0, r] = o1[0, 0, r]
                want_lse[0, 0, r] = l1[0, 0, r]
            sel = np.asarray(rows)
        check_heads(got[b:b + 1, h:h + 1], want, q1, k1, v1, w.causal, heads=[(0, 0)], rows=sel,
                    what=f"{name} head ({b},{h})")
        check_lse(lse[b, h, sel], want_lse[0, 0, sel], f"{name} head ({b},{h})")


def test_attention_bounded_wait_reports_timeout(hk):
    """The test flag withholds the first K/V block: the kernel's bounded wait
    runs out, the status word reports HK_ERR_TIMEOUT, and the next call on
    the same device works."""
    import torch
    Q, K, V = _inputs(1, 2, 1, 256, 128, 41)
    q, k, v = _dev(Q), _dev(K), _dev(V)
    o = torch.empty_like(q)
    st = hk.hk_attention_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), 0, 1, 2, 1, 256, 128, 0,
                                hk.HK_FLAG_FAULT_DROP_ARRIVE, 20_000_000, 0)
    assert st == hk.HK_OK
    torch.cuda.synchronize()
    assert hk.hk_gemm_last_device_status(torch.cuda.current_device()) == hk.HK_ERR_TIMEOUT
    got, _ = run_attention(hk, Q, K, V, False)
    assert np.all(np.isfinite(_f64(got)))
    assert hk.hk_gemm_last_device_status(torch.cuda.current_device()) == hk.HK_OK


def test_attention_torch_helper(hk, oracle):
    import torch
    Q, K, V = _inputs(1, 4, 2, 200, 64, 51)
    o, lse = hk.attention(_dev(Q), _dev(K), _dev(V), causal=True, return_lse=True)
    torch.cuda.synchronize()
    want, want_lse = oracle.attention_fwd(Q, K, V, causal=True, with_lse=True)
    check_heads(_host(o), want, Q, K, V, True, what="torch helper")
    check_lse(lse.cpu().numpy().astype(np.float64), want_lse, "torch helper")
