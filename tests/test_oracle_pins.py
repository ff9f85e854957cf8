"""Pins of the fp64 oracle against what the pages and the mathematics fix (CPU only).

Each test checks the oracle against something other than itself: a value printed on a page,
a closed form, an algebraic identity, an invariance, or an independent formulation (matrix
form with the relative-shift pad-and-reshape) that a plausible slip in the oracle (dropped
term, wrong sign of the distance, wrong head slice, transposed W_R, wrong frequency exponent,
unmasked key) would break.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- sinusoid R_delta
def test_worked_example_r_minus_2():
    """跨窗口的相对位置编码 §2: R_{-2} for d = 4 is printed as [-0.909, -0.416, -0.020, 0.999]."""
    g = json.load(open(os.path.join(GOLDEN, "sinusoid_worked_example.json")))
    R = oracle.sinusoid(g["delta"], g["d"])
    assert np.all(np.abs(R - np.array(g["printed"])) <= g["bound"] + 1e-12)
    # the page also prints the arguments: sin(-2), cos(-2), sin(-0.02), cos(-0.02)
    args = g["printed_arguments"]
    assert R[0] == pytest.approx(math.sin(args["R^(0)"]), abs=1e-15)
    assert R[1] == pytest.approx(math.cos(args["R^(1)"]), abs=1e-15)
    assert R[2] == pytest.approx(math.sin(args["R^(2)"]), abs=1e-15)
    assert R[3] == pytest.approx(math.cos(args["R^(3)"]), abs=1e-15)


@pytest.mark.parametrize("d_model", [4, 16, 410, 1024])
def test_sinusoid_closed_forms(d_model):
    R0 = oracle.sinusoid(0.0, d_model)
    assert np.array_equal(R0[0::2], np.zeros(d_model // 2))
    assert np.array_equal(R0[1::2], np.ones(d_model // 2))
    for delta in [1.0, 7.0, 300.0, 1000.0]:
        R = oracle.sinusoid(delta, d_model)
        Rn = oracle.sinusoid(-delta, d_model)
        assert np.allclose(R[0::2] ** 2 + R[1::2] ** 2, 1.0, atol=1e-14, rtol=0)
        assert np.allclose(Rn[0::2], -R[0::2], atol=1e-15, rtol=0)   # sine part is odd
        assert np.allclose(Rn[1::2], R[1::2], atol=1e-15, rtol=0)    # cosine part is even
    # frequencies: the angle at delta = 1 for pair k is 10000^(-2k/d_model); the first is 1
    # and the ratio between neighbours is the constant 10000^(-2/d_model)
    R1 = oracle.sinusoid(1.0, d_model)
    w = np.arctan2(R1[0::2], R1[1::2])
    assert w[0] == pytest.approx(1.0, abs=1e-14)
    assert np.allclose(w[1:] / w[:-1], 10000.0 ** (-2.0 / d_model), rtol=1e-12, atol=0)
    assert w[-1] == pytest.approx(10000.0 ** (-(d_model - 2) / d_model), rel=1e-12)


def test_rel_table_head_slicing_and_projection():
    """With d_model = H*D and W_R = I, r[delta][h][d] is R_delta[h*D + d]; with a random W_R it
    is the sinusoid row times W_R (a library matmul on an independently built table)."""
    H, D, n = 3, 4, 9
    dm = H * D
    r = oracle.rel_table(n, dm, H, D, np.eye(dm))
    for delta in range(n):
        assert np.array_equal(r[delta].reshape(-1), oracle.sinusoid(delta, dm))
    rng = np.random.default_rng(0)
    W = rng.standard_normal((dm, H * D + 5))       # padded row stride
    r = oracle.rel_table(n, dm, H, D, W)
    pos = np.arange(n, dtype=np.float64)[:, None]
    inv = 10000.0 ** (-np.arange(0, dm, 2, dtype=np.float64) / dm)
    tab = np.empty((n, dm))
    tab[:, 0::2] = np.sin(pos * inv)
    tab[:, 1::2] = np.cos(pos * inv)
    ref = (tab @ W[:, : H * D]).reshape(n, H, D)
    assert np.allclose(r, ref, rtol=0, atol=1e-12)


# ---------------------------------------------------------------- four-term score
def test_four_terms_equal_absolute_expansion():
    """TransformerXL 相对位置编码 §2.1 / Transformer-XL 和相对位置编码 §2.3.2: replacing the
    relative pieces by absolute ones (r := W_k U_j, u = v := W_q U_i) turns the four-term sum
    into (W_q(E_i+U_i))^T W_k (E_j+U_j), term by term (a)-(d)."""
    rng = np.random.default_rng(1)
    n, D = 12, 8
    Wq, Wk = rng.standard_normal((D, n)), rng.standard_normal((D, n))
    for _ in range(20):
        Ei, Ej, Ui, Uj = (rng.standard_normal(n) for _ in range(4))
        q, k, r, uv = Wq @ Ei, Wk @ Ej, Wk @ Uj, Wq @ Ui
        s, terms = oracle.score_terms(q, k, r, uv, uv)
        absolute = (Wq @ (Ei + Ui)) @ (Wk @ (Ej + Uj))
        assert s == pytest.approx(absolute, rel=1e-12, abs=1e-12)
        assert terms[0] == pytest.approx(Ei @ Wq.T @ Wk @ Ej, rel=1e-12, abs=1e-12)
        assert terms[1] == pytest.approx(Ei @ Wq.T @ Wk @ Uj, rel=1e-12, abs=1e-12)
        assert terms[2] == pytest.approx(Ui @ Wq.T @ Wk @ Ej, rel=1e-12, abs=1e-12)
        assert terms[3] == pytest.approx(Ui @ Wq.T @ Wk @ Uj, rel=1e-12, abs=1e-12)


# ---------------------------------------------------------------- helpers
def _rand_case(rng, B, H, D, dm, L, M):
    q = rng.standard_normal((B, L, H, D))
    k = rng.standard_normal((B, M + L, H, D))
    v = rng.standard_normal((B, M + L, H, D))
    u = 0.5 * rng.standard_normal((H, D))
    vb = 0.5 * rng.standard_normal((H, D))
    W = rng.standard_normal((dm, H * D)) / math.sqrt(dm)
    return q, k, v, u, vb, W


def _visible(M, mem_valid, L):
    i = np.arange(L)[:, None]
    j = np.arange(M + L)[None, :]
    return (j >= M - mem_valid) & (j <= M + i)


def _softmax_rows(S, vis):
    S = np.where(vis, S, -np.inf)
    S = S - S.max(axis=-1, keepdims=True)
    P = np.exp(S)
    return P / P.sum(axis=-1, keepdims=True)


def _skew_reference(q, k, v, u, vb, W, M, mem_valid, C, scale):
    """Independent matrix formulation: AC = (Q+u)K^T; BD = (Q+v) r_desc^T over keys in
    decreasing distance, then the relative shift by zero-pad + reshape (the engineering trick
    the qidao123 page names "Relative Shift"); mask; softmax; PV."""
    B, L, H, D = q.shape
    K = M + L
    dm = W.shape[0]
    inv = 10000.0 ** (-np.arange(0, dm, 2, dtype=np.float64) / dm)
    dist = np.minimum(np.arange(K - 1, -1, -1, dtype=np.float64), C)   # K-1 ... 0, clamped
    tab = np.empty((K, dm))
    tab[:, 0::2] = np.sin(dist[:, None] * inv)
    tab[:, 1::2] = np.cos(dist[:, None] * inv)
    rdesc = (tab @ W[:, : H * D]).reshape(K, H, D)
    vis = _visible(M, mem_valid, L)
    out = np.zeros_like(q)
    for b in range(B):
        for h in range(H):
            Q = q[b, :, h]
            AC = (Q + u[h]) @ k[b, :, h].T                       # [L, K]
            raw = (Q + vb[h]) @ rdesc[:, h].T                    # [L, K], column c: dist K-1-c
            padded = np.concatenate([np.zeros((L, 1)), raw], axis=1)   # [L, K+1]
            BD = padded.reshape(K + 1, L)[1:].reshape(L, K)      # shift row i left by L-1-i
            P = _softmax_rows(scale * (AC + BD), vis)
            out[b, :, h] = P @ v[b, :, h]
    return out


# ---------------------------------------------------------------- full-path pins
@pytest.mark.parametrize("shape", [
    dict(B=2, H=3, D=8, dm=12, L=5, M=7, mv=7, C=100),
    dict(B=1, H=2, D=4, dm=6, L=6, M=0, mv=0, C=100),
    dict(B=1, H=2, D=6, dm=8, L=4, M=9, mv=5, C=100),
    dict(B=2, H=1, D=5, dm=10, L=7, M=6, mv=6, C=3),
    dict(B=1, H=2, D=8, dm=16, L=8, M=8, mv=8, C=0),
])
def test_matches_relative_shift_matrix_form(shape):
    rng = np.random.default_rng(2)
    s = shape
    q, k, v, u, vb, W = _rand_case(rng, s["B"], s["H"], s["D"], s["dm"], s["L"], s["M"])
    scale = 1.0 / math.sqrt(s["D"])
    got = oracle.rel_attn(q, k, v, u, vb, W, s["M"], s["mv"], s["C"])
    ref = _skew_reference(q, k, v, u, vb, W, s["M"], s["mv"], s["C"], scale)
    assert np.allclose(got, ref, rtol=0, atol=1e-11)


def test_reduces_to_textbook_attention():
    """u = v = 0 and W_R = 0 leave softmax(QK^T/sqrt(d)) V with the causal-with-memory mask
    (跨窗口的相对位置编码 §3; Transformer-XL 和相对位置编码 §1)."""
    rng = np.random.default_rng(3)
    B, H, D, dm, L, M, mv = 2, 2, 8, 10, 6, 5, 4
    q, k, v, _, _, _ = _rand_case(rng, B, H, D, dm, L, M)
    z = np.zeros((H, D))
    got = oracle.rel_attn(q, k, v, z, z, np.zeros((dm, H * D)), M, mv, 1000)
    vis = _visible(M, mv, L)
    ref = np.zeros_like(q)
    for b in range(B):
        for h in range(H):
            P = _softmax_rows(q[b, :, h] @ k[b, :, h].T / math.sqrt(D), vis)
            ref[b, :, h] = P @ v[b, :, h]
    assert np.allclose(got, ref, rtol=0, atol=1e-12)


def test_translation_invariance():
    """TransformerXL 相对位置编码 §1.3: moving every absolute position by t0 changes nothing.
    Prepending t0 invisible memory slots shifts all positions and keeps each distance."""
    rng = np.random.default_rng(4)
    B, H, D, dm, L, M = 1, 2, 6, 8, 5, 4
    q, k, v, u, vb, W = _rand_case(rng, B, H, D, dm, L, M)
    base = oracle.rel_attn(q, k, v, u, vb, W, M, M, 1000)
    for t0 in [1, 3, 17]:
        junk_k = 100.0 * rng.standard_normal((B, t0, H, D))
        junk_v = 100.0 * rng.standard_normal((B, t0, H, D))
        k2 = np.concatenate([junk_k, k], axis=1)
        v2 = np.concatenate([junk_v, v], axis=1)
        shifted = oracle.rel_attn(q, k2, v2, u, vb, W, M + t0, M, 1000)
        assert np.allclose(shifted, base, rtol=0, atol=1e-13)


def test_clamp_makes_far_distances_identical():
    """TransformerXL 相对位置编码 §2.4: every distance beyond the window counts as the window
    edge.  With q = 0 and u = 0 the score depends on the distance alone, so all keys at
    distance >= C get exactly the same weight."""
    rng = np.random.default_rng(5)
    B, H, D, dm, L, M, C = 1, 1, 8, 8, 6, 10, 3
    _, _, _, u, vb, W = _rand_case(rng, B, H, D, dm, L, M)
    k = rng.standard_normal((B, M + L, H, D))
    Dv = M + L
    # value of key j is the unit vector e_j, so out[i] is the probability row of query i
    v = np.zeros((B, M + L, H, Dv))
    for j in range(M + L):
        v[0, j, 0, j] = 1.0
    qq = np.zeros((B, L, H, Dv))
    kk = np.zeros((B, M + L, H, Dv))
    kk[..., :D] = k
    uu = np.zeros((H, Dv))
    vv = np.zeros((H, Dv))
    vv[:, :D] = vb
    WW = np.zeros((dm, H * Dv))
    WW[:, :D] = W
    P = oracle.rel_attn(qq, kk, v, uu, vv, WW, M, M, C)[0, :, 0, :]
    for i in range(L):
        far = [j for j in range(M + i + 1) if M + i - j >= C]
        assert len(far) >= 2
        assert np.allclose(P[i, far], P[i, far[0]], rtol=1e-14, atol=0)
        assert np.sum(P[i]) == pytest.approx(1.0, abs=1e-14)
        assert np.all(P[i, M + i + 1:] == 0.0)
    assert not np.allclose(P[L - 1, M + L - 1], P[L - 1, M + L - 2])   # near ones do differ


def test_clamp_zero_removes_position_dependence():
    rng = np.random.default_rng(6)
    B, H, D, dm, L, M = 2, 2, 8, 12, 5, 6
    q, k, v, u, vb, W = _rand_case(rng, B, H, D, dm, L, M)
    a = oracle.rel_attn(q, k, v, u, vb, W, M, M, 0)
    b = oracle.rel_attn(q, k, v, u, 3.0 * rng.standard_normal((H, D)),
                        rng.standard_normal(W.shape), M, M, 0)
    assert np.allclose(a, b, rtol=0, atol=1e-12)
    c = oracle.rel_attn(q, k, v, u, vb, W, M, M, M + L - 1)
    d = oracle.rel_attn(q, k, v, u, vb, W, M, M, 10 ** 6)
    assert np.array_equal(c, d)


def test_softmax_invariants_and_masking():
    """TransformerXL 相对位置编码 §4.2: masking applies to the summed score -- masked keys must
    not contribute at all, whatever their content."""
    rng = np.random.default_rng(7)
    B, H, D, dm, L, M, mv = 1, 2, 6, 8, 5, 7, 3
    q, k, v, u, vb, W = _rand_case(rng, B, H, D, dm, L, M)
    ones = oracle.rel_attn(q, k, np.ones_like(v), u, vb, W, M, mv, 1000)
    assert np.allclose(ones, 1.0, rtol=0, atol=1e-14)
    base = oracle.rel_attn(q, k, v, u, vb, W, M, mv, 1000)
    k2, v2 = k.copy(), v.copy()
    k2[:, : M - mv] = 1e3 * rng.standard_normal(k2[:, : M - mv].shape)
    v2[:, : M - mv] = 1e6
    assert np.array_equal(oracle.rel_attn(q, k2, v2, u, vb, W, M, mv, 1000), base)
    for i in range(L):          # future keys of query i do not reach it
        k3, v3 = k.copy(), v.copy()
        k3[:, M + i + 1:] = 1e3
        v3[:, M + i + 1:] = -1e6
        got = oracle.rel_attn(q, k3, v3, u, vb, W, M, mv, 1000)
        assert np.array_equal(got[:, i], base[:, i])
    # no memory, first query: exactly one visible key, so the output is that key's value
    q0, k0, v0, u0, vb0, W0 = _rand_case(rng, 1, 2, 6, 8, 3, 0)
    o = oracle.rel_attn(q0, k0, v0, u0, vb0, W0, 0, 0, 1000)
    assert np.array_equal(o[:, 0], v0[:, 0])


def test_memo_is_the_same_function():
    rng = np.random.default_rng(8)
    q, k, v, u, vb, W = _rand_case(rng, 1, 2, 8, 16, 8, 8)
    a = oracle.rel_attn(q, k, v, u, vb, W, 8, 8, 5, memo=True)
    b = oracle.rel_attn(q, k, v, u, vb, W, 8, 8, 5, memo=False)
    assert np.array_equal(a, b)


def test_row_subset_matches_full():
    rng = np.random.default_rng(9)
    q, k, v, u, vb, W = _rand_case(rng, 2, 3, 8, 16, 6, 4)
    full = oracle.rel_attn(q, k, v, u, vb, W, 4, 4, 1000)
    rows = [(1, 2, 5), (0, 0, 0), (1, 0, 3)]
    part = oracle.rel_attn(q, k, v, u, vb, W, 4, 4, 1000, rows=rows)
    for b, h, i in rows:
        assert np.array_equal(part[b, i, h], full[b, i, h])
    assert np.isnan(part[0, 1, 1]).all()


def test_repeated_rows_in_a_selection():
    """A row listed several times in a multi-threaded selection gets the same value as alone."""
    rng = np.random.default_rng(12)
    q, k, v, u, vb, W = _rand_case(rng, 2, 2, 8, 16, 40, 30)
    row = (1, 1, 33)
    alone = oracle.rel_attn(q, k, v, u, vb, W, 30, 30, 1000, rows=[row], threads=1)
    dup = oracle.rel_attn(q, k, v, u, vb, W, 30, 30, 1000, rows=[row] * 8 + [(0, 0, 1)], threads=8)
    assert np.array_equal(alone[1, 33, 1], dup[1, 33, 1])
    T = 3 * 16
    qs, ks, vs = (rng.standard_normal((2, T, 2, 8)) for _ in range(3))
    alone = oracle.stream_attn(qs, ks, vs, u, vb, W, 16, 20, 1000, rows=[(1, 0, 40)], threads=1)
    dup = oracle.stream_attn(qs, ks, vs, u, vb, W, 16, 20, 1000, rows=[(1, 0, 40)] * 8, threads=8)
    assert np.array_equal(alone[1, 40, 0], dup[1, 40, 0])


# ---------------------------------------------------------------- recurrence and FIFO memory
def test_stream_equals_single_calls_over_fifo_memory():
    """Transformer-XL 和相对位置编码 §2.3.1 + Transformer-XL架构解析 §1.1: segment s attends
    to the cached last min(s*L, M) positions plus itself; the concatenated-sequence definition
    and the per-call definition with a right-aligned, partly valid memory agree."""
    rng = np.random.default_rng(10)
    B, H, D, dm, L, M, S, C = 2, 2, 6, 10, 4, 6, 4, 7
    T = S * L
    q = rng.standard_normal((B, T, H, D))
    k = rng.standard_normal((B, T, H, D))
    v = rng.standard_normal((B, T, H, D))
    u, vb = rng.standard_normal((H, D)), rng.standard_normal((H, D))
    W = rng.standard_normal((dm, H * D)) / math.sqrt(dm)
    st = oracle.stream_attn(q, k, v, u, vb, W, L, M, C)
    for s in range(S):
        mv = min(s * L, M)
        km = np.zeros((B, M + L, H, D))
        vm = np.zeros((B, M + L, H, D))
        km[:, M - mv:M] = k[:, s * L - mv: s * L]
        vm[:, M - mv:M] = v[:, s * L - mv: s * L]
        km[:, M:] = k[:, s * L: (s + 1) * L]
        vm[:, M:] = v[:, s * L: (s + 1) * L]
        one = oracle.rel_attn(q[:, s * L:(s + 1) * L], km, vm, u, vb, W, M, mv, C)
        assert np.allclose(one, st[:, s * L:(s + 1) * L], rtol=0, atol=1e-12)


@pytest.mark.parametrize("M,L,S", [(6, 4, 5), (4, 4, 3), (3, 5, 3), (8, 3, 7), (1, 2, 3)])
def test_ring_keeps_last_m_positions(M, L, S):
    rng = np.random.default_rng(11)
    B = 2
    stream_k = rng.integers(0, 1 << 30, size=(B, S * L, 3))
    stream_v = rng.integers(0, 1 << 30, size=(B, S * L, 3))
    rk = np.zeros((B, M, 3), dtype=stream_k.dtype)
    rv = np.zeros_like(rk)
    wp, valid = 0, 0
    for s in range(S):
        rk, rv, wp, valid = oracle.ring_push(rk, rv, wp, valid, stream_k[:, s * L:(s + 1) * L],
                                             stream_v[:, s * L:(s + 1) * L])
        seen = (s + 1) * L
        assert valid == min(seen, M)
        lk = oracle.ring_logical(rk, wp, valid)
        lv = oracle.ring_logical(rv, wp, valid)
        assert np.array_equal(lk[:, M - valid:], stream_k[:, seen - valid: seen])
        assert np.array_equal(lv[:, M - valid:], stream_v[:, seen - valid: seen])


def test_flop_count_is_visible_pairs():
    for (L, M, mv) in [(5, 7, 7), (384, 384, 384), (128, 1600, 1600), (6, 4, 2), (3, 0, 0)]:
        pairs = int(_visible(M, mv, L).sum())
        assert oracle.attn_flops(1, 1, 1, L, M, mv) == 6 * pairs
