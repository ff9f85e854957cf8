"""Pins of the backward oracle (oracle.rel_attn_bwd) against the pinned forward oracle: every
gradient entry equals the central finite difference of the forward's loss sum(dO * out) (fp64,
step 1e-6, agreement to 1e-7), on tiny shapes that exercise a partly valid memory and the clamp;
plus the softmax shift invariance of the key gradient.  CPU only."""
import numpy as np
import pytest

import oracle


def _case(seed, B=2, L=3, M=2, H=2, D=3, dm=4):
    rng = np.random.default_rng(seed)
    return dict(q=rng.standard_normal((B, L, H, D)), k=rng.standard_normal((B, M + L, H, D)),
                v=rng.standard_normal((B, M + L, H, D)), u=rng.standard_normal((H, D)) * 0.3,
                vb=rng.standard_normal((H, D)) * 0.3, W_R=rng.standard_normal((dm, H * D)) * 0.7,
                dO=rng.standard_normal((B, L, H, D)))


def _loss(c, M, valid, C):
    out = oracle.rel_attn(c["q"], c["k"], c["v"], c["u"], c["vb"], c["W_R"], M, valid, C, memo=False)
    return float(np.sum(c["dO"] * out))


@pytest.mark.parametrize("M,valid,C", [(2, 2, 10), (2, 1, 3), (0, 0, 1)])
def test_gradients_match_finite_differences(M, valid, C):
    c = _case(5 + M + valid + C, M=M)
    g = oracle.rel_attn_bwd(c["q"], c["k"], c["v"], c["u"], c["vb"], c["W_R"], M, valid, C, c["dO"])
    names = {"q": "dq", "k": "dk", "v": "dv", "u": "du", "vb": "dvb", "W_R": "dW_R"}
    eps = 1e-6
    for x, gname in names.items():
        a = c[x]
        fd = np.empty_like(a)
        for idx in np.ndindex(a.shape):
            keep = a[idx]
            a[idx] = keep + eps
            lp = _loss(c, M, valid, C)
            a[idx] = keep - eps
            lm = _loss(c, M, valid, C)
            a[idx] = keep
            fd[idx] = (lp - lm) / (2 * eps)
        err = np.max(np.abs(fd - g[gname]))
        assert err <= 1e-7 * max(1.0, np.max(np.abs(fd))), (x, err)


def test_key_gradient_sums_to_zero():
    """Adding one vector to every key adds the same amount to a query's scores over all keys, which
    the softmax ignores: the key gradients of each (b, h) sum to zero (masked keys contribute 0)."""
    c = _case(21, B=2, L=4, M=3, H=2, D=5, dm=6)
    g = oracle.rel_attn_bwd(c["q"], c["k"], c["v"], c["u"], c["vb"], c["W_R"], 3, 2, 4, c["dO"])
    assert np.allclose(g["dk"].sum(axis=1), 0.0, atol=1e-12)
    assert np.all(g["dk"][:, 0] == 0.0) and np.all(g["dv"][:, 0] == 0.0)      # the invalid memory key


def test_value_gradients_sum_to_the_upstream_gradient():
    """Every row of P sums to one, so the value gradients dv_j = sum_i P_ij dO_i of one (b, h),
    summed over all its keys (memory included), equal sum_i dO_i."""
    c = _case(33, B=2, L=5, M=4, H=3, D=4, dm=6)
    g = oracle.rel_attn_bwd(c["q"], c["k"], c["v"], c["u"], c["vb"], c["W_R"], 4, 3, 6, c["dO"])
    assert np.allclose(g["dv"].sum(axis=1), c["dO"].sum(axis=1), atol=1e-12)


def test_clamp_zero_leaves_no_position_bias_gradient():
    """With clamp_len 0 every pair uses r[0]: the position term (q + v_bias) . r[0] is the same for all
    keys of a query and the softmax ignores it, so v_bias gets no gradient, and dr puts the whole
    gradient of that term, which is zero, on row 0."""
    c = _case(44, B=2, L=4, M=3, H=2, D=3, dm=4)
    g = oracle.rel_attn_bwd(c["q"], c["k"], c["v"], c["u"], c["vb"], c["W_R"], 3, 3, 0, c["dO"])
    assert np.max(np.abs(g["dvb"])) <= 1e-12
    assert np.max(np.abs(g["dr"])) <= 1e-12


@pytest.mark.parametrize("M,valid,C", [(2, 2, 10), (2, 1, 3), (0, 0, 1)])
def test_log_sum_exp_matches_pairwise_scores(M, valid, C):
    """oracle.rel_attn_lse against a brute-force sum over the visible keys of each row, each score
    from the C oracle's four-term score (score_terms), in log2 units; and the weights
    2^(log2(e) s_ij - lse_i) it implies reproduce the forward oracle's output."""
    import math
    c = _case(40 + M + valid + C, M=M)
    B, L, H, D = c["q"].shape
    scale = 1.0 / math.sqrt(D)
    lse = oracle.rel_attn_lse(c["q"], c["k"], c["u"], c["vb"], c["W_R"], M, valid, C)
    out = oracle.rel_attn(c["q"], c["k"], c["v"], c["u"], c["vb"], c["W_R"], M, valid, C, memo=False)
    n_rows = min(M + L, C + 1)
    r = oracle.rel_table(n_rows, c["W_R"].shape[0], H, D, c["W_R"])
    for b in range(B):
        for h in range(H):
            for i in range(L):
                js = [j for j in range(M - valid, M + L) if M + i - j >= 0]
                s2 = {j: math.log2(math.e) * scale * oracle.score_terms(
                    c["q"][b, i, h], c["k"][b, j, h], r[min(M + i - j, C), h], c["u"][h], c["vb"][h])[0] for j in js}
                mx = max(s2.values())
                want = mx + math.log2(math.fsum(2.0 ** (x - mx) for x in s2.values()))
                assert abs(lse[b, i, h] - want) <= 1e-12 * max(1.0, abs(want))
                o = sum(2.0 ** (s2[j] - lse[b, i, h]) * c["v"][b, j, h] for j in js)
                assert np.max(np.abs(o - out[b, i, h])) <= 1e-12
