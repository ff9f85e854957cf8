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
