"""Pins of the layer oracle (oracle.rel_layer / oracle.stream_layer: projections with a memory of
hidden states, "Transformer-XL 和相对位置编码" §2.3.1, and the output projection of
"TransformerXL 相对位置编码" §3.1) against facts that do not come from the layer oracle itself: the
pinned attention oracle on explicitly permuted inputs, independence and linearity properties, and
the equivalence of re-projecting the memory's hidden states with projecting each position once
(the pinned segment-recurrence oracle on pre-projected sequences).  CPU only."""
import numpy as np

import oracle


def _weights(rng, dm, H, D, scale=None):
    s = scale if scale is not None else dm ** -0.5
    return [rng.standard_normal((dm, H * D)) * s for _ in range(3)] + [rng.standard_normal((H * D, dm)) * s]


def _small(rng, B=2, L=5, M=4, H=2, D=3, dm=6):
    h = rng.standard_normal((B, L, dm))
    h_mem = rng.standard_normal((B, M, dm))
    u = rng.standard_normal((H, D)) * 0.02
    vb = rng.standard_normal((H, D)) * 0.02
    W_R = rng.standard_normal((dm, H * D)) * dm ** -0.5
    return h, h_mem, u, vb, W_R


def test_permutation_weights_reduce_to_the_attention_oracle():
    """With permutation matrices as W_q, W_k, W_v, W_o (d_model = H*D, none of them its own
    inverse), the layer is the attention oracle on column-permuted inputs, its output permuted:
    this fixes which weight projects q, k and v, that the memory comes first in h~, and that W_o
    is applied as stated (a transposed W_o would apply the inverse permutation)."""
    rng = np.random.default_rng(11)
    B, L, M, H, D = 2, 5, 4, 2, 3
    dm = H * D
    h, h_mem, u, vb, W_R = _small(rng, B, L, M, H, D, dm)
    perms = [np.roll(np.arange(dm), s) for s in (1, 2, 4)] + [np.array([2, 0, 4, 1, 5, 3])]
    mats = []
    for p in perms:
        P = np.zeros((dm, dm))
        P[p, np.arange(dm)] = 1.0          # X @ P takes column j of the result from column p[j]
        mats.append(P)
    y = oracle.rel_layer(h_mem, h, *mats, u, vb, W_R, H, D, M, clamp_len=6)
    h_ext = np.concatenate([h_mem, h], axis=1)
    q = h[:, :, perms[0]].reshape(B, L, H, D)
    k = h_ext[:, :, perms[1]].reshape(B, M + L, H, D)
    v = h_ext[:, :, perms[2]].reshape(B, M + L, H, D)
    a = oracle.rel_attn(q, k, v, u, vb, W_R, M, M, 6).reshape(B, L, dm)
    assert np.allclose(y, a[:, :, perms[3]], rtol=0, atol=1e-12)


def test_invalid_memory_is_not_read_and_valid_memory_is():
    rng = np.random.default_rng(12)
    B, L, M, H, D, dm = 2, 4, 6, 2, 4, 10
    h, h_mem, u, vb, W_R = _small(rng, B, L, M, H, D, dm)
    W = _weights(rng, dm, H, D)
    other = rng.standard_normal(h_mem.shape)
    y0 = oracle.rel_layer(h_mem, h, *W, u, vb, W_R, H, D, 0, clamp_len=8)
    y1 = oracle.rel_layer(other, h, *W, u, vb, W_R, H, D, 0, clamp_len=8)
    assert np.array_equal(y0, y1)
    # with three valid positions, only the last three memory rows matter
    mixed = h_mem.copy()
    mixed[:, :M - 3] = other[:, :M - 3]
    y2 = oracle.rel_layer(h_mem, h, *W, u, vb, W_R, H, D, 3, clamp_len=8)
    y3 = oracle.rel_layer(mixed, h, *W, u, vb, W_R, H, D, 3, clamp_len=8)
    assert np.allclose(y2, y3, rtol=0, atol=1e-13)
    y4 = oracle.rel_layer(other, h, *W, u, vb, W_R, H, D, 3, clamp_len=8)
    assert np.max(np.abs(y4 - y2)) > 1e-3


def test_linear_in_the_value_and_output_weights():
    """The softmax weights depend on W_q, W_k only: scaling W_v scales y, and y is linear in W_o."""
    rng = np.random.default_rng(13)
    B, L, M, H, D, dm = 1, 6, 3, 3, 2, 8
    h, h_mem, u, vb, W_R = _small(rng, B, L, M, H, D, dm)
    Wq, Wk, Wv, Wo = _weights(rng, dm, H, D)
    Wo2 = rng.standard_normal(Wo.shape)
    y = oracle.rel_layer(h_mem, h, Wq, Wk, Wv, Wo, u, vb, W_R, H, D, M, clamp_len=5)
    y2 = oracle.rel_layer(h_mem, h, Wq, Wk, Wv, Wo2, u, vb, W_R, H, D, M, clamp_len=5)
    ys = oracle.rel_layer(h_mem, h, Wq, Wk, Wv, Wo + Wo2, u, vb, W_R, H, D, M, clamp_len=5)
    assert np.allclose(ys, y + y2, rtol=0, atol=1e-12)
    yv = oracle.rel_layer(h_mem, h, Wq, Wk, -2.5 * Wv, Wo, u, vb, W_R, H, D, M, clamp_len=5)
    assert np.allclose(yv, -2.5 * y, rtol=0, atol=1e-12)
    # W_q, W_k do enter the weights: scaling W_k changes y non-linearly
    yk = oracle.rel_layer(h_mem, h, Wq, 3.0 * Wk, Wv, Wo, u, vb, W_R, H, D, M, clamp_len=5)
    assert np.max(np.abs(yk - y)) > 1e-3


def test_reprojected_hidden_memory_equals_projecting_each_position_once():
    """Re-projecting the memory's hidden states at every segment (the recurrence as the pages
    write it) gives the segment-recurrence attention oracle over the whole sequence projected once
    (the reading that lets the memory cache projected keys and values)."""
    rng = np.random.default_rng(14)
    B, L, M, S, H, D, dm = 2, 4, 6, 3, 2, 4, 8
    h_all = rng.standard_normal((B, S * L, dm))
    u = rng.standard_normal((H, D)) * 0.02
    vb = rng.standard_normal((H, D)) * 0.02
    W_R = rng.standard_normal((dm, H * D)) * dm ** -0.5
    Wq, Wk, Wv, Wo = _weights(rng, dm, H, D)
    y = oracle.stream_layer(h_all, Wq, Wk, Wv, Wo, u, vb, W_R, H, D, L, M, clamp_len=7)
    T = S * L
    q = (h_all @ Wq).reshape(B, T, H, D)
    k = (h_all @ Wk).reshape(B, T, H, D)
    v = (h_all @ Wv).reshape(B, T, H, D)
    a = oracle.stream_attn(q, k, v, u, vb, W_R, L, M, 7).reshape(B, T, H * D)
    assert np.allclose(y, a @ Wo, rtol=0, atol=1e-12)


def test_layer_flops():
    assert oracle.layer_flops(2, 3, 4, 5, 6, 7) == 2 * 2 * 5 * 7 * 4 * 12 + oracle.attn_flops(2, 3, 4, 5, 6)
