"""Pins of the learned-table variant oracle (oracle.table_attn, "TransformerXL 相对位置编码" §3.1) against
a plain softmax attention written here with numpy, closed forms of the index and the clamp, and the
masking rule of that page.  CPU only."""
import math

import numpy as np

import oracle


def _plain(q, k, v, scale, key_bias=None, mask=None):
    """softmax(scale q k^T + key_bias) v per (b, h), straight from the textbook definition."""
    B, L, H, D = q.shape
    out = np.empty_like(q)
    for b in range(B):
        for h in range(H):
            s = scale * q[b, :, h] @ k[b, :, h].T
            if key_bias is not None:
                s = s + key_bias[b, h][None, :]
            if mask is not None:
                s = np.where(mask[b][None, :] == 0, -1e9, s)
            e = np.exp(s - s.max(axis=1, keepdims=True))
            out[b, :, h] = (e / e.sum(axis=1, keepdims=True)) @ v[b, :, h]
    return out


def _rand(seed, B=2, L=6, H=2, D=4, max_len=8):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((B, L, H, D)), rng.standard_normal((B, L, H, D)), rng.standard_normal((B, L, H, D)),
            rng.standard_normal((H, D)) * 0.3, rng.standard_normal((H, D)) * 0.3,
            rng.standard_normal((2 * max_len - 1, H, D)))


def test_zero_table_is_textbook_attention_with_a_key_bias():
    q, k, v, u, vb, rt = _rand(1)
    D = q.shape[-1]
    got = oracle.table_attn(q, k, v, u, vb, np.zeros_like(rt), 8)
    bias = np.einsum("bjhd,hd->bhj", k, u)                  # term (c), unscaled
    assert np.allclose(got, _plain(q, k, v, 1 / math.sqrt(D), key_bias=bias), atol=1e-12)
    got0 = oracle.table_attn(q, k, v, np.zeros_like(u), vb, np.zeros_like(rt), 8)
    assert np.allclose(got0, _plain(q, k, v, 1 / math.sqrt(D)), atol=1e-12)


def test_one_row_table_changes_nothing():
    """max_len = 1: every pair reads row 0, so terms (b) and (d) are constant along each row."""
    q, k, v, u, vb, rt = _rand(2, max_len=1)
    got = oracle.table_attn(q, k, v, u, vb, rt, 1)
    ref = oracle.table_attn(q, k, v, u, vb, np.zeros_like(rt), 1)
    assert np.allclose(got, ref, atol=1e-12)


def test_index_sign_and_clamp():
    """With only term (d) (q = k = 0, u = 0) and a steep table rising with its index, each query puts
    its weight on the keys with the largest index clamp(i - j + max_len - 1, 0, 2 max_len - 2): for
    max_len = 3 that is key 0 alone while i - j + 2 < 4 (queries 0, 1), and for i >= 2 every key
    j <= i - 2, all clamped to the last row, equally (out = their mean value j)."""
    B, L, H, D, max_len = 1, 7, 1, 1, 3
    q = np.zeros((B, L, H, D))
    k = np.zeros((B, L, H, D))
    v = np.arange(L, dtype=np.float64).reshape(B, L, H, D)
    u = np.zeros((H, D))
    vb = np.ones((H, D))
    rt = (60.0 * np.arange(2 * max_len - 1, dtype=np.float64)).reshape(-1, 1, 1)
    out = oracle.table_attn(q, k, v, u, vb, rt, max_len)[0, :, 0, 0]
    expect = [0.0, 0.0] + [(i - 2) / 2.0 for i in range(2, L)]
    assert np.allclose(out, expect, atol=1e-9), out


def test_masking_follows_the_page():
    q, k, v, u, vb, rt = _rand(3)
    mask = np.ones((2, 6), dtype=np.int64)
    mask[0, [1, 4]] = 0
    mask[1, :] = 0                                           # every key masked: uniform weights
    got = oracle.table_attn(q, k, v, u, vb, rt, 8, key_mask=mask)
    # batch 0: the masked keys' weights underflow to exactly zero; the rest is the page's score
    # evaluated pair by pair over the kept keys
    keep = [0, 2, 3, 5]
    B, L, H, D = q.shape
    rel = np.clip(np.arange(L)[:, None] - np.arange(L)[None, :] + 7, 0, 14)
    for h in range(H):
        for i in range(L):
            s = np.array([(q[0, i, h] @ k[0, j, h] + q[0, i, h] @ rt[rel[i, j], h]) / math.sqrt(D) + u[h] @ k[0, j, h]
                          + vb[h] @ rt[rel[i, j], h] for j in keep])
            w = np.exp(s - s.max())
            w /= w.sum()
            assert np.allclose(got[0, i, h], w @ v[0, keep, h], atol=1e-12)
    assert np.allclose(got[1], np.broadcast_to(v[1].mean(axis=0), got[1].shape), atol=1e-12)
