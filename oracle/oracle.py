"""ctypes front end of the fp64 C oracle (``txl_oracle.c``) and the FIFO memory semantics.

TEST INFRASTRUCTURE ONLY -- see the package docstring.  All arithmetic of the method lives in
``txl_oracle.c``; this module only converts arrays to float64 and passes pointers, except for
``ring_push``/``ring_logical``, which restate the FIFO memory of "Transformer-XL架构解析" §1.1
(the newest segment evicts the oldest cached positions) with plain per-position loops.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "txl_oracle.c")
_SO = os.path.join(_HERE, "_txl_oracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into ``oracle/_txl_oracle.so`` (host-specific, git-ignored)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + ".tmp%d" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm", "-lpthread"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


def library():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_SO)
            lib.txlo_sinusoid.argtypes = [ctypes.c_double, ctypes.c_int, _dp]
            lib.txlo_sinusoid.restype = None
            lib.txlo_rel_table.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           _dp, ctypes.c_int64, _dp]
            lib.txlo_rel_table.restype = None
            lib.txlo_score_terms.argtypes = [ctypes.c_int, _dp, _dp, _dp, _dp, _dp, _dp]
            lib.txlo_score_terms.restype = ctypes.c_double
            lib.txlo_rel_attn.argtypes = [ctypes.c_int] * 8 + [_dp] * 6 + [
                ctypes.c_int64, ctypes.c_double, _dp, ctypes.c_int, ctypes.c_int, _ip, ctypes.c_int64]
            lib.txlo_rel_attn.restype = ctypes.c_int
            lib.txlo_stream_attn.argtypes = [ctypes.c_int] * 8 + [_dp] * 6 + [
                ctypes.c_int64, ctypes.c_double, _dp, ctypes.c_int, ctypes.c_int, _ip, ctypes.c_int64]
            lib.txlo_stream_attn.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    """float64, C-contiguous copy of a numpy array or a CPU torch tensor (bf16 upcast exactly)."""
    if hasattr(a, "detach"):
        a = a.detach().to("cpu")
        import torch  # local: only when a tensor is passed
        a = a.to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _p(a: np.ndarray):
    return a.ctypes.data_as(_dp)


def _threads(n):
    return int(n) if n else (os.cpu_count() or 1)


def sinusoid(delta: float, d_model: int) -> np.ndarray:
    out = np.empty(d_model, dtype=np.float64)
    library().txlo_sinusoid(float(delta), int(d_model), _p(out))
    return out


def rel_table(n_rows: int, d_model: int, H: int, D: int, W_R) -> np.ndarray:
    """r[delta][h][d] = sum_m R_delta[m] W_R[m][h*D+d] for delta = 0..n_rows-1."""
    W = _f64(W_R)
    assert W.shape[0] == d_model and W.shape[1] >= H * D
    out = np.empty((n_rows, H, D), dtype=np.float64)
    library().txlo_rel_table(n_rows, d_model, H, D, _p(W), W.shape[1], _p(out))
    return out


def score_terms(q, k, r, u, v):
    """Four-term relative score for explicit vectors; returns (sum, [a, b, c, d])."""
    q, k, r, u, v = (_f64(x).reshape(-1) for x in (q, k, r, u, v))
    D = q.shape[0]
    terms = np.empty(4, dtype=np.float64)
    s = library().txlo_score_terms(D, _p(q), _p(k), _p(r), _p(u), _p(v), _p(terms))
    return s, terms


def _sel(rows):
    if rows is None:
        return None, 0
    sel = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 3))
    return sel, sel.shape[0]


def rel_attn(q, k, v, u, vb, W_R, M: int, mem_valid: int, clamp_len: int, scale=None,
             memo: bool = True, threads=None, rows=None) -> np.ndarray:
    """One call over [memory ++ current].

    q [B,L,H,D]; k, v [B,M+L,H,D] in logical order (memory first); u, vb [H,D];
    W_R [d_model, >=H*D].  ``rows``: optional (b, h, i) triples; other rows come back NaN.
    """
    q, k, v, u, vb, W = (_f64(x) for x in (q, k, v, u, vb, W_R))
    B, L, H, D = q.shape
    assert k.shape == (B, M + L, H, D) and v.shape == k.shape
    d_model = W.shape[0]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    out = np.full((B, L, H, D), np.nan, dtype=np.float64)
    sel, n_sel = _sel(rows)
    rc = library().txlo_rel_attn(
        B, L, H, D, M, mem_valid, clamp_len, d_model, _p(q), _p(k), _p(v), _p(u), _p(vb), _p(W),
        W.shape[1], float(scale), _p(out), int(bool(memo)), _threads(threads),
        sel.ctypes.data_as(_ip) if sel is not None else None, n_sel)
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return out


def stream_attn(q, k, v, u, vb, W_R, L: int, M: int, clamp_len: int, scale=None,
                memo: bool = True, threads=None, rows=None) -> np.ndarray:
    """Segment recurrence evaluated on the concatenated sequence.

    q, k, v [B, S*L, H, D] hold all S segments back to back.  A query at global position t
    (segment s = t // L) sees keys g in [max(0, s*L - M), t] with distance t - g.
    ``rows``: optional (b, h, t) triples.
    """
    q, k, v, u, vb, W = (_f64(x) for x in (q, k, v, u, vb, W_R))
    B, T, H, D = q.shape
    assert T % L == 0
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    out = np.full((B, T, H, D), np.nan, dtype=np.float64)
    sel, n_sel = _sel(rows)
    rc = library().txlo_stream_attn(
        B, H, D, L, M, T // L, clamp_len, W.shape[0], _p(q), _p(k), _p(v), _p(u), _p(vb), _p(W),
        W.shape[1], float(scale), _p(out), int(bool(memo)), _threads(threads),
        sel.ctypes.data_as(_ip) if sel is not None else None, n_sel)
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return out


def ring_push(ring_k: np.ndarray, ring_v: np.ndarray, wp: int, valid: int, k_new: np.ndarray,
              v_new: np.ndarray):
    """FIFO memory of M positions ("Transformer-XL架构解析" §1.1: the newest segment's states
    evict the oldest).  ring_* [B, M, ...] hold position slots; the oldest valid position is at
    slot ``wp`` once the ring is full.  Returns (ring_k, ring_v, wp, valid) after appending the
    L positions of k_new/v_new [B, L, ...], one position at a time, oldest first."""
    ring_k = ring_k.copy()
    ring_v = ring_v.copy()
    M = ring_k.shape[1]
    L = k_new.shape[1]
    for t in range(L):
        if M == 0:
            break
        ring_k[:, wp] = k_new[:, t]
        ring_v[:, wp] = v_new[:, t]
        wp = (wp + 1) % M
        valid = min(valid + 1, M)
    return ring_k, ring_v, wp, valid


def ring_logical(ring: np.ndarray, wp: int, valid: int) -> np.ndarray:
    """Logical memory [B, M, ...]: index M-1 is the newest position, M-valid the oldest valid
    one; positions below M-valid are not valid (returned as zeros)."""
    M = ring.shape[1]
    out = np.zeros_like(ring)
    for j in range(M - valid, M):
        out[:, j] = ring[:, (wp + j) % M]
    return out


def rel_attn_bwd(q, k, v, u, vb, W_R, M: int, mem_valid: int, clamp_len: int, dO, scale=None,
                 bh=None) -> dict:
    """Gradients of one call of ``rel_attn`` with respect to q, k, v, u, v_bias, the position
    rows r and W_R, for an upstream gradient dO [B, L, H, D] (chain rule through the four-term
    score of "Transformer-XL 和相对位置编码" §2.3.2 and the softmax; no gradient is formed for
    anything the pages put behind stop-gradient: that is the caller's choice of which slices of
    dk, dv to use).  Plain fp64 linear algebra per (b, h): scores S = scale (q' K^T + BD) with
    q' = q + u, q'' = q + v_bias and BD[i, j] = q''_i . r[min(M + i - j, C)]; P = softmax over the
    visible keys; dP = dO V^T; dS = P (dP - rowsum(P dP)) * scale; then

        dq_i = sum_j dS_ij (k_j + r[delta_ij]),   dk_j = sum_i dS_ij q'_i,   dv_j = sum_i P_ij dO_i,
        du   = sum_{b,i,j} dS_ij k_j,              dv_bias = sum_{b,i,j} dS_ij r[delta_ij],
        dr[delta] = sum_{b,(i,j): delta_ij = delta} dS_ij q''_i,   dW_R = sum_delta R_delta^T dr[delta].

    The position term is handled through E[i, delta] = sum over keys j with clamped distance delta
    of dS_ij, a scatter written out with np.add.at.  ``bh``: optional list of (b, h) pairs to
    evaluate (dq, dk, dv of the others come back NaN; du, dv_bias, dr, dW_R then cover only them).
    Returns float64 arrays: dq [B,L,H,D], dk, dv [B,M+L,H,D], du, dvb [H,D], dr [n_rows,H,D],
    dW_R [d_model, H*D]."""
    q, k, v, u, vb, W, dO = (_f64(x) for x in (q, k, v, u, vb, W_R, dO))
    B, L, H, D = q.shape
    T = M + L
    d_model = W.shape[0]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    n_rows = min(T, clamp_len + 1)
    r = rel_table(n_rows, d_model, H, D, W)                       # [n_rows, H, D]
    i_idx = np.arange(L)[:, None]
    j_idx = np.arange(T)[None, :]
    delta = M + i_idx - j_idx
    vis = (j_idx >= M - mem_valid) & (delta >= 0)
    dcl = np.clip(np.minimum(delta, clamp_len), 0, n_rows - 1)
    out = {"dq": np.full((B, L, H, D), np.nan), "dk": np.full((B, T, H, D), np.nan),
           "dv": np.full((B, T, H, D), np.nan), "du": np.zeros((H, D)), "dvb": np.zeros((H, D)),
           "dr": np.zeros((n_rows, H, D))}
    pairs = bh if bh is not None else [(b, h) for b in range(B) for h in range(H)]
    for b, h in pairs:
        qp = q[b, :, h] + u[h]
        qpp = q[b, :, h] + vb[h]
        K, V, rh, g = k[b, :, h], v[b, :, h], r[:, h], dO[b, :, h]
        G = qpp @ rh.T                                              # [L, n_rows]
        S = scale * (qp @ K.T + np.take_along_axis(G, dcl, axis=1))
        S = np.where(vis, S, -np.inf)
        P = np.exp(S - S.max(axis=1, keepdims=True))
        P /= P.sum(axis=1, keepdims=True)
        dP = g @ V.T
        dS = scale * P * (dP - (P * dP).sum(axis=1, keepdims=True))
        dS = np.where(vis, dS, 0.0)
        E = np.zeros((L, n_rows))
        np.add.at(E, (np.broadcast_to(i_idx, dcl.shape), dcl), dS)
        dq_ac = dS @ K
        dq_bd = E @ rh
        out["dq"][b, :, h] = dq_ac + dq_bd
        out["dk"][b, :, h] = dS.T @ qp
        out["dv"][b, :, h] = P.T @ g
        out["du"][h] += dq_ac.sum(axis=0)
        out["dvb"][h] += dq_bd.sum(axis=0)
        out["dr"][:, h] += E.T @ qpp
    Rm = np.stack([sinusoid(float(dd), d_model) for dd in range(n_rows)])     # [n_rows, d_model]
    out["dW_R"] = Rm.T @ out["dr"].reshape(n_rows, H * D)
    return out


def rel_attn_lse(q, k, u, vb, W_R, M: int, mem_valid: int, clamp_len: int, scale=None) -> np.ndarray:
    """Per query row of one ``rel_attn`` call, the log-sum-exp of its visible scores in log2 units:
    lse[b, i, h] = log2 sum_j 2^(log2(e) S_ij) = log2(e) ln sum_j exp(S_ij), with the scores S of
    ``rel_attn_bwd`` (the four-term score of "Transformer-XL 和相对位置编码" §2.3.2, scaled, over the
    visible keys), i.e. the statistic a forward pass keeps for its backward.  Returns float64
    [B, L, H]."""
    q, k, u, vb, W = (_f64(x) for x in (q, k, u, vb, W_R))
    B, L, H, D = q.shape
    T = M + L
    d_model = W.shape[0]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    n_rows = min(T, clamp_len + 1)
    r = rel_table(n_rows, d_model, H, D, W)
    i_idx = np.arange(L)[:, None]
    j_idx = np.arange(T)[None, :]
    delta = M + i_idx - j_idx
    vis = (j_idx >= M - mem_valid) & (delta >= 0)
    dcl = np.clip(np.minimum(delta, clamp_len), 0, n_rows - 1)
    out = np.empty((B, L, H))
    for b in range(B):
        for h in range(H):
            G = (q[b, :, h] + vb[h]) @ r[:, h].T
            S = scale * ((q[b, :, h] + u[h]) @ k[b, :, h].T + np.take_along_axis(G, dcl, axis=1))
            S = np.where(vis, S, -np.inf)
            m = S.max(axis=1)
            out[b, :, h] = (m + np.log(np.exp(S - m[:, None]).sum(axis=1))) / math.log(2.0)
    return out


def table_attn(q, k, v, u, vb, r_table, max_len: int, key_mask=None, scale=None) -> np.ndarray:
    """The learned-table variant of "TransformerXL 相对位置编码" §3.1 (bidirectional, no memory):
    the relative index rel(i, j) = clamp(i - j + max_len - 1, 0, 2 max_len - 2) selects a row of the
    projected table r_table [2 max_len - 1, H, D] (pos_emb W_R: the projection commutes with the
    lookup); the score is (a) scale q_i.k_j + (b) scale q_i.r_rel + (c) u.k_j + (d) v.r_rel, with the
    scale on terms (a) and (b) only, as that page computes it; keys with key_mask[b, j] == 0 have
    their score replaced by -1e9 before the softmax (so a row whose keys are all masked averages
    every value uniformly); out = softmax . V.  q, k, v [B, L, H, D]; returns fp64 [B, L, H, D]."""
    q, k, v, u, vb, rt = (_f64(x) for x in (q, k, v, u, vb, r_table))
    B, L, H, D = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    pos = np.arange(L)
    rel = np.clip(pos[:, None] - pos[None, :] + max_len - 1, 0, 2 * max_len - 2)     # [L, L]
    out = np.empty((B, L, H, D), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            R = rt[rel, h]                                                       # [L, L, D]
            a = scale * (q[b, :, h] @ k[b, :, h].T)
            bt = scale * np.einsum("id,ijd->ij", q[b, :, h], R)
            c = (k[b, :, h] @ u[h])[None, :]
            d = R @ vb[h]
            s = a + bt + c + d
            if key_mask is not None:
                s = np.where(np.asarray(key_mask)[b][None, :] == 0, -1e9, s)
            p = np.exp(s - s.max(axis=1, keepdims=True))
            p /= p.sum(axis=1, keepdims=True)
            out[b, :, h] = p @ v[b, :, h]
    return out


def linear(X, W) -> np.ndarray:
    """Y = X W in fp64 (a library matmul as the step): q_proj / k_proj / v_proj / o_proj of
    "TransformerXL 相对位置编码" §3.1, linear maps without bias."""
    return _f64(X) @ _f64(W)


def rel_layer(h_mem, h, W_q, W_k, W_v, W_o, u, vb, W_R, H: int, D: int, mem_valid: int,
              clamp_len: int, scale=None, threads=None, rows=None) -> np.ndarray:
    """One attention-layer step with a memory of hidden states, in the order
    "Transformer-XL 和相对位置编码" §2.3.1 gives it: the memory-extended states
    h~ = [SG(h_mem) o h] (memory first, along the sequence), Q = h W_q, K = h~ W_k, V = h~ W_v,
    then the relative attention (``rel_attn``) and the output projection over the concatenated
    heads, y = attn W_o ("TransformerXL 相对位置编码" §3.1).  Stop-gradient has no effect on the
    forward values.

    h_mem [B, M, d_model] (logical order, oldest first; the first M - mem_valid rows are not
    valid), h [B, L, d_model]; W_q, W_k, W_v [d_model, H*D]; W_o [H*D, d_model].  Returns
    y [B, L, d_model] (rows not selected by ``rows`` = (b, h, i) triples come back NaN).
    """
    h_mem, h = _f64(h_mem), _f64(h)
    B, L, dm = h.shape
    M = h_mem.shape[1]
    h_ext = np.concatenate([h_mem, h], axis=1)                   # [B, M+L, d_model]
    q = linear(h, W_q).reshape(B, L, H, D)
    k = linear(h_ext, W_k).reshape(B, M + L, H, D)
    v = linear(h_ext, W_v).reshape(B, M + L, H, D)
    a = rel_attn(q, k, v, u, vb, W_R, M, mem_valid, clamp_len, scale=scale, threads=threads, rows=rows)
    return linear(a.reshape(B, L, H * D), W_o)


def stream_layer(h_all, W_q, W_k, W_v, W_o, u, vb, W_R, H: int, D: int, L: int, M: int,
                 clamp_len: int, scale=None, threads=None) -> np.ndarray:
    """The layer over S consecutive segments of h_all [B, S*L, d_model]: segment s attends to
    the hidden states of the M positions before it (fewer at the start of the sequence, the rest
    of the memory not valid), re-projected at every step, as the recurrence of
    "Transformer-XL 和相对位置编码" §2.3.1 defines it."""
    h_all = _f64(h_all)
    B, T, dm = h_all.shape
    assert T % L == 0
    out = np.empty((B, T, _f64(W_o).shape[1]), dtype=np.float64)
    for s in range(T // L):
        t0 = s * L
        valid = min(t0, M)
        h_mem = np.zeros((B, M, dm), dtype=np.float64)
        if valid:
            h_mem[:, M - valid:] = h_all[:, t0 - valid:t0]
        out[:, t0:t0 + L] = rel_layer(h_mem, h_all[:, t0:t0 + L], W_q, W_k, W_v, W_o, u, vb, W_R, H, D,
                                      valid, clamp_len, scale=scale, threads=threads)
    return out


def layer_flops(B: int, H: int, D: int, L: int, M: int, d_model: int, mem_valid: int | None = None) -> int:
    """Algorithmic flops of one layer step: the projections of the segment (q, k, v: 2*d_model*3HD
    per position; output: 2*HD*d_model per position) plus the attention (``attn_flops``).  The
    memory's keys and values are projected when they enter the memory, once per position."""
    return 2 * B * L * d_model * 4 * H * D + attn_flops(B, H, D, L, M, mem_valid)


def attn_flops(B: int, H: int, D: int, L: int, M: int, mem_valid: int | None = None) -> int:
    """Algorithmic flops of one call: 6*D per visible (query, key) pair (AC 2D, BD 2D, PV 2D)."""
    if mem_valid is None:
        mem_valid = M
    pairs = L * mem_valid + L * (L + 1) // 2
    return 6 * D * pairs * B * H
