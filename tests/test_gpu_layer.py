"""GPU parity of the projection product (txl_linear) and of the attention-layer step
(txl_rel_attn_layer: projections, relative attention over [memory ++ segment], output projection,
memory push) against the fp64 oracle.

txl_linear: bf16 products are exact in fp32, so the GPU result differs from the fp64 product of
the same bf16 inputs by the fp32 accumulation (at most k * 2^-24 * sum|x w|, taken here as 2^-14 of
sum|x w| for k <= 1024) plus one rounding to bf16 (half an ulp, at most 2^-9 |y|); the test allows
2^-8 |y| + 2^-13 sum|x w|.
Layer: the oracle re-projects the memory's hidden states at every step in fp64, the GPU caches the
bf16-rounded projections; q, k, v and the attention output are rounded to bf16 once each.  With
unit-variance activations and W_o columns of unit norm the output error stays at the attention's
level, and the bf16 attention tolerance (2e-2, max abs) is used for y."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import txl_inputs
from gpu_common import TOL, ld_r_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def txl():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import transformer_xl_relative_gb300 as m
    return m


def _check_linear(Y, X, W, rows=None):
    Xd = X.double().cpu().numpy()
    Wd = W.double().cpu().numpy()
    if rows is not None:
        Xd = Xd[rows]
    ref = oracle.linear(Xd, Wd)
    bound = np.abs(Xd) @ np.abs(Wd)
    got = Y.double().cpu().numpy()
    if rows is not None:
        got = got[rows]
    err = np.abs(got - ref)
    assert np.isfinite(got).all()
    assert np.all(err <= 2.0 ** -8 * np.abs(ref) + 2.0 ** -13 * bound), float(np.max(err))


LINEAR = [
    # m, n, k, ld_y extra
    (128, 256, 64, 0),       # one tile, one K slice
    (1, 8, 8, 0),            # degenerate: one row, K far below the slice
    (300, 520, 200, 0),      # ragged rows, a 8-column tail, K not a multiple of 64
    (777, 1000, 1000, 24),   # Y rows padded (ld_y > n)
    (384, 3072, 1024, 0),    # the fused q|k|v product of one batch entry of the large workload
]


@pytest.mark.parametrize("shape", LINEAR, ids=["m%d_n%d_k%d_pad%d" % s for s in LINEAR])
def test_linear_matches_fp64(txl, shape):
    m, n, k, pad = shape
    X = txl_inputs.make_matrix(m, k, seed=m + n).cuda()
    W = txl_inputs.make_matrix(k, n, seed=m + k + 1, std=k ** -0.5).cuda()
    store = torch.full((m, n + pad), float("nan"), dtype=torch.bfloat16, device="cuda")
    Y = txl.linear(X, W, store[:, :n])
    torch.cuda.synchronize()
    _check_linear(Y, X, W)
    if pad:
        assert torch.isnan(store[:, n:].float()).all()       # nothing past n is written


def test_linear_large_sampled_rows(txl):
    """The q|k|v product of the whole large workload (6144 x 3072 x 1024), checked on sampled rows."""
    m, n, k = 16 * 384, 3 * 1024, 1024
    X = txl_inputs.make_matrix(m, k, seed=5).cuda()
    W = txl_inputs.make_matrix(k, n, seed=6, std=k ** -0.5).cuda()
    Y = txl.linear(X, W)
    torch.cuda.synchronize()
    rows = np.random.default_rng(0).choice(m, 96, replace=False)
    rows = np.sort(np.concatenate([rows, [0, 127, 128, m - 1]]))
    _check_linear(Y, X, W, rows=rows)


def _layer_stream(txl, cfg, S):
    """GPU: S layer steps over segments of h with an initially empty memory; oracle: the
    recurrence over the hidden states."""
    lay = txl_inputs.make_layer(cfg, segments=S)
    H, D, L, M, dm = cfg.H, cfg.D, cfg.L, cfg.M, cfg.d_model
    HD = H * D
    n_rows = min(M + L, cfg.clamp_len + 1)
    r = torch.empty(n_rows, H, ld_r_for(D), dtype=torch.bfloat16, device="cuda")
    txl.rel_pos_gen(lay["W_R"].cuda(), r, n_rows, dm, H, D)
    mem = txl.Memory.empty(cfg.B, M, H, D) if M > 0 else None
    h = lay["h"].cuda()
    W_qkv, W_o = lay["W_qkv"].cuda(), lay["W_o"].cuda()
    u, vb = lay["u"].cuda(), lay["vb"].cuda()
    ys = []
    for s in range(S):
        y = torch.full((cfg.B, L, dm), float("nan"), dtype=torch.bfloat16, device="cuda")
        txl.rel_attn_layer(h[:, s * L:(s + 1) * L].contiguous(), mem, W_qkv, W_o, u, vb, r, n_rows,
                           cfg.clamp_len, H, D, y)
        ys.append(y)
    torch.cuda.synchronize()
    got = torch.cat(ys, dim=1).double().cpu().numpy()
    Wf = lay["W_qkv"].double().numpy()
    ref = oracle.stream_layer(lay["h"].double().numpy(), Wf[:, :HD], Wf[:, HD:2 * HD], Wf[:, 2 * HD:],
                              lay["W_o"].double().numpy(), lay["u"], lay["vb"], lay["W_R"][:, :HD], H, D, L, M,
                              cfg.clamp_len)
    return got, ref, mem


LAYER = [
    # B, H, D, d_model, L, M, clamp, segments
    (2, 2, 64, 128, 128, 128, 1000, 3),     # memory of one segment, three steps
    (1, 4, 64, 256, 128, 256, 100, 3),      # memory of two segments, clamp inside the window
    (2, 2, 64, 192, 256, 128, 1000, 2),     # segment longer than the memory
]


@pytest.mark.parametrize("shape", LAYER, ids=["B%dH%dD%d_dm%d_L%dM%d_C%d_S%d" % s for s in LAYER])
def test_layer_stream_matches_oracle(txl, shape):
    B, H, D, dm, L, M, C, S = shape
    cfg = txl_inputs.custom(B=B, H=H, D=D, d_model=dm, L=L, M=M, clamp_len=C, dtype="bf16", seed=40 + S + L)
    got, ref, mem = _layer_stream(txl, cfg, S)
    err = np.max(np.abs(got - ref))
    assert np.isfinite(got).all() and err <= TOL["bf16"], err
    assert mem.valid == min(S * L, M)


def test_layer_without_memory(txl):
    cfg = txl_inputs.custom(B=2, H=2, D=64, d_model=128, L=128, M=0, dtype="bf16", seed=9)
    got, ref, _ = _layer_stream(txl, cfg, 1)
    assert np.max(np.abs(got - ref)) <= TOL["bf16"]


def test_layer_large_sampled(txl):
    """The large workload (B16 H16 D64 d_model 1024 L384 M384): two steps, the second over a full
    memory, checked on sampled positions (every head of each)."""
    cfg = txl_inputs.CONFIGS["large"]
    lay = txl_inputs.make_layer(cfg, segments=2)
    H, D, L, M, dm = cfg.H, cfg.D, cfg.L, cfg.M, cfg.d_model
    HD = H * D
    n_rows = min(M + L, cfg.clamp_len + 1)
    r = torch.empty(n_rows, H, D, dtype=torch.bfloat16, device="cuda")
    txl.rel_pos_gen(lay["W_R"].cuda(), r, n_rows, dm, H, D)
    mem = txl.Memory.empty(cfg.B, M, H, D)
    h = lay["h"].cuda()
    W_qkv, W_o, u, vb = lay["W_qkv"].cuda(), lay["W_o"].cuda(), lay["u"].cuda(), lay["vb"].cuda()
    ys = [txl.rel_attn_layer(h[:, s * L:(s + 1) * L].contiguous(), mem, W_qkv, W_o, u, vb, r, n_rows,
                             cfg.clamp_len, H, D) for s in range(2)]
    torch.cuda.synchronize()
    y1 = ys[1].double().cpu().numpy()
    rng = np.random.default_rng(1)
    pos = [(int(b), int(i)) for b, i in zip(rng.integers(0, cfg.B, 12), rng.integers(0, L, 12))]
    pos += [(0, 0), (cfg.B - 1, L - 1)]
    rows = [(b, hh, i) for b, i in pos for hh in range(H)]
    hd = lay["h"].double().numpy()
    Wf = lay["W_qkv"].double().numpy()
    ref = oracle.rel_layer(hd[:, :L], hd[:, L:], Wf[:, :HD], Wf[:, HD:2 * HD], Wf[:, 2 * HD:],
                           lay["W_o"].double().numpy(), lay["u"], lay["vb"], lay["W_R"][:, :HD], H, D, M,
                           cfg.clamp_len, rows=rows)
    for b, i in pos:
        err = np.max(np.abs(y1[b, i] - ref[b, i]))
        assert np.isfinite(ref[b, i]).all() and err <= TOL["bf16"], (b, i, err)


def test_layer_rejections(txl):
    cfg = txl_inputs.custom(B=1, H=2, D=64, d_model=128, L=128, M=128, dtype="bf16", seed=3)
    lay = txl_inputs.make_layer(cfg)
    r = torch.zeros(257, 2, 64, dtype=torch.bfloat16, device="cuda")
    mem = txl.Memory.empty(1, 128, 2, 64)
    args = (lay["h"].cuda(), mem, lay["W_qkv"].cuda(), lay["W_o"].cuda(), lay["u"].cuda(), lay["vb"].cuda(), r,
            257, 1000, 2, 64)
    with pytest.raises(txl.TxlError):                    # workspace too small
        txl.rel_attn_layer(*args, workspace=torch.empty(64, dtype=torch.uint8, device="cuda"))
    with pytest.raises(txl.TxlError):                    # fp32 projections are not provided
        txl.linear(torch.zeros(4, 8, device="cuda"), torch.zeros(8, 8, device="cuda"))
    assert mem.valid == 0 and mem.wp == 0                # a rejected call leaves the memory alone


# --------------------------------------------------------------------------- fused layer step
def _fused_stream(txl, cfg, S, extra_slots=0):
    """S steps of txl_rel_attn_layer_fused (memory of M positions in a ring of M + L + extra_slots
    slots) beside S steps of txl_rel_attn_layer on the same inputs."""
    lay = txl_inputs.make_layer(cfg, segments=S)
    H, D, L, M, dm = cfg.H, cfg.D, cfg.L, cfg.M, cfg.d_model
    n_rows = min(M + L, cfg.clamp_len + 1)
    r = torch.empty(n_rows, H, ld_r_for(D), dtype=torch.bfloat16, device="cuda")
    txl.rel_pos_gen(lay["W_R"].cuda(), r, n_rows, dm, H, D)
    ring = txl.Memory.empty(cfg.B, M + L + extra_slots, H, D)
    mem = txl.Memory.empty(cfg.B, M, H, D) if M > 0 else None
    h = lay["h"].cuda()
    W_qkv, W_o, u, vb = lay["W_qkv"].cuda(), lay["W_o"].cuda(), lay["u"].cuda(), lay["vb"].cuda()
    fused, plain = [], []
    for s in range(S):
        hs = h[:, s * L:(s + 1) * L].contiguous()
        fused.append(txl.rel_attn_layer_fused(hs, ring, M, W_qkv, W_o, u, vb, r, n_rows, cfg.clamp_len, H, D))
        plain.append(txl.rel_attn_layer(hs, mem, W_qkv, W_o, u, vb, r, n_rows, cfg.clamp_len, H, D))
    torch.cuda.synchronize()
    return lay, fused, plain, ring


FUSED = [
    # B, H, D, d_model, L, M, clamp, segments, extra ring slots
    (2, 2, 64, 128, 128, 128, 1000, 3, 0),   # memory of one segment, the ring exactly M + L
    (1, 4, 64, 256, 128, 256, 100, 3, 0),    # memory of two segments, clamp inside the window
    (2, 2, 64, 192, 256, 128, 1000, 2, 0),   # segment longer than the memory
    (1, 2, 64, 128, 128, 256, 1000, 5, 128), # spare slots: the window wraps around the ring
    (2, 2, 64, 128, 128, 0, 1000, 2, 0),     # no memory
]


@pytest.mark.parametrize("shape", FUSED, ids=["B%dH%dD%d_dm%d_L%dM%d_C%d_S%d_x%d" % s for s in FUSED])
def test_fused_layer_matches_oracle_and_unfused(txl, shape):
    B, H, D, dm, L, M, C, S, extra = shape
    cfg = txl_inputs.custom(B=B, H=H, D=D, d_model=dm, L=L, M=M, clamp_len=C, dtype="bf16", seed=70 + S + L + M)
    lay, fused, plain, ring = _fused_stream(txl, cfg, S, extra)
    for s in range(S):                      # the same products and the same attention, step by step
        assert torch.equal(fused[s], plain[s]), s
    HD = H * D
    got = torch.cat(fused, dim=1).double().cpu().numpy()
    Wf = lay["W_qkv"].double().numpy()
    ref = oracle.stream_layer(lay["h"].double().numpy(), Wf[:, :HD], Wf[:, HD:2 * HD], Wf[:, 2 * HD:],
                              lay["W_o"].double().numpy(), lay["u"], lay["vb"], lay["W_R"][:, :HD], H, D, L, M, C)
    err = np.max(np.abs(got - ref))
    assert np.isfinite(got).all() and err <= TOL["bf16"], err
    assert ring.valid == min(S * L, M) and ring.wp == (S * L) % (M + L + extra)


def test_fused_layer_large_workload(txl):
    """The large workload's layer step (B16 H16 D64 d_model 1024 L384 M384), two steps in a ring
    of 768 slots, bit-identical to the unfused step."""
    cfg = txl_inputs.CONFIGS["large"]
    _, fused, plain, ring = _fused_stream(txl, cfg, 2)
    assert torch.equal(fused[0], plain[0]) and torch.equal(fused[1], plain[1])
    assert ring.valid == cfg.M and ring.wp == 0


def test_fused_layer_rejections(txl):
    cfg = txl_inputs.custom(B=1, H=2, D=64, d_model=128, L=128, M=128, dtype="bf16", seed=3)
    lay = txl_inputs.make_layer(cfg)
    r = torch.zeros(257, 2, 64, dtype=torch.bfloat16, device="cuda")
    h, W_qkv, W_o, u, vb = (lay[n].cuda() for n in ("h", "W_qkv", "W_o", "u", "vb"))
    small = txl.Memory.empty(1, 128, 2, 64)              # no room for the segment after the memory
    with pytest.raises(txl.TxlError):
        txl.rel_attn_layer_fused(h, small, 128, W_qkv, W_o, u, vb, r, 257, 1000, 2, 64)
    odd = txl.Memory.empty(1, 320, 2, 64)                # slots not a multiple of 128
    with pytest.raises(txl.TxlError):
        txl.rel_attn_layer_fused(h, odd, 128, W_qkv, W_o, u, vb, r, 257, 1000, 2, 64)
    ring = txl.Memory.empty(1, 256, 2, 64)
    with pytest.raises(txl.TxlError):                    # workspace too small
        txl.rel_attn_layer_fused(h, ring, 128, W_qkv, W_o, u, vb, r, 257, 1000, 2, 64,
                                 workspace=torch.empty(64, dtype=torch.uint8, device="cuda"))
    assert (small.wp, small.valid, odd.wp, odd.valid, ring.wp, ring.valid) == (0, 0, 0, 0, 0, 0)
