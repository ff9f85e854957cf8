"""GPU parity of the backward (txl_rel_attn_bwd, txl_rel_pos_bwd) against the fp64 backward oracle
(itself pinned against finite differences of the forward oracle).

The GPU recomputes the scores in fp32 from the same inputs and takes D_i = d_out_i . out_i from
the forward output it is given (here the library's own forward, rounded to the compute dtype),
while the oracle uses the exact fp64 attention.  The rounding of out (half an ulp: 2^-9 relative in
bf16, 2^-24 in fp32) enters every dS_ij of the row through D_i, so gradients are compared with a
tolerance relative to their largest entry: 2e-2 for bf16 inputs, 1e-4 for fp32."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import txl_inputs
from gpu_common import ld_r_for, to_dev

pytestmark = pytest.mark.gpu
RTOL = {"bf16": 2e-2, "f32": 1e-4}


@pytest.fixture(scope="module")
def txl():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import transformer_xl_relative_gb300 as m
    return m


def _close(got, ref, tol, what):
    got = np.asarray(got, dtype=np.float64)
    scale = max(np.max(np.abs(ref)), 1e-30)
    err = np.max(np.abs(got - ref)) if ref.size else 0.0
    assert np.isfinite(got).all(), what
    assert err <= tol * scale, (what, err, scale)


BWD = [
    # B, H, D, d_model, L, M, valid, wp, C, dtype, head_stride
    (1, 2, 16, 32, 8, 8, 8, 0, 1000, "f32", 0),          # tiny fp32, full memory
    (2, 2, 64, 128, 64, 64, 40, 0, 1000, "bf16", 0),     # partly valid memory
    (1, 2, 32, 64, 40, 30, 30, 7, 20, "bf16", 0),        # ring with an unaligned write pointer, clamp inside
    (2, 3, 41, 82, 24, 0, 0, 0, 10, "bf16", 48),         # no memory, clamp, padded heads
    (2, 4, 64, 128, 128, 128, 128, 0, 1000, "bf16", 0),  # a full 128-key tile on each side
    (1, 2, 128, 128, 30, 33, 20, 5, 40, "bf16", 0),      # D = 128, ring, clamp, L not a multiple of 4
    # d_head 64 with 16-byte rows takes the tensor-core kernel: ragged query tiles, ring write
    # pointers, clamps inside a key tile's distance window, no memory, one query, the large
    # workload's per-head shape; a 68-element head stride keeps d_head 64 on the SIMT kernels
    (1, 2, 64, 128, 100, 70, 70, 13, 30, "bf16", 0),
    (2, 2, 64, 128, 200, 0, 0, 0, 50, "bf16", 0),
    (1, 1, 64, 64, 5, 3, 2, 1, 1000, "bf16", 0),
    (1, 2, 64, 64, 1, 130, 130, 0, 1000, "bf16", 0),
    (1, 2, 64, 128, 384, 384, 384, 0, 1000, "bf16", 0),
    (1, 2, 64, 128, 70, 64, 64, 0, 40, "bf16", 0),
    (1, 2, 64, 128, 40, 30, 30, 0, 1000, "bf16", 68),
    # the tcgen05 gradient kernel (the fused forward takes the inputs: a ring's write pointer and length
    # multiples of 128): a wrapped ring with part of the memory valid, ragged query tiles, a clamp
    # inside the window of the third key tile
    (2, 2, 64, 128, 200, 256, 200, 128, 300, "bf16", 0),
]


@pytest.mark.parametrize("shape", BWD, ids=["B%dH%dD%d_L%dM%dv%dwp%dC%d_%s" % (s[0], s[1], s[2], s[4], s[5], s[6], s[7], s[8], s[9])
                                            for s in BWD])
def test_backward_matches_oracle(txl, shape):
    B, H, D, dm, L, M, valid, wp, C, dtype, hs = shape
    cfg = txl_inputs.custom(B=B, H=H, D=D, d_model=dm, L=L, M=M, clamp_len=C, dtype=dtype, seed=500 + L + M, head_stride=hs)
    case = txl_inputs.make_case(cfg)
    dO = txl_inputs.make_qkv(cfg, seed=900 + L, L=L, T=1)[0]                    # [B, L, H, D] upstream gradient
    q, k, v = (to_dev(case[n], cfg.hs) for n in ("q", "k", "v"))
    g_dev = to_dev(dO, cfg.hs)
    dt = cfg.torch_dtype
    n_rows = min(M + L, C + 1)
    r = torch.empty(n_rows, H, ld_r_for(D), dtype=dt, device="cuda")
    txl.rel_pos_gen(case["W_R"].cuda(), r, n_rows, dm, H, D)
    mem = None
    if M > 0:
        store_k = to_dev(torch.zeros_like(case["k"][:, :M]), cfg.hs)
        store_v = to_dev(torch.zeros_like(case["v"][:, :M]), cfg.hs)
        slots = (wp + torch.arange(M)) % M
        store_k[:, slots] = k[:, :M]
        store_v[:, slots] = v[:, :M]
        mem = txl.Memory(store_k, store_v, wp, valid)
    u, vb = case["u"].cuda(), case["vb"].cuda()
    out = to_dev(torch.zeros_like(case["q"]), cfg.hs)
    txl.rel_attn_fwd(q, mem, k[:, M:], v[:, M:], u, vb, r, n_rows, C, out)
    g = txl.rel_attn_bwd(q, mem, k[:, M:], v[:, M:], u, vb, r, n_rows, C, out, g_dev)
    path = txl.rel_attn_bwd_path(q, mem, k[:, M:], v[:, M:], r, out, g_dev, g)
    if dtype == "f32" or D != 64 or hs:
        assert path == 3
    elif M > 0 and wp != 0 and (M % 128 or wp % 128):
        assert path == 2                                   # the fused forward declines the ring
    else:
        assert path == 1
    dW = txl.rel_pos_bwd(g["dr"], dm)
    torch.cuda.synchronize()
    ref = oracle.rel_attn_bwd(case["q"], case["k"], case["v"], case["u"], case["vb"], case["W_R"][:, :H * D], M, valid,
                              C, dO)
    tol = RTOL[dtype]
    _close(g["dq"].cpu().numpy(), ref["dq"], tol, "dq")
    _close(g["dk_cur"].cpu().numpy(), ref["dk"][:, M:], tol, "dk")
    _close(g["dv_cur"].cpu().numpy(), ref["dv"][:, M:], tol, "dv")
    _close(g["du"].cpu().numpy(), ref["du"], tol, "du")
    _close(g["dv_bias"].cpu().numpy(), ref["dvb"], tol, "dv_bias")
    _close(g["dr"].cpu().numpy(), ref["dr"], tol, "dr")
    _close(dW.cpu().numpy(), ref["dW_R"], tol, "dW_R")


def test_pos_backward_closed_form(txl):
    """dW_R for a one-hot dr: row delta of dr selects the sinusoid R_delta (column h*D + d)."""
    n_rows, dm, H, D = 50, 64, 2, 8
    dr = torch.zeros(n_rows, H, D, dtype=torch.float32, device="cuda")
    dr[37, 1, 5] = 1.0
    dr[3, 0, 0] = -2.0
    dW = txl.rel_pos_bwd(dr, dm)
    torch.cuda.synchronize()
    ref = np.zeros((dm, H * D))
    ref[:, 1 * D + 5] = oracle.sinusoid(37.0, dm)
    ref[:, 0] = -2.0 * oracle.sinusoid(3.0, dm)
    assert np.max(np.abs(dW.cpu().numpy() - ref)) <= 1e-6


def test_backward_large_workload_sampled(txl):
    """The bench's backward workload at full size (B16 H16 D64 L384 M384 clamp 1000, bf16: the
    tensor-core kernel, in the launch the bench times): dq, dk and dv of sampled (b, h) pairs against
    the oracle evaluated on those pairs alone (the pairs are independent; du, dv_bias and dr sum over
    every pair and are covered by the smaller cases)."""
    B, H, D, dm, L, M, C = 16, 16, 64, 1024, 384, 384, 1000
    cfg = txl_inputs.custom(B=B, H=H, D=D, d_model=dm, L=L, M=M, clamp_len=C, dtype="bf16", seed=4242)
    case = txl_inputs.make_case(cfg)
    dO = txl_inputs.make_qkv(cfg, seed=4243, L=L, T=1)[0]
    q, k, v = (to_dev(case[n]) for n in ("q", "k", "v"))
    n_rows = min(M + L, C + 1)
    r = torch.empty(n_rows, H, D, dtype=torch.bfloat16, device="cuda")
    txl.rel_pos_gen(case["W_R"].cuda(), r, n_rows, dm, H, D)
    mem = txl.Memory(k[:, :M], v[:, :M], 0, M)
    u, vb = case["u"].cuda(), case["vb"].cuda()
    out = torch.empty_like(q)
    txl.rel_attn_fwd(q, mem, k[:, M:], v[:, M:], u, vb, r, n_rows, C, out)
    g = txl.rel_attn_bwd(q, mem, k[:, M:], v[:, M:], u, vb, r, n_rows, C, out, to_dev(dO))
    assert txl.rel_attn_bwd_path(q, mem, k[:, M:], v[:, M:], r, out, to_dev(dO), g) == 1
    torch.cuda.synchronize()
    pairs = [(0, 0), (7, 11), (15, 15)]
    ref = oracle.rel_attn_bwd(case["q"], case["k"], case["v"], case["u"], case["vb"], case["W_R"][:, :H * D], M, M,
                              C, dO, bh=pairs)
    for b, h in pairs:
        _close(g["dq"][b, :, h].cpu().numpy(), ref["dq"][b, :, h], RTOL["bf16"], "dq %d %d" % (b, h))
        _close(g["dk_cur"][b, :, h].cpu().numpy(), ref["dk"][b, M:, h], RTOL["bf16"], "dk %d %d" % (b, h))
        _close(g["dv_cur"][b, :, h].cpu().numpy(), ref["dv"][b, M:, h], RTOL["bf16"], "dv %d %d" % (b, h))


LSE_CASES = [
    # B, H, D, d_model, L, M, valid, C
    (2, 2, 64, 128, 200, 150, 100, 1000),   # partly valid memory, ragged query tiles
    (1, 2, 64, 128, 130, 0, 0, 60),         # no memory, clamp inside the sequence
]


@pytest.mark.parametrize("shape", LSE_CASES, ids=["B%dH%dL%dM%dv%dC%d" % (s[0], s[1], s[4], s[5], s[6], s[7])
                                                  for s in LSE_CASES])
def test_saved_statistics_and_the_backward_given_them(txl, shape):
    """rel_attn_fwd with lse (txl_rel_attn_fwd_lse): the output is txl_rel_attn_fwd's, bit for bit,
    and the saved row log-sum-exp is the oracle's (oracle.rel_attn_lse, log2 units) within the bf16
    rounding of the query forms and of BD (|error| <= 0.05); rel_attn_bwd given it
    (txl_rel_attn_bwd_lse) matches the oracle's gradients like the call without it."""
    B, H, D, dm, L, M, valid, C = shape
    cfg = txl_inputs.custom(B=B, H=H, D=D, d_model=dm, L=L, M=M, clamp_len=C, dtype="bf16", seed=700 + L + M)
    case = txl_inputs.make_case(cfg)
    dO = txl_inputs.make_qkv(cfg, seed=701 + L, L=L, T=1)[0]
    q, k, v = (to_dev(case[n]) for n in ("q", "k", "v"))
    n_rows = min(M + L, C + 1)
    r = torch.empty(n_rows, H, D, dtype=torch.bfloat16, device="cuda")
    txl.rel_pos_gen(case["W_R"].cuda(), r, n_rows, dm, H, D)
    mem = txl.Memory(k[:, :M].contiguous(), v[:, :M].contiguous(), 0, valid) if M > 0 else None
    u, vb = case["u"].cuda(), case["vb"].cuda()
    out0, out1 = torch.empty_like(q), torch.empty_like(q)
    lse = torch.full((B, L, H), float("nan"), dtype=torch.float32, device="cuda")
    txl.rel_attn_fwd(q, mem, k[:, M:], v[:, M:], u, vb, r, n_rows, C, out0)
    txl.rel_attn_fwd(q, mem, k[:, M:], v[:, M:], u, vb, r, n_rows, C, out1, lse=lse)
    g = txl.rel_attn_bwd(q, mem, k[:, M:], v[:, M:], u, vb, r, n_rows, C, out1, to_dev(dO), lse=lse)
    torch.cuda.synchronize()
    assert torch.equal(out0, out1)
    want = oracle.rel_attn_lse(case["q"], case["k"], case["u"], case["vb"], case["W_R"][:, :H * D], M, valid, C)
    got = lse.cpu().numpy()
    assert np.isfinite(got).all()
    assert np.max(np.abs(got - want)) <= 0.05, np.max(np.abs(got - want))
    ref = oracle.rel_attn_bwd(case["q"], case["k"], case["v"], case["u"], case["vb"], case["W_R"][:, :H * D], M, valid,
                              C, dO)
    tol = RTOL["bf16"]
    _close(g["dq"].cpu().numpy(), ref["dq"], tol, "dq")
    _close(g["dk_cur"].cpu().numpy(), ref["dk"][:, M:], tol, "dk")
    _close(g["dv_cur"].cpu().numpy(), ref["dv"][:, M:], tol, "dv")
    _close(g["du"].cpu().numpy(), ref["du"], tol, "du")
    _close(g["dv_bias"].cpu().numpy(), ref["dvb"], tol, "dv_bias")
    _close(g["dr"].cpu().numpy(), ref["dr"], tol, "dr")


def test_saved_statistics_need_the_fused_kernel(txl):
    """txl_rel_attn_fwd_lse refuses (TXL_ERR_UNSUPPORTED, nothing launched) inputs the fused kernel
    does not take: fp32 here."""
    B, L, H, D = 1, 16, 2, 64
    q = torch.randn(B, L, H, D, device="cuda")
    k, v = torch.randn_like(q), torch.randn_like(q)
    u = torch.zeros(H, D, device="cuda")
    r = torch.zeros(L, H, D, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty(B, L, H, device="cuda")
    with pytest.raises(RuntimeError, match="txl_rel_attn_fwd_lse"):
        txl.rel_attn_fwd(q, None, k, v, u, u, r, L, 1000, out, lse=lse)


def test_backward_fallback_with_unaligned_output(txl):
    """An output view 8 bytes past a 16-byte boundary: the tcgen05 gradient kernel declines (it reads out
    and writes the gradients with 16-byte accesses) and the mma.sync kernel takes the call; its gradients
    match the oracle like the main path's."""
    B, H, D, dm, L, M, valid, C = 1, 2, 64, 128, 96, 64, 50, 1000
    cfg = txl_inputs.custom(B=B, H=H, D=D, d_model=dm, L=L, M=M, clamp_len=C, dtype="bf16", seed=811)
    case = txl_inputs.make_case(cfg)
    dO = txl_inputs.make_qkv(cfg, seed=812, L=L, T=1)[0]
    q, k, v = (to_dev(case[n]) for n in ("q", "k", "v"))
    n_rows = min(M + L, C + 1)
    r = torch.empty(n_rows, H, D, dtype=torch.bfloat16, device="cuda")
    txl.rel_pos_gen(case["W_R"].cuda(), r, n_rows, dm, H, D)
    mem = txl.Memory(k[:, :M].contiguous(), v[:, :M].contiguous(), 0, valid)
    u, vb = case["u"].cuda(), case["vb"].cuda()
    base = torch.zeros(B * L * H * D + 8, dtype=torch.bfloat16, device="cuda")
    out = base[4:4 + B * L * H * D].view(B, L, H, D)          # 8 bytes off alignment
    assert out.data_ptr() % 16 == 8
    txl.rel_attn_fwd(q, mem, k[:, M:], v[:, M:], u, vb, r, n_rows, C, out)
    g = txl.rel_attn_bwd(q, mem, k[:, M:], v[:, M:], u, vb, r, n_rows, C, out, to_dev(dO))
    assert txl.rel_attn_bwd_path(q, mem, k[:, M:], v[:, M:], r, out, to_dev(dO), g) == 2
    torch.cuda.synchronize()
    ref = oracle.rel_attn_bwd(case["q"], case["k"], case["v"], case["u"], case["vb"], case["W_R"][:, :H * D], M, valid,
                              C, dO)
    tol = RTOL["bf16"]
    _close(g["dq"].cpu().numpy(), ref["dq"], tol, "dq")
    _close(g["dk_cur"].cpu().numpy(), ref["dk"][:, M:], tol, "dk")
    _close(g["dv_cur"].cpu().numpy(), ref["dv"][:, M:], tol, "dv")
    _close(g["du"].cpu().numpy(), ref["du"], tol, "du")
    _close(g["dv_bias"].cpu().numpy(), ref["dvb"], tol, "dv_bias")
    _close(g["dr"].cpu().numpy(), ref["dr"], tol, "dr")
