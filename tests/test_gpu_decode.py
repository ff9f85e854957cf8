"""GPU parity of the decode path (txl_rel_attn_decode: 1..16 queries over a long memory, keys split
across CTAs and merged) against the fp64 oracle, including ring memories whose write pointer is not
a multiple of 128, partly valid memories, clamps inside the window, padded head strides and fp32."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import txl_inputs
from gpu_common import TOL, ld_r_for, max_err, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def txl():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import transformer_xl_relative_gb300 as m
    return m


def run_decode(txl, cfg, case, M, valid, wp, C, via_fwd=False):
    """Device inputs with the memory stored as a ring (logical key j in slot (wp + j) mod M)."""
    q, k, v = (to_dev(case[n], cfg.hs) for n in ("q", "k", "v"))
    L = q.shape[1]
    dt = cfg.torch_dtype
    n_rows = min(M + L, C + 1)
    r = torch.empty(n_rows, cfg.H, ld_r_for(cfg.D), dtype=dt, device="cuda")
    txl.rel_pos_gen(case["W_R"].cuda(), r, n_rows, cfg.d_model, cfg.H, cfg.D)
    mem = None
    if M > 0:
        store_k = to_dev(torch.zeros_like(case["k"][:, :M]), cfg.hs)
        store_v = to_dev(torch.zeros_like(case["v"][:, :M]), cfg.hs)
        slots = (wp + torch.arange(M)) % M
        store_k[:, slots] = k[:, :M]
        store_v[:, slots] = v[:, :M]
        mem = txl.Memory(store_k, store_v, wp, valid)
    out = to_dev(torch.full_like(case["q"], float("nan")), cfg.hs)
    u, vb = case["u"].cuda(), case["vb"].cuda()
    if not via_fwd:
        # three or more bf16 queries with d_head <= 64 on inputs the fused kernel takes (16-byte rows,
        # a ring's write pointer and length multiples of 128) go to it; everything else to the
        # split-key decode kernels
        fused = (cfg.dtype == "bf16" and L >= 3 and cfg.D <= 64 and
                 (M == 0 or wp == 0 or (wp % 128 == 0 and M % 128 == 0)))
        assert txl.rel_attn_decode_path(q, mem, k[:, M:], v[:, M:], r, out) == (1 if fused else 4)
    if via_fwd:
        txl.rel_attn_fwd(q, mem, k[:, M:], v[:, M:], u, vb, r, n_rows, C, out)
    else:
        txl.rel_attn_decode(q, mem, k[:, M:], v[:, M:], u, vb, r, n_rows, C, out)
    torch.cuda.synchronize()
    return out


DECODE = [
    # B, H, D, d_model, L, M, valid, wp, C, dtype, head_stride
    (2, 4, 64, 128, 1, 1000, 1000, 0, 1000, "bf16", 0),     # one new token, plain memory
    (2, 3, 64, 128, 1, 700, 700, 37, 300, "bf16", 0),       # ring, wp not a multiple of 128, clamp inside
    (1, 2, 64, 64, 5, 600, 400, 123, 1000, "bf16", 0),      # partly valid ring memory
    (1, 2, 128, 128, 16, 513, 513, 200, 200, "bf16", 0),    # 16 queries, D = 128
    (2, 2, 41, 82, 3, 300, 300, 5, 1000, "bf16", 48),       # D = 41, padded head stride
    (1, 2, 64, 64, 16, 0, 0, 0, 1000, "bf16", 0),           # no memory
    (2, 4, 64, 128, 1, 4096, 4096, 1000, 1000, "bf16", 0),  # long memory: 17 chunks, distances clamp
    (1, 2, 8, 16, 8, 8, 8, 3, 16, "f32", 0),                # fp32, tiny
    (1, 2, 32, 32, 2, 777, 500, 600, 64, "f32", 0),         # fp32 ring, clamp far inside
    # three or more queries with d_head <= 64 on memories the fused kernel takes go to it: a plain
    # memory, and a partly valid ring whose write pointer and length are multiples of 128
    (2, 4, 64, 128, 8, 1024, 1024, 0, 1000, "bf16", 0),
    (1, 3, 64, 128, 4, 512, 300, 256, 200, "bf16", 0),
]


@pytest.mark.parametrize("shape", DECODE, ids=[
    "B%dH%dD%d_L%dM%dv%dwp%dC%d_%s" % (s[0], s[1], s[2], s[4], s[5], s[6], s[7], s[8], s[9]) for s in DECODE])
def test_decode_matches_oracle(txl, shape):
    B, H, D, dm, L, M, valid, wp, C, dtype, hs = shape
    cfg = txl_inputs.custom(B=B, H=H, D=D, d_model=dm, L=L, M=M, clamp_len=C, dtype=dtype,
                            seed=300 + L + M + wp, head_stride=hs)
    case = txl_inputs.make_case(cfg)
    out = run_decode(txl, cfg, case, M, valid, wp, C)
    ref = oracle.rel_attn(case["q"], case["k"], case["v"], case["u"], case["vb"],
                          case["W_R"][:, : H * D], M, valid, C)
    err = max_err(out, ref)
    assert np.isfinite(err) and err <= TOL[dtype], err


def test_decode_agrees_with_the_general_path(txl):
    """The split-key decode and txl_rel_attn_fwd on the same ring and queries."""
    cfg = txl_inputs.custom(B=2, H=4, D=64, d_model=128, L=4, M=900, clamp_len=500, dtype="bf16", seed=77)
    case = txl_inputs.make_case(cfg)
    a = run_decode(txl, cfg, case, 900, 850, 77, 500)
    b = run_decode(txl, cfg, case, 900, 850, 77, 500, via_fwd=True)
    assert torch.max(torch.abs(a.float() - b.float())).item() <= TOL["bf16"]


def test_decode_rejects_without_workspace(txl):
    cfg = txl_inputs.custom(B=1, H=1, D=64, d_model=64, L=1, M=300, clamp_len=1000, dtype="bf16", seed=5)
    case = txl_inputs.make_case(cfg)
    q = case["q"].cuda()
    out = torch.empty_like(q)
    tiny = torch.empty(16, dtype=torch.uint8, device="cuda")
    mem = txl.Memory(case["k"][:, :300].cuda(), case["v"][:, :300].cuda(), 0, 300)
    r = torch.zeros(301, 1, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(txl.TxlError):
        txl.rel_attn_decode(q, mem, case["k"][:, 300:].cuda(), case["v"][:, 300:].cuda(),
                            case["u"].cuda(), case["vb"].cuda(), r, 301, 1000, out, workspace=tiny)


def test_decode_full_workload_several_queries(txl):
    """The decode workload's full size (B8 H16 D64, a 4096-key memory, clamp 1000) with four new
    queries per (b, h): the fused kernel's route, sampled rows against the oracle."""
    B, H, D, L, M, C = 8, 16, 64, 4, 4096, 1000
    cfg = txl_inputs.custom(B=B, H=H, D=D, d_model=1024, L=L, M=M, clamp_len=C, dtype="bf16", seed=4444)
    case = txl_inputs.make_case(cfg)
    out = run_decode(txl, cfg, case, M, M, 0, C)
    rows = [(b, h, i) for b in (0, 5, 7) for h in (0, 9, 15) for i in range(L)]
    ref = oracle.rel_attn(case["q"], case["k"], case["v"], case["u"], case["vb"],
                          case["W_R"][:, : H * D], M, M, C, rows=rows)
    assert max_err(out, ref, rows=rows) <= TOL["bf16"]
