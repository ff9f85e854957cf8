"""GPU tests of txl_rel_attn_decode_noalloc, the decode entry point for callers that cannot obtain
device memory when they call (a serving process whose device memory is a pre-sized arena, a plugin
whose interface passes only inputs and outputs, a generation loop that cannot afford cudaMalloc):
it keeps its partial results in the library's fixed 8 MiB scratch array instead of a caller
workspace.

Every call goes through the C ABI.  The entry point runs the same kernels as txl_rel_attn_decode
on the same inputs, so its output must be bit-identical to that entry point's; one call of each
dtype is also checked against the fp64 oracle within the tolerance of the other tests.  Two
different calls run in a row on one stream, so a stale scratch from the first call would show in
the second.  The size limit is checked at its edge: a shape whose partial results take exactly
8388608 bytes is accepted, one more chunk of keys is refused with TXL_ERR_WORKSPACE.  This file is
collected last."""
from __future__ import annotations

import ctypes

import pytest
import torch

import oracle
import txl_inputs
from gpu_common import TOL, ld_r_for, max_err, to_dev

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 8 << 20


@pytest.fixture(scope="module")
def txl():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import transformer_xl_relative_gb300 as m
    return m


def make_call(txl, B, H, D, L, M, valid, wp, C, seed, dtype="bf16"):
    """Device inputs of one decode call, the memory stored as a ring (logical key j in slot
    (wp + j) mod M), plus the CPU case for the oracle."""
    cfg = txl_inputs.custom(B=B, H=H, D=D, d_model=2 * D, L=L, M=M, clamp_len=C, dtype=dtype, seed=seed)
    case = txl_inputs.make_case(cfg)
    q, k, v = (to_dev(case[n]) for n in ("q", "k", "v"))
    n_rows = min(M + L, C + 1)
    r = torch.empty(n_rows, H, ld_r_for(D), dtype=cfg.torch_dtype, device="cuda")
    txl.rel_pos_gen(case["W_R"].cuda(), r, n_rows, cfg.d_model, H, D)
    store_k = torch.zeros_like(k[:, :M])
    store_v = torch.zeros_like(v[:, :M])
    slots = (wp + torch.arange(M)) % M
    store_k[:, slots] = k[:, :M]
    store_v[:, slots] = v[:, :M]
    mem = txl.Memory(store_k, store_v, wp, valid)
    return dict(q=q, mem=mem, k_cur=k[:, M:], v_cur=v[:, M:], u=case["u"].cuda(), vb=case["vb"].cuda(),
                r=r, n_rows=n_rows, C=C, M=M, valid=valid, case=case, cfg=cfg)


def scratch_need(B, H, D, L, M):
    chunks = (M + L + 255) // 256
    return B * H * L * chunks * (D + 2) * 4


def noalloc(txl, c, out):
    """txl_rel_attn_decode_noalloc through the C ABI; returns its status."""
    from transformer_xl_relative_gb300 import api, native
    q = c["q"]
    B, L, H, D = q.shape
    vq, vk, vv, vo = api.view(q), api.view(c["k_cur"]), api.view(c["v_cur"]), api.view(out)
    return native.load().txl_rel_attn_decode_noalloc(
        B, L, H, D, c["C"], ctypes.byref(vq), ctypes.byref(c["mem"].c_struct), ctypes.byref(vk),
        ctypes.byref(vv), c["u"].data_ptr(), c["vb"].data_ptr(), c["r"].data_ptr(), c["r"].stride(1),
        c["n_rows"], 0.0, ctypes.byref(vo), api.dtype_code(q), None)


def with_workspace(txl, c):
    out = torch.full_like(c["q"], float("nan"))
    txl.rel_attn_decode(c["q"], c["mem"], c["k_cur"], c["v_cur"], c["u"], c["vb"], c["r"], c["n_rows"],
                        c["C"], out)
    return out


def oracle_of(c, rows=None):
    case, cfg = c["case"], c["cfg"]
    return oracle.rel_attn(case["q"], case["k"], case["v"], case["u"], case["vb"],
                           case["W_R"][:, : cfg.H * cfg.D], c["M"], c["valid"], c["C"], rows=rows)


def test_noalloc_matches_the_workspace_entry_point_twice(txl):
    from transformer_xl_relative_gb300 import native
    calls = [make_call(txl, 2, 4, 64, 3, 1000, 900, 37, 500, seed=11),     # 4 chunks per (b, h)
             make_call(txl, 3, 2, 64, 1, 2200, 2200, 300, 1000, seed=12),  # 9 chunks, other shape
             make_call(txl, 2, 2, 64, 4, 640, 640, 128, 1000, seed=16)]    # the fused kernel's route
    refs = [with_workspace(txl, c) for c in calls]
    outs = [torch.full_like(c["q"], float("nan")) for c in calls]
    # two calls in a row on one stream: the second reuses the scratch the first has just used
    for c, out in zip(calls, outs):
        assert noalloc(txl, c, out) == native.TXL_OK
    torch.cuda.synchronize()
    for ref, out in zip(refs, outs):
        assert torch.equal(out, ref)
    # and the first call against the fp64 oracle
    assert max_err(outs[0], oracle_of(calls[0])) <= TOL["bf16"]


def test_noalloc_fp32(txl):
    from transformer_xl_relative_gb300 import native
    c = make_call(txl, 2, 3, 32, 2, 700, 650, 5, 300, seed=13, dtype="f32")
    ref = with_workspace(txl, c)
    out = torch.full_like(c["q"], float("nan"))
    assert noalloc(txl, c, out) == native.TXL_OK
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    assert max_err(out, oracle_of(c)) <= TOL["f32"]


def test_noalloc_size_limit_at_its_edge(txl):
    """D = 62, so a chunk's partials of one query take 64 floats: B2 H16 L16 with M + L = 16384
    keys (64 chunks) need exactly 8388608 bytes; one more key needs a 65th chunk."""
    from transformer_xl_relative_gb300 import native
    B, H, D, L, C = 2, 16, 62, 16, 1000
    M = 64 * 256 - L
    assert scratch_need(B, H, D, L, M) == SCRATCH_BYTES
    c = make_call(txl, B, H, D, L, M, M, 1234, C, seed=14)
    ref = with_workspace(txl, c)
    out = torch.full_like(c["q"], float("nan"))
    assert noalloc(txl, c, out) == native.TXL_OK
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    rows = [(b, h, i) for b in range(B) for h in (0, 7, 15) for i in (0, 9, L - 1)]
    assert max_err(out, oracle_of(c, rows=rows), rows=rows) <= TOL["bf16"]

    M1 = M + 1
    assert scratch_need(B, H, D, L, M1) > SCRATCH_BYTES
    big = make_call(txl, B, H, D, L, M1, M1, 0, C, seed=15)
    out1 = torch.full_like(big["q"], float("nan"))
    assert noalloc(txl, big, out1) == native.TXL_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.isnan(out1.float()).all()          # refused before anything was enqueued
