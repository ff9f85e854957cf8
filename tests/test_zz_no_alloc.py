"""GPU test of txl_rel_attn_decode_noalloc, the decode entry point for callers that cannot obtain
device memory when they call (a serving process whose device memory is a pre-sized arena, a plugin
whose interface passes only inputs and outputs, a generation loop that cannot afford cudaMalloc):
it keeps its partial results in the library's fixed scratch array instead of a caller workspace.

Called through the C ABI on two different calls in a row on one stream (so a stale scratch from the
first call would show in the second), each checked against txl_rel_attn_decode with a workspace
within the bf16 tolerance of the other tests.  This file is collected last."""
from __future__ import annotations

import ctypes

import pytest
import torch

import txl_inputs
from gpu_common import TOL, ld_r_for, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def txl():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import transformer_xl_relative_gb300 as m
    return m


def make_call(txl, B, H, D, L, M, valid, wp, C, seed):
    """Device inputs of one decode call, the memory stored as a ring (logical key j in slot
    (wp + j) mod M)."""
    cfg = txl_inputs.custom(B=B, H=H, D=D, d_model=2 * D, L=L, M=M, clamp_len=C, dtype="bf16", seed=seed)
    case = txl_inputs.make_case(cfg)
    q, k, v = (to_dev(case[n]) for n in ("q", "k", "v"))
    n_rows = min(M + L, C + 1)
    r = torch.empty(n_rows, H, ld_r_for(D), dtype=torch.bfloat16, device="cuda")
    txl.rel_pos_gen(case["W_R"].cuda(), r, n_rows, cfg.d_model, H, D)
    store_k = torch.zeros_like(k[:, :M])
    store_v = torch.zeros_like(v[:, :M])
    slots = (wp + torch.arange(M)) % M
    store_k[:, slots] = k[:, :M]
    store_v[:, slots] = v[:, :M]
    mem = txl.Memory(store_k, store_v, wp, valid)
    return dict(q=q, mem=mem, k_cur=k[:, M:], v_cur=v[:, M:], u=case["u"].cuda(), vb=case["vb"].cuda(),
                r=r, n_rows=n_rows, C=C)


def noalloc(txl, c, out):
    """txl_rel_attn_decode_noalloc through the C ABI."""
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


def test_noalloc_matches_the_workspace_entry_point_twice(txl):
    from transformer_xl_relative_gb300 import native
    calls = [make_call(txl, 2, 4, 64, 3, 1000, 900, 37, 500, seed=11),     # 4 chunks per (b, h)
             make_call(txl, 3, 2, 64, 1, 2200, 2200, 300, 1000, seed=12)]  # 9 chunks, other shape
    refs = [with_workspace(txl, c) for c in calls]
    outs = [torch.full_like(c["q"], float("nan")) for c in calls]
    # two calls in a row on one stream: the second reuses the scratch the first has just used
    for c, out in zip(calls, outs):
        assert noalloc(txl, c, out) == native.TXL_OK
    torch.cuda.synchronize()
    for ref, out in zip(refs, outs):
        assert torch.isfinite(out.float()).all()
        err = torch.max(torch.abs(out.float() - ref.float())).item()
        assert err <= TOL["bf16"], err
