"""Shared helpers of the GPU tests: move seeded inputs to the device (keeping padded layouts),
run the library path through its Python binding, and compare with the fp64 oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import txl_inputs

TOL = {"f32": 1e-5, "bf16": 2e-2}     # max abs error on outputs (fp32 path / bf16 with fp32 acc)


def to_dev(t: torch.Tensor, head_stride: int | None = None, device="cuda") -> torch.Tensor:
    """Copy a CPU tensor to the device; a [..., D] view is placed in [..., head_stride] storage."""
    if head_stride is None or head_stride == t.shape[-1]:
        return t.contiguous().to(device)
    store = torch.zeros(*t.shape[:-1], head_stride, dtype=t.dtype, device=device)
    view = store[..., : t.shape[-1]]
    view.copy_(t.to(device))
    return view


def ld_r_for(D: int) -> int:
    return (D + 7) // 8 * 8


def run_case(cfg, case, txl, M=None, valid=None, clamp_len=None, r_override=None, L=None):
    """rel_pos_gen + rel_attn_fwd on one call's inputs; returns (out, r, path)."""
    M = cfg.M if M is None else M
    valid = M if valid is None else valid
    C = cfg.clamp_len if clamp_len is None else clamp_len
    q, k, v = (to_dev(case[n], cfg.hs) for n in ("q", "k", "v"))
    L = q.shape[1]
    u, vb = case["u"].cuda(), case["vb"].cuda()
    W = case["W_R"].cuda()
    dt = cfg.torch_dtype
    n_rows = min(M + L, C + 1)
    if r_override is not None:
        r = r_override.cuda()
        n_rows = r.shape[0]
    else:
        r = torch.empty(n_rows, cfg.H, ld_r_for(cfg.D), dtype=dt, device="cuda")
        txl.rel_pos_gen(W, r, n_rows, cfg.d_model, cfg.H, cfg.D)
    mem = txl.Memory(k[:, :M], v[:, :M], 0, valid) if M > 0 else None
    out = to_dev(torch.zeros_like(case["q"]), cfg.hs)
    path = txl.rel_attn_path(q, mem, k[:, M:], v[:, M:], r, out)
    txl.rel_attn_fwd(q, mem, k[:, M:], v[:, M:], u, vb, r, n_rows, C, out)
    torch.cuda.synchronize()
    return out, r, path


def oracle_out(cfg, case, M=None, valid=None, clamp_len=None, rows=None):
    M = cfg.M if M is None else M
    valid = M if valid is None else valid
    C = cfg.clamp_len if clamp_len is None else clamp_len
    return oracle.rel_attn(case["q"], case["k"], case["v"], case["u"], case["vb"],
                           case["W_R"][:, : cfg.H * cfg.D], M, valid, C, rows=rows)


def max_err(out: torch.Tensor, ref: np.ndarray, rows=None) -> float:
    got = out.detach().to(torch.float64).cpu().numpy()
    if rows is None:
        return float(np.max(np.abs(got - ref)))
    errs = [np.max(np.abs(got[b, i, h] - ref[b, i, h])) for b, h, i in rows]
    return float(max(errs))
