"""GPU parity: libtxl (through its C ABI) against the fp64 oracle, element by element.

Tolerances (stated by the benchmark spec for this path): max |gpu - oracle| <= 1e-5 for the fp32 path and
<= 2e-2 for bf16 inputs with fp32 accumulation.  The bf16 cases must run the fused tcgen05
kernel (path 1); the fp32 case runs the SIMT kernel (path 2).
"""
import numpy as np
import pytest
import torch

import oracle
import txl_inputs
from gpu_common import TOL, ld_r_for, max_err, oracle_out, run_case, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def txl():
    import transformer_xl_relative_gb300 as m
    return m


# ---------------------------------------------------------------- position table
@pytest.mark.parametrize("dtype,H,D,d_model,n_rows,ld_w", [
    ("f32", 2, 8, 16, 16, 0),
    ("bf16", 16, 64, 1024, 768, 0),
    ("bf16", 10, 41, 410, 300, 416),
    ("bf16", 2, 64, 96, 200, 0),          # d_model not a multiple of 64
    ("bf16", 16, 128, 2048, 1001, 0),
    ("bf16", 4, 64, 96, 300, 0),          # two column tiles: clusters of 2, K tail
    ("bf16", 12, 64, 768, 257, 0),        # six column tiles: clusters of 2
    ("bf16", 6, 64, 384, 130, 0),         # three column tiles: one CTA per tile
])
def test_rel_pos_gen(txl, dtype, H, D, d_model, n_rows, ld_w):
    cfg = txl_inputs.custom(H=H, D=D, d_model=d_model, dtype=dtype, seed=3, ld_w=ld_w)
    _, _, W = txl_inputs.make_params(cfg)
    r = torch.full((n_rows, H, ld_r_for(D)), float("nan"), dtype=cfg.torch_dtype, device="cuda")
    txl.rel_pos_gen(W.cuda(), r, n_rows, d_model, H, D)
    torch.cuda.synchronize()
    ref = oracle.rel_table(n_rows, d_model, H, D, W[:, : H * D])
    got = r[..., :D].double().cpu().numpy()
    # bf16: R rounded to bf16 before the product, fp32 accumulation, one output rounding
    tol = 1e-5 if dtype == "f32" else 2e-2
    assert np.max(np.abs(got - ref)) <= tol
    if ld_r_for(D) > D:
        assert torch.isnan(r[..., D:].float()).all()       # padding is never written


# ---------------------------------------------------------------- fp32 tiny workload
def test_tiny_fp32(txl):
    cfg = txl_inputs.CONFIGS["tiny"]
    case = txl_inputs.make_case(cfg)
    out, _, path = run_case(cfg, case, txl)
    assert path == 2
    assert max_err(out, oracle_out(cfg, case)) <= TOL["f32"]


# ---------------------------------------------------------------- bf16 shapes on the tcgen05 path
SHAPES = [
    # B, H, D, d_model, L, M, valid, C, head_stride
    (1, 1, 64, 64, 128, 128, 128, 1000, 0),        # one query tile, one memory tile
    (2, 2, 64, 128, 200, 150, 150, 1000, 0),       # ragged query tile, M not a multiple of 128
    (1, 2, 64, 64, 1, 300, 300, 1000, 0),          # single query
    (2, 2, 64, 64, 300, 0, 0, 1000, 0),            # no memory
    (1, 2, 64, 64, 130, 260, 100, 1000, 0),        # partly valid memory
    (1, 2, 64, 64, 256, 256, 256, 100, 0),         # clamp inside the window
    (1, 1, 64, 64, 200, 200, 200, 0, 0),           # clamp 0: one position vector for all
    (1, 2, 64, 64, 384, 384, 384, 128, 0),         # clamp at a chunk boundary
    (1, 2, 64, 64, 150, 140, 140, 257, 0),
    (2, 2, 32, 64, 160, 96, 96, 1000, 0),          # D = 32
    (2, 2, 16, 32, 64, 64, 64, 1000, 0),           # D = 16
    (2, 3, 41, 82, 150, 150, 150, 1000, 48),       # D = 41, padded head stride
    (1, 2, 96, 192, 200, 128, 128, 1000, 0),       # two 64-column atoms
    (1, 2, 128, 256, 256, 256, 256, 1000, 0),      # D = 128
    (1, 1, 128, 128, 130, 300, 250, 200, 0),       # D = 128, partial memory, clamp
    # one CTA per SM over all (b, h, query tile) items: odd L (the odd-row q map has fewer rows),
    # tiny L, more items than SMs in odd counts, and more than 32 query tiles per sequence (items
    # dealt in serpentine order instead of the balanced count table)
    (1, 2, 64, 64, 129, 128, 128, 1000, 0),
    (1, 1, 64, 64, 3, 5, 5, 1000, 0),
    (3, 5, 64, 128, 257, 200, 180, 300, 0),
    (13, 16, 64, 128, 256, 128, 128, 1000, 0),
    (1, 1, 64, 64, 4160, 0, 0, 1000, 0),
]


@pytest.mark.parametrize("shape", SHAPES, ids=[
    "B%dH%dD%d_L%dM%dv%dC%d" % (s[0], s[1], s[2], s[4], s[5], s[6], s[7]) for s in SHAPES])
def test_bf16_shapes(txl, shape):
    B, H, D, dm, L, M, valid, C, hs = shape
    cfg = txl_inputs.custom(B=B, H=H, D=D, d_model=dm, L=L, M=M, clamp_len=C, dtype="bf16",
                            seed=100 + D + L + M, head_stride=hs)
    case = txl_inputs.make_case(cfg)
    out, _, path = run_case(cfg, case, txl, valid=valid)
    assert path == 1
    err = max_err(out, oracle_out(cfg, case, valid=valid))
    assert err <= TOL["bf16"], err


# ---------------------------------------------------------------- the workloads at full size
@pytest.mark.parametrize("name", ["base", "large", "longmem"])
def test_workload_full(txl, name):
    cfg = txl_inputs.CONFIGS[name]
    case = txl_inputs.make_case(cfg)
    out, _, path = run_case(cfg, case, txl)
    assert path == 1
    err = max_err(out, oracle_out(cfg, case))
    assert err <= TOL["bf16"], err


# ---------------------------------------------------------------- output views without 16-byte rows
@pytest.mark.parametrize("D", [64, 128])
def test_out_view_unaligned(txl, D):
    """An output view whose head stride is not a multiple of 16 bytes takes the scalar stores of
    the fused kernels: the same values as a contiguous output, nothing written outside the view."""
    cfg = txl_inputs.custom(B=2, H=3, D=D, d_model=2 * D, L=200, M=150, clamp_len=1000, dtype="bf16",
                            seed=77 + D)
    case = txl_inputs.make_case(cfg)
    out, r, path = run_case(cfg, case, txl)
    assert path == 1
    q, k, v = (to_dev(case[n]) for n in ("q", "k", "v"))
    M = cfg.M
    mem = txl.Memory(k[:, :M], v[:, :M], 0, M)
    store = torch.full((cfg.B, cfg.L, cfg.H, D + 1), 7.0, dtype=torch.bfloat16, device="cuda")
    out2 = store[..., :D]
    txl.rel_attn_fwd(q, mem, k[:, M:], v[:, M:], case["u"].cuda(), case["vb"].cuda(), r, r.shape[0],
                     cfg.clamp_len, out2)
    torch.cuda.synchronize()
    assert torch.equal(out, out2)
    assert bool((store[..., D] == 7.0).all())
