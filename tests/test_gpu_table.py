"""GPU parity of the learned-table variant (txl_rel_attn_table_fwd, "TransformerXL 相对位置编码" §3.1)
against the fp64 oracle (oracle.table_attn): bidirectional attention with the clamped
non-negative relative index, the page's scaling of the four terms and its -1e9 key masking.
Tolerances as for the main path: 1e-5 (fp32), 2e-2 (bf16 inputs, fp32 arithmetic)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import txl_inputs
from gpu_common import TOL, ld_r_for, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def txl():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import transformer_xl_relative_gb300 as m
    return m


TABLE = [
    # B, H, D, L, max_len, dtype, mask kind, head_stride
    (2, 4, 32, 10, 512, "f32", "none", 0),      # the page's example sizes (d_model 128 = 4 x 32)
    (2, 4, 64, 200, 64, "bf16", "random", 0),   # L > max_len: the index clamps at both ends
    (3, 3, 41, 37, 16, "bf16", "one_empty", 48),  # padded heads; batch entry 1 has every key masked
    (2, 2, 128, 33, 8, "f32", "random", 0),     # D = 128, L not a multiple of four
    # bf16 with d_head 64 and 16-byte rows takes a tensor-core kernel: one position, a ragged
    # key tile with a fully masked batch entry, the bench's per-head shape, a table of five rows
    # (nearly every pair clamped); a 68-element head stride keeps d_head 64 on the SIMT kernel
    (1, 2, 64, 1, 4, "bf16", "none", 0),
    (2, 2, 64, 130, 512, "bf16", "one_empty", 0),
    (1, 3, 64, 384, 512, "bf16", "none", 0),
    (1, 2, 64, 70, 3, "bf16", "random", 0),
    (1, 2, 64, 50, 16, "bf16", "none", 68),
    # unmasked bf16 with L <= max_len and d_head <= 64 takes the persistent tcgen05 kernel in its
    # learned-table mode: a ragged last key tile (130 = 128 + 2 keys), L == max_len (the first and
    # the last row of the table both used), padded heads with d_head 41, three query tiles with a
    # ragged tail, and more (b, h) items than SMs
    (2, 2, 64, 130, 512, "bf16", "none", 0),
    (1, 2, 64, 257, 257, "bf16", "none", 0),
    (2, 3, 41, 200, 300, "bf16", "none", 48),
    (1, 4, 64, 300, 400, "bf16", "none", 0),
    (8, 24, 32, 128, 128, "bf16", "none", 0),
    # ... and with a key mask (masked keys read a score of about -1e30 from the ring): random masks
    # over three query tiles and over padded heads; the one_empty case above (L = 130) takes it too
    (2, 3, 64, 300, 512, "bf16", "random", 0),
    (1, 2, 41, 150, 200, "bf16", "random", 48),
]


@pytest.mark.parametrize("shape", TABLE, ids=["B%dH%dD%d_L%d_max%d_%s_%s" % s[:7] for s in TABLE])
def test_table_variant_matches_oracle(txl, shape):
    B, H, D, L, max_len, dtype, mk, hs = shape
    cfg = txl_inputs.custom(B=B, H=H, D=D, d_model=2 * D, L=L, M=0, dtype=dtype, seed=700 + L, head_stride=hs)
    q, k, v = txl_inputs.make_qkv(cfg, seed=701 + L, L=L, T=L)
    u, vb, _ = txl_inputs.make_params(cfg, seed=702 + L)
    nt = 2 * max_len - 1
    rt = txl_inputs.make_matrix(nt, H * D, seed=703 + L, dtype=cfg.torch_dtype).reshape(nt, H, D)
    mask = None
    if mk != "none":
        gen = torch.Generator().manual_seed(704 + L)
        mask = (torch.rand(B, L, generator=gen) > 0.25).to(torch.uint8)
        if mk == "one_empty":
            mask[1] = 0
    r_dev = torch.zeros(nt, H, ld_r_for(D), dtype=cfg.torch_dtype, device="cuda")
    r_dev[..., :D] = rt.cuda()
    out = to_dev(torch.full_like(q, float("nan")), cfg.hs)
    qd, kd, vd = to_dev(q, cfg.hs), to_dev(k, cfg.hs), to_dev(v, cfg.hs)
    md = mask.cuda() if mask is not None else None
    # the route the host takes: the persistent tcgen05 kernel for bf16, d_head <= 64, L <= max_len and
    # 16-byte rows; the mma.sync kernel for the other bf16 calls with d_head 64 and 16-byte rows
    path = txl.rel_attn_table_path(qd, kd, vd, r_dev, max_len, out, key_mask=md)
    if dtype == "bf16" and D <= 64 and L <= max_len and hs != 68:
        assert path == 1, path
    elif dtype == "bf16" and D == 64 and hs == 0:
        assert path == 3, path
    else:
        assert path in (2, 3), path
    txl.rel_attn_table_fwd(qd, kd, vd, u.cuda(), vb.cuda(), r_dev, max_len, out, key_mask=md)
    torch.cuda.synchronize()
    ref = oracle.table_attn(q, k, v, u, vb, rt, max_len, key_mask=mask.numpy() if mask is not None else None)
    err = np.max(np.abs(out.double().cpu().numpy() - ref))
    assert np.isfinite(err) and err <= TOL[dtype], err


def test_table_from_a_projected_learned_table(txl):
    """The page's composition: r_table = pos_emb W_R, projected with txl_linear, then the variant."""
    B, H, D, L, max_len, dm = 2, 4, 64, 96, 64, 256
    cfg = txl_inputs.custom(B=B, H=H, D=D, d_model=dm, L=L, M=0, dtype="bf16", seed=77)
    q, k, v = txl_inputs.make_qkv(cfg, seed=78, L=L, T=L)
    u, vb, W = txl_inputs.make_params(cfg, seed=79)
    pos_emb = txl_inputs.make_matrix(2 * max_len - 1, dm, seed=80)
    r = txl.linear(pos_emb.cuda(), W[:, :H * D].contiguous().cuda()).view(2 * max_len - 1, H, D)
    out = torch.empty_like(q).cuda()
    txl.rel_attn_table_fwd(q.cuda(), k.cuda(), v.cuda(), u.cuda(), vb.cuda(), r, max_len, out)
    torch.cuda.synchronize()
    # the oracle projects the same learned table itself, in fp64 (the GPU table is rounded to bf16
    # once, which the bf16 tolerance covers)
    r_ref = oracle.linear(pos_emb, W[:, :H * D]).reshape(2 * max_len - 1, H, D)
    ref = oracle.table_attn(q, k, v, u, vb, r_ref, max_len)
    assert np.max(np.abs(out.double().cpu().numpy() - ref)) <= TOL["bf16"]


def test_table_large_workload_sampled(txl):
    """The bench's table-variant workload at full size (B16 L384 H16 D64 max_len 512, bf16: the
    tensor-core kernel): sampled (b, h) pairs against the oracle on those slices."""
    B, H, D, L, max_len = 16, 16, 64, 384, 512
    cfg = txl_inputs.custom(B=B, H=H, D=D, d_model=2 * D, L=L, M=0, dtype="bf16", seed=5151)
    q, k, v = txl_inputs.make_qkv(cfg, seed=5152, L=L, T=L)
    u, vb, _ = txl_inputs.make_params(cfg, seed=5153)
    nt = 2 * max_len - 1
    rt = txl_inputs.make_matrix(nt, H * D, seed=5154, dtype=torch.bfloat16).reshape(nt, H, D)
    out = torch.empty_like(q).cuda()
    txl.rel_attn_table_fwd(q.cuda(), k.cuda(), v.cuda(), u.cuda(), vb.cuda(), rt.cuda(), max_len, out)
    torch.cuda.synchronize()
    for b, h in [(0, 0), (9, 4), (15, 15)]:
        sl = (slice(b, b + 1), slice(None), slice(h, h + 1))
        ref = oracle.table_attn(q[sl], k[sl], v[sl], u[h:h + 1], vb[h:h + 1], rt[:, h:h + 1], max_len)
        err = np.max(np.abs(out[sl].double().cpu().numpy() - ref))
        assert err <= TOL["bf16"], (b, h, err)


def test_table_large_workload_masked_sampled(txl):
    """The same full-size workload with a random key mask (a quarter of the keys masked, batch entry
    3 fully masked): the persistent kernel's masked instantiation, sampled (b, h) slices."""
    B, H, D, L, max_len = 16, 16, 64, 384, 512
    cfg = txl_inputs.custom(B=B, H=H, D=D, d_model=2 * D, L=L, M=0, dtype="bf16", seed=6161)
    q, k, v = txl_inputs.make_qkv(cfg, seed=6162, L=L, T=L)
    u, vb, _ = txl_inputs.make_params(cfg, seed=6163)
    nt = 2 * max_len - 1
    rt = txl_inputs.make_matrix(nt, H * D, seed=6164, dtype=torch.bfloat16).reshape(nt, H, D)
    gen = torch.Generator().manual_seed(6165)
    mask = (torch.rand(B, L, generator=gen) > 0.25).to(torch.uint8)
    mask[3] = 0
    out = torch.empty_like(q).cuda()
    qd, kd, vd, rd, md = q.cuda(), k.cuda(), v.cuda(), rt.cuda(), mask.cuda()
    assert txl.rel_attn_table_path(qd, kd, vd, rd, max_len, out, key_mask=md) == 1
    txl.rel_attn_table_fwd(qd, kd, vd, u.cuda(), vb.cuda(), rd, max_len, out, key_mask=md)
    torch.cuda.synchronize()
    for b, h in [(0, 0), (3, 7), (15, 15)]:
        sl = (slice(b, b + 1), slice(None), slice(h, h + 1))
        ref = oracle.table_attn(q[sl], k[sl], v[sl], u[h:h + 1], vb[h:h + 1], rt[:, h:h + 1], max_len,
                                key_mask=mask[b:b + 1].numpy())
        err = np.max(np.abs(out[sl].double().cpu().numpy() - ref))
        assert err <= TOL["bf16"], (b, h, err)
