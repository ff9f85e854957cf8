"""GPU tests of the FIFO K/V memory (txl_mem_push) and of attention over it.

Push is byte work: compared bit-exactly with the oracle's FIFO.  Streaming attention over the
ring is compared with the oracle evaluated on the concatenated sequence ("Transformer-XL 和相对
位置编码" §2.3.1: each segment attends to the cached previous positions plus itself).
"""
import numpy as np
import pytest
import torch

import oracle
import txl_inputs
from gpu_common import TOL, ld_r_for, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def txl():
    import transformer_xl_relative_gb300 as m
    return m


@pytest.mark.parametrize("dtype,B,H,D,M,L,S,hs", [
    (torch.bfloat16, 2, 3, 64, 6, 4, 5, 0),
    (torch.bfloat16, 2, 2, 64, 4, 4, 3, 0),
    (torch.bfloat16, 1, 2, 64, 3, 5, 3, 0),        # segment longer than the memory
    (torch.bfloat16, 2, 2, 41, 7, 3, 6, 48),       # scalar copy path
    (torch.float32, 2, 2, 8, 5, 2, 7, 0),
    (torch.bfloat16, 1, 4, 128, 256, 96, 5, 0),
])
def test_push_matches_fifo(txl, dtype, B, H, D, M, L, S, hs):
    g = torch.Generator().manual_seed(5)
    ring = txl.Memory.empty(B, M, H, D, dtype=dtype, device="cuda", head_stride=hs or None)
    rk = np.zeros((B, M, H, D), dtype=np.float32)
    rv = np.zeros_like(rk)
    wp, valid = 0, 0
    for s in range(S):
        kn = torch.randn(B, L, H, D, generator=g).to(dtype)
        vn = torch.randn(B, L, H, D, generator=g).to(dtype)
        txl.mem_push(ring, to_dev(kn, hs or None), to_dev(vn, hs or None))
        rk, rv, wp, valid = oracle.ring_push(rk, rv, wp, valid, kn.float().numpy(), vn.float().numpy())
        assert ring.state() == (wp, valid)
        torch.cuda.synchronize()
        assert np.array_equal(ring.k.float().cpu().numpy(), rk)
        assert np.array_equal(ring.v.float().cpu().numpy(), rv)


def _stream_run(txl, cfg, segs, ring, rows_per_seg, seed_rows, start=0, stop=None):
    """Run segments start..stop-1 through attention + push; return {s: (out, rows)}."""
    u, vb, W = txl_inputs.make_params(cfg, cfg.seed + 10_000)
    dt = cfg.torch_dtype
    n_rows = min(cfg.M + cfg.L, cfg.clamp_len + 1)
    r = torch.empty(n_rows, cfg.H, ld_r_for(cfg.D), dtype=dt, device="cuda")
    txl.rel_pos_gen(W.cuda(), r, n_rows, cfg.d_model, cfg.H, cfg.D)
    uu, vv = u.cuda(), vb.cuda()
    rng = np.random.default_rng(seed_rows)
    results = {}
    stop = cfg.segments if stop is None else stop
    for s in range(start, stop):
        q, k, v = segs[s]
        qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
        out = torch.empty_like(qd)
        path = txl.rel_attn_path(qd, ring, kd, vd, r, out)
        txl.rel_attn_fwd(qd, ring, kd, vd, uu, vv, r, n_rows, cfg.clamp_len, out)
        txl.mem_push(ring, kd, vd)
        rows = [(int(rng.integers(cfg.B)), int(rng.integers(cfg.H)), int(rng.integers(cfg.L)))
                for _ in range(rows_per_seg)]
        results[s] = (out.cpu(), rows, path)
    return results, (u, vb, W)


def _check_against_concat(cfg, segs, results, params, per_segment=None):
    u, vb, W = params
    q = torch.cat([segs[s][0] for s in range(cfg.segments)], dim=1)
    k = torch.cat([segs[s][1] for s in range(cfg.segments)], dim=1)
    v = torch.cat([segs[s][2] for s in range(cfg.segments)], dim=1)
    sel = []
    for s, (_, rows, _) in results.items():
        sel += [(b, h, s * cfg.L + i) for b, h, i in rows]
    ref = oracle.stream_attn(q, k, v, u, vb, W[:, : cfg.H * cfg.D], cfg.L, cfg.M, cfg.clamp_len,
                             rows=sel)
    worst = 0.0
    for s, (out, rows, _) in results.items():
        o = out.double().numpy()
        seg_worst = 0.0
        for b, h, i in rows:
            e = float(np.max(np.abs(o[b, i, h] - ref[b, s * cfg.L + i, h])))
            seg_worst = max(seg_worst, e)
            if per_segment is not None and e > TOL["bf16"]:
                per_segment.setdefault("bad_rows", []).append((s, b, h, i, e))
        if per_segment is not None:
            per_segment[s] = seg_worst
        worst = max(worst, seg_worst)
    return worst


def test_stream_workload_sampled(txl):
    """8 segments, ring starts empty, each segment pushed after its attention; sampled rows of
    every segment checked against the concatenated-sequence oracle."""
    cfg = txl_inputs.CONFIGS["stream"]
    segs = [txl_inputs.make_segment(cfg, s) for s in range(cfg.segments)]
    ring = txl.Memory.empty(cfg.B, cfg.M, cfg.H, cfg.D, dtype=cfg.torch_dtype)
    results, params = _stream_run(txl, cfg, segs, ring, rows_per_seg=48, seed_rows=1)
    assert all(p == 1 for (_, _, p) in results.values())        # aligned ring: fused kernel
    per_seg = {}
    worst = _check_against_concat(cfg, segs, results, params, per_seg)
    assert worst <= TOL["bf16"], per_seg


@pytest.mark.parametrize("L,M,S,D", [(100, 300, 5, 64), (128, 384, 5, 64), (64, 96, 6, 128)])
def test_stream_small_every_row(txl, L, M, S, D):
    """Rings whose write pointer is not a multiple of 128 (SIMT path) and aligned ones (fused
    path); every row of every segment checked."""
    cfg = txl_inputs.custom(B=2, H=2, D=D, d_model=2 * D, L=L, M=M, clamp_len=200, dtype="bf16",
                            seed=77, segments=S)
    segs = [txl_inputs.make_segment(cfg, s) for s in range(S)]
    ring = txl.Memory.empty(cfg.B, cfg.M, cfg.H, cfg.D, dtype=cfg.torch_dtype)
    results, params = _stream_run(txl, cfg, segs, ring, rows_per_seg=0, seed_rows=2)
    full = [(b, h, i) for b in range(cfg.B) for h in range(cfg.H) for i in range(cfg.L)]
    results = {s: (o, full, p) for s, (o, _, p) in results.items()}
    assert _check_against_concat(cfg, segs, results, params) <= TOL["bf16"]


def test_checkpoint_resume_is_bit_identical(txl):
    """Ring buffers + (wp, valid) are the whole state: a copy restored into fresh tensors
    continues the stream with bit-identical outputs."""
    cfg = txl_inputs.custom(B=2, H=2, D=64, d_model=128, L=128, M=256, clamp_len=300,
                            dtype="bf16", seed=9, segments=6)
    segs = [txl_inputs.make_segment(cfg, s) for s in range(cfg.segments)]
    ring = txl.Memory.empty(cfg.B, cfg.M, cfg.H, cfg.D)
    _stream_run(txl, cfg, segs, ring, 0, 3, start=0, stop=3)
    saved_k, saved_v, state = ring.k.clone(), ring.v.clone(), ring.state()
    a, _ = _stream_run(txl, cfg, segs, ring, 0, 3, start=3, stop=6)
    ring2 = txl.Memory(saved_k.clone(), saved_v.clone())
    ring2.restore(*state)
    b, _ = _stream_run(txl, cfg, segs, ring2, 0, 3, start=3, stop=6)
    for s in range(3, 6):
        assert torch.equal(a[s][0], b[s][0])
    assert torch.equal(ring.k, ring2.k) and ring.state() == ring2.state()
