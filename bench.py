"""Benchmark of the Transformer-XL relative-attention hot path on GB300.

One step = one pass of the whole path over one batch of the workload:
    txl_rel_pos_gen  (sinusoid R on chip, r = R W_R, tcgen05)
    txl_rel_attn_fwd (fused TMA + tcgen05 attention over [memory ++ current])
    txl_mem_push     (FIFO update of the K/V memory with the current segment)
on the large workload (B16 H16 D64 L384 M384, clamp 1000, bf16).  Inputs are resident in HBM;
four input sets (252 MB > 129 MB L2) rotate so no step reads L2-warm inputs.  Steps are replayed
from a CUDA graph of four consecutive steps (no host launch overhead in the timed region).

Prints one JSON line (rank 0).  ``--impl reference`` times the fp64 oracle on the host cores on
bounded samples of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "large"        # B16 H16 D64 L384 M384 clamp 1000 bf16


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return d["bf16_tflops"], d.get("bf16_tflops_sustained"), d["hbm_gbs"], "measured"
    except Exception:
        return 1900.0, 1700.0, 6800.0, "fallback"


NOMINAL_BF16_TFLOPS = 2250.0     # GB300 dense bf16 tensor rate, nominal (2:4-sparse figures are 2x)
NOMINAL_HBM_GBS = 7900.0         # GB300 HBM3e bandwidth, nominal

METRIC = "rel-attn TFLOP/s (L384 M384 H16 D64 bf16), whole step: pos-gen + fused attention + memory push"
WORKLOAD_NAME = "large: B16 H16 D64 d_model1024 L384 M384 clamp1000 (per GPU)"


def _flops(cfg):
    import oracle
    attn = oracle.attn_flops(cfg.B, cfg.H, cfg.D, cfg.L, cfg.M)
    pos = 2 * cfg.n_rows * cfg.d_model * cfg.H * cfg.D
    return attn, pos


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.rows.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        sel = [p for (t, p) in self.rows if t0 <= t <= t1]
        if not sel:
            sel = [p for (_, p) in self.rows]
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        mhz = sorted(float(p[1]) for p in sel if p[1].replace(".", "").isdigit())
        mx = max((float(p[2]) for p in sel if p[2].replace(".", "").isdigit()), default=None)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for p in sel for k in range(4) if p[5 + k].lower() == "active"})
        return {"sm_mhz": mhz[len(mhz) // 2] if mhz else None, "sm_max_mhz": mx,
                "reasons": reasons, "samples": len(sel)}


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_value(world: int, step_flops: float, t_step_ms_max: float) -> float:
    """Whole-job TFLOP/s of weak scaling: every rank runs one full replica of the workload per
    step, and the job's step time is the slowest rank's."""
    return world * step_flops / (t_step_ms_max * 1e-3) / 1e12


def rank_seed(base: int, rank: int) -> int:
    """Each replica draws its own inputs."""
    return base + 7919 * rank


def _barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _profile_traffic(kernel_src: str, summary: str = "rel_attn_fwd_large.json"):
    """DRAM bytes per launch of a kernel from its committed ncu summary, if it was taken on the
    current kernel source (sha256 recorded next to it); else None."""
    path = os.path.join(ROOT, "profiles", summary)
    try:
        with open(path) as f:
            d = json.load(f)
        with open(kernel_src, "rb") as f:
            sha = hashlib.sha256(f.read()).hexdigest()
        if d.get("kernel_sha256") == sha:
            return d.get("dram_bytes_per_launch")
    except Exception:
        pass
    return None


def cpu_baseline(cfg, target_s: float = 12.0, threads=None):
    """The oracle as it stands on the host cores, on a bounded sample of the workload: whole
    batch entries (every head and query) until about target_s seconds of work."""
    import oracle
    import txl_inputs
    threads = threads or (os.cpu_count() or 1)
    case = txl_inputs.make_case(cfg)
    from oracle.oracle import _f64
    q, k, v, u, vb = (_f64(case[n]) for n in ("q", "k", "v", "u", "vb"))
    W = _f64(case["W_R"][:, : cfg.H * cfg.D])
    t_total, nb = 0.0, 0
    while nb < cfg.B and t_total < target_s:
        rows = [(nb, h, i) for h in range(cfg.H) for i in range(cfg.L)]
        t0 = time.perf_counter()
        oracle.rel_attn(q, k, v, u, vb, W, cfg.M, cfg.M, cfg.clamp_len, threads=threads, rows=rows)
        t_total += time.perf_counter() - t0
        nb += 1
    # the metric's flops for the sampled share of one step: attention of nb batch entries plus
    # nb / B of the position table's product (the oracle recomputes it per call, as it stands)
    attn, pos = _flops(cfg)
    done_flops = (attn + pos) * nb / cfg.B
    return {"value": done_flops / t_total / 1e12, "unit": "TFLOP/s", "cores": threads,
            "kind": "oracle",
            "sample": "%d of %d batch entries (all %d heads x %d queries), fp64, %.1f s" % (
                nb, cfg.B, cfg.H, cfg.L, t_total)}


def row_baselines(threads=None) -> dict:
    """The oracle as it stands, timed on the host cores beside each of the next-row measurements,
    on a bounded sample of its workload (a few seconds each), scaled to the sub-bench's unit."""
    import numpy as np
    import oracle
    threads = threads or (os.cpu_count() or 1)
    rng = np.random.default_rng(99)
    res = {}
    # decode: B8 H16 D64 L1 M4096 clamp 1000; sampled (b, h) pairs of the single query
    B, H, D, L, M, C, dm = 8, 16, 64, 1, 4096, 1000, 1024
    q = rng.standard_normal((1, L, H, D)); k = rng.standard_normal((1, M + L, H, D))
    v = rng.standard_normal((1, M + L, H, D)); u = 0.02 * rng.standard_normal((H, D))
    vb = 0.02 * rng.standard_normal((H, D)); W = rng.standard_normal((dm, H * D)) * dm ** -0.5
    t0 = time.perf_counter()
    oracle.rel_attn(q, k, v, u, vb, W, M, M, C, threads=threads, rows=[(0, h, 0) for h in range(H)])
    t = time.perf_counter() - t0
    res["decode"] = {"value": 1e6 * t * B, "unit": "us per call", "cores": threads, "kind": "oracle",
                     "sample": "1 of 8 batch entries (16 heads, the position table included), fp64, %.1f s" % t}
    # layer: B16 L384 M384 H16 D64 d_model 1024; one batch entry, every head and position
    L, M, C = 384, 384, 1000
    h_mem = rng.standard_normal((1, M, dm)); hh = rng.standard_normal((1, L, dm))
    Wq, Wk, Wv = (rng.standard_normal((dm, H * D)) * dm ** -0.5 for _ in range(3))
    Wo = rng.standard_normal((H * D, dm)) * (H * D) ** -0.5
    t0 = time.perf_counter()
    oracle.rel_layer(h_mem, hh, Wq, Wk, Wv, Wo, u, vb, W, H, D, M, C, threads=threads)
    t = time.perf_counter() - t0
    res["layer"] = {"value": oracle.layer_flops(1, H, D, L, M, dm) / t / 1e12, "unit": "TFLOP/s", "cores": threads,
                    "kind": "oracle", "sample": "1 of 16 batch entries (every head and position), fp64, %.1f s" % t}
    # backward: the large workload's call; two (b, h) pairs of one batch entry
    q = rng.standard_normal((1, L, H, D)); k = rng.standard_normal((1, M + L, H, D))
    v = rng.standard_normal((1, M + L, H, D)); dO = rng.standard_normal((1, L, H, D))
    t0 = time.perf_counter()
    oracle.rel_attn_bwd(q, k, v, u, vb, W, M, M, C, dO, bh=[(0, 0), (0, 1)])
    t = time.perf_counter() - t0
    f_attn, _ = bwd_flops(1, 2, D, L, M, min(M + L, C + 1), dm)          # the two sampled (b, h)
    _, f_pos = bwd_flops(1, H, D, L, M, min(M + L, C + 1), dm)           # dW_R is taken whole
    res["backward"] = {"value": (f_attn + f_pos) / t / 1e12, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                       "sample": "2 of 256 (b, h) pairs (numpy, the position table and dW_R included), fp64, %.1f s" % t}
    # table variant: B16 L384 H16 D64 max_len 512; four batch entries, every head
    qt, kt, vt = (rng.standard_normal((4, L, H, D)) for _ in range(3))
    rt = rng.standard_normal((1023, H, D))
    t0 = time.perf_counter()
    oracle.table_attn(qt, kt, vt, u, vb, rt, 512)
    t = time.perf_counter() - t0
    res["table"] = {"value": 6 * D * 4 * H * L * L / t / 1e12, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                    "sample": "4 of 16 batch entries, every head (numpy), fp64, %.1f s" % t}
    return res


def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return 0
    import txl_inputs
    cfg = txl_inputs.CONFIGS[WORKLOAD]
    for _ in range(args.warmup):
        cpu_baseline(cfg, target_s=0.5)
    vals, t0 = [], time.perf_counter()
    for _ in range(args.steps):
        vals.append(cpu_baseline(cfg, target_s=max(1.0, 60.0 / max(args.steps, 1))))
    dt = time.perf_counter() - t0
    value = sum(v["value"] for v in vals) / len(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value,
        "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * dt / max(args.steps, 1), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD_NAME, "sample": vals[-1]["sample"]},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": vals[-1]["cores"],
                         "kind": "oracle", "sample": vals[-1]["sample"]},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def _graph_us(stream, fn, n_calls, reps):
    """Mean device time per call of `fn(i)`, i = 0 .. n_calls-1 captured in one CUDA graph and
    replayed `reps` times back to back (CUDA events on the launching stream)."""
    import torch
    with torch.cuda.stream(stream):
        for i in range(n_calls):
            fn(i)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(n_calls):
            fn(i)
    with torch.cuda.stream(stream):
        graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            graph.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / (n_calls * reps)


def _padded_randn(g, shape, hs, dt, device):
    """[..., D] N(0, 1) values in [..., hs] storage (the base workload's 48-element head stride)."""
    import torch
    D = shape[-1]
    x = torch.randn(*shape, generator=g, device=device).to(dt)
    if hs == D:
        return x
    store = torch.zeros(*shape[:-1], hs, dtype=dt, device=device)
    store[..., :D] = x
    return store[..., :D]


def _oracle_sample(cfg, rows, mem_valid=None, stream=False, threads=None):
    """The oracle as it stands, on the host cores, for the listed (b, h, i) rows of one call (or of
    the concatenated stream): (seconds, algorithmic flops of the sampled rows)."""
    import oracle
    import txl_inputs
    from oracle.oracle import _f64
    threads = threads or (os.cpu_count() or 1)
    u, vb, W = txl_inputs.make_params(cfg, cfg.seed + 10_000)
    W = _f64(W[:, : cfg.H * cfg.D])
    if not stream:
        q, k, v = txl_inputs.make_qkv(cfg, cfg.seed)
        valid = cfg.M if mem_valid is None else mem_valid
        t0 = time.perf_counter()
        oracle.rel_attn(q, k, v, u, vb, W, cfg.M, valid, cfg.clamp_len, threads=threads, rows=rows)
        dt = time.perf_counter() - t0
        keys = [valid + i + 1 for (_, _, i) in rows]
    else:
        import torch
        segs = [txl_inputs.make_segment(cfg, s_) for s_ in range(cfg.segments)]
        q, k, v = (torch.cat([sg[j] for sg in segs], dim=1) for j in range(3))
        t0 = time.perf_counter()
        oracle.stream_attn(q, k, v, u, vb, W, cfg.L, cfg.M, cfg.clamp_len, threads=threads, rows=rows)
        dt = time.perf_counter() - t0
        keys = [t - max(0, (t // cfg.L) * cfg.L - cfg.M) + 1 for (_, _, t) in rows]
    return dt, 6 * cfg.D * sum(keys), threads


def bench_configs(txl, device, stream, rank, args, with_oracle, legs=("base", "longmem", "stream")):
    """The other synthetic workloads at one GPU: base (B32 H10 D41 L150 M150), long memory
    (B8 H16 D64 L128 M1600) and the 8-segment stream through the FIFO memory (B4 H16 D128 L512
    M2048).  Each reports the attention kernel's time per call, TFLOP/s (6 D per visible pair),
    query tokens/s and its fraction of the bound it sits under, plus the oracle on a sample."""
    import torch
    import oracle
    import txl_inputs
    peak, _, hbm, kind = _peaks()
    out = {}
    for name in [n for n in ("base", "longmem") if n in legs]:
        cfg = txl_inputs.CONFIGS[name]
        B, H, D, L, M, C, hs = cfg.B, cfg.H, cfg.D, cfg.L, cfg.M, cfg.clamp_len, cfg.hs
        dt = cfg.torch_dtype
        g = torch.Generator(device=device).manual_seed(rank_seed(cfg.seed, rank))
        per_set = 2 * B * (2 * (M + L) + 2 * L) * H * hs                       # q, k, v, out bytes
        nsets = max(2, min(8, -(-400_000_000 // per_set)))   # rotate > L2
        sets = [(_padded_randn(g, (B, L, H, D), hs, dt, device), _padded_randn(g, (B, M + L, H, D), hs, dt, device),
                 _padded_randn(g, (B, M + L, H, D), hs, dt, device), _padded_randn(g, (B, L, H, D), hs, dt, device))
                for _ in range(nsets)]
        mems = [txl.Memory.full(k[:, :M], v[:, :M]) for (_, k, v, _) in sets]
        u = (0.02 * torch.randn(H, D, generator=g, device=device)).float()
        vb = (0.02 * torch.randn(H, D, generator=g, device=device)).float()
        W = torch.zeros(cfg.d_model, cfg.ldw, dtype=dt, device=device)
        W[:, : H * D] = (torch.randn(cfg.d_model, H * D, generator=g, device=device) * cfg.d_model ** -0.5).to(dt)
        ld_r = (D + 7) // 8 * 8
        r = torch.empty(cfg.n_rows, H, ld_r, dtype=dt, device=device)
        txl.rel_pos_gen(W, r, cfg.n_rows, cfg.d_model, H, D)
        q0, k0, v0, o0 = sets[0]
        path = txl.rel_attn_path(q0, mems[0], k0[:, M:], v0[:, M:], r, o0)

        def call(i):
            q, k, v, o = sets[i % nsets]
            txl.rel_attn_fwd(q, mems[i % nsets], k[:, M:], v[:, M:], u, vb, r, cfg.n_rows, C, o)

        t_us = _graph_us(stream, call, nsets, max(2, 40 // nsets))
        flops = oracle.attn_flops(B, H, D, L, M)
        tf = flops / (t_us * 1e-6) / 1e12
        nbytes = 2 * (2 * B * L * H * D + 2 * B * (M + L) * H * D + cfg.n_rows * H * D)   # q, out, k, v, r
        gbs = nbytes / (t_us * 1e-6) / 1e9
        ai = flops / nbytes
        ridge = peak * 1e12 / (hbm * 1e9)
        bound = "hbm" if ai < ridge else "tensor"
        roof = ({"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                 "peak_source": "%s HBM copy" % kind} if bound == "hbm" else
                {"bound": "tensor", "achieved": tf, "peak": peak, "unit": "TFLOP/s", "frac": tf / peak,
                 "peak_source": "%s bf16 burst" % kind})
        roof.update({"algorithmic_flops_per_call": flops, "algorithmic_bytes_per_call": nbytes,
                     "arithmetic_intensity": ai, "ridge_flop_per_byte": ridge, "tensor_frac": tf / peak})
        res = {"workload": "%s: B%d H%d D%d d_model%d L%d M%d clamp%d bf16%s" % (
                   name, B, H, D, cfg.d_model, L, M, C, ", head stride %d" % hs if hs != D else ""),
               "path": "fused tcgen05 (attn_persist_kernel)" if path == 1 else "SIMT", "us_per_call": t_us,
               "tflops": tf, "tokens_per_s": B * L / (t_us * 1e-6), "roofline": roof,
               "l2": "%d rotating input sets" % nsets}
        if with_oracle:
            rows = [(0, h, i) for h in range(H) for i in range(0, L, max(1, L // (64 if name == "longmem" else 150)))]
            sec, fl, th = _oracle_sample(cfg, rows)
            res["cpu_baseline"] = {"value": fl / sec / 1e12, "unit": "TFLOP/s", "cores": th, "kind": "oracle",
                                   "sample": "%d of %d query rows of batch entry 0, fp64, %.1f s" % (len(rows), B * H * L, sec)}
        out[name] = res
        del sets, mems

    if "stream" not in legs:
        return out
    # the stream: 8 consecutive segments, each attending over the FIFO memory (empty at the start)
    # and then pushed into it; one pass = the position table + 8 x (attention + push)
    cfg = txl_inputs.CONFIGS["stream"]
    B, H, D, L, M, C, S = cfg.B, cfg.H, cfg.D, cfg.L, cfg.M, cfg.clamp_len, cfg.segments
    dt = cfg.torch_dtype
    g = torch.Generator(device=device).manual_seed(rank_seed(cfg.seed, rank))
    segs = [tuple(torch.randn(B, L, H, D, generator=g, device=device).to(dt) for _ in range(3)) for _ in range(S)]
    outs = [torch.empty(B, L, H, D, dtype=dt, device=device) for _ in range(S)]
    u = (0.02 * torch.randn(H, D, generator=g, device=device)).float()
    vb = (0.02 * torch.randn(H, D, generator=g, device=device)).float()
    W = (torch.randn(cfg.d_model, H * D, generator=g, device=device) * cfg.d_model ** -0.5).to(dt)
    r = torch.empty(cfg.n_rows, H, D, dtype=dt, device=device)
    ring = txl.Memory.empty(B, M, H, D, dtype=dt, device=device)
    path = txl.rel_attn_path(segs[0][0], ring, segs[0][1], segs[0][2], r, outs[0])

    def one_pass(_i):
        ring.restore(0, 0)
        txl.rel_pos_gen(W, r, cfg.n_rows, cfg.d_model, H, D)
        for s_ in range(S):
            q, k, v = segs[s_]
            txl.rel_attn_fwd(q, ring, k, v, u, vb, r, cfg.n_rows, C, outs[s_])
            txl.mem_push(ring, k, v)

    def attn_only(_i):
        ring.restore(0, 0)
        for s_ in range(S):
            q, k, v = segs[s_]
            txl.rel_attn_fwd(q, ring, k, v, u, vb, r, cfg.n_rows, C, outs[s_])
            ring.restore((ring.wp + L) % M, min(ring.valid + L, M))    # the push's state, no copy

    t_pass = _graph_us(stream, one_pass, 1, 10)
    t_attn = _graph_us(stream, attn_only, 1, 10)
    flops = sum(oracle.attn_flops(B, H, D, L, M, min(s_ * L, M)) for s_ in range(S))
    pos_flops = 2 * cfg.n_rows * cfg.d_model * H * D
    tf = flops / (t_attn * 1e-6) / 1e12
    res = {"workload": "stream: B%d H%d D%d d_model%d L%d M%d clamp%d bf16, %d segments through the FIFO memory "
                       "(empty at the start)" % (B, H, D, cfg.d_model, L, M, C, S),
           "path": "fused tcgen05 (attn_tc_kernel<2>)" if path == 1 else "SIMT",
           "us_per_pass": t_pass, "us_attention_per_segment": t_attn / S,
           "tflops": tf, "tflops_pass": (flops + pos_flops) / (t_pass * 1e-6) / 1e12,
           "tokens_per_s": S * B * L / (t_pass * 1e-6),
           "roofline": {"bound": "tensor", "achieved": tf, "peak": peak, "unit": "TFLOP/s", "frac": tf / peak,
                        "peak_source": "%s bf16 burst" % kind, "algorithmic_flops_per_pass": flops},
           "gpu_launches_per_pass": 1 + 2 * S}
    if with_oracle:
        T = S * L
        rows = [(0, h, t) for h in (0, 7) for t in range(L - 1, T, L // 4)]
        sec, fl, th = _oracle_sample(cfg, rows, stream=True)
        res["cpu_baseline"] = {"value": fl / sec / 1e12, "unit": "TFLOP/s", "cores": th, "kind": "oracle",
                               "sample": "%d of %d query rows (batch entry 0, heads 0 and 7, every segment), fp64, %.1f s"
                                         % (len(rows), B * H * T, sec)}
    out["stream"] = res
    return out


def bench_decode(txl, device, stream, rank, args):
    """One new token per (b, h) over a long memory (txl_rel_attn_decode): B8 H16 D64 L1 M4096,
    clamp 1000, bf16, the K/V cache head-major ([B][H][T][D]: each (b, h) stream contiguous).
    HBM-bound: reported as algorithmic bytes (K and V of every key, the r rows, q and out) per
    call over the call time, against the measured HBM copy bandwidth.  Two input sets of 134 MB
    alternate so no call reads L2-warm K/V."""
    import torch
    B, H, D, L, M, C, dm = 8, 16, 64, 1, 4096, 1000, 1024
    dt = torch.bfloat16
    g = torch.Generator(device=device).manual_seed(rank_seed(4242, rank))
    n_rows = min(M + L, C + 1)
    W = (torch.randn(dm, H * D, generator=g, device=device) * dm ** -0.5).to(dt)
    r = torch.empty(n_rows, H, D, dtype=dt, device=device)
    txl.rel_pos_gen(W, r, n_rows, dm, H, D)
    u = (0.02 * torch.randn(H, D, generator=g, device=device)).float()
    vb = (0.02 * torch.randn(H, D, generator=g, device=device)).float()
    sets = []
    for _ in range(2):
        # head-major cache [B][H][M + L][D] (each (b, h) key stream contiguous), viewed [B][T][H][D]
        kv = torch.randn(2, B, H, M + L, D, generator=g, device=device).to(dt).permute(0, 1, 3, 2, 4)
        q = torch.randn(B, L, H, D, generator=g, device=device).to(dt)
        mem = txl.Memory(kv[0, :, :M], kv[1, :, :M], 0, M)
        sets.append((q, kv, mem, torch.empty(B, L, H, D, dtype=dt, device=device)))
    ws = torch.empty(txl.rel_attn_decode_workspace_size(sets[0][0], sets[0][2]), dtype=torch.uint8,
                     device=device)

    def call(s_):
        q, kv, mem, out = sets[s_]
        txl.rel_attn_decode(q, mem, kv[0, :, M:], kv[1, :, M:], u, vb, r, n_rows, C, out, workspace=ws)

    with torch.cuda.stream(stream):
        for i in range(4):
            call(i & 1)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        call(0)
        call(1)
    reps = 50
    with torch.cuda.stream(stream):
        graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            graph.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    t_us = e0.elapsed_time(e1) * 1e3 / (2 * reps)
    nbytes = (2 * B * H * (M + L) * D + H * n_rows * D + 2 * B * H * L * D) * 2
    _, _, hbm, kind = _peaks()
    gbs = nbytes / (t_us * 1e-6) / 1e9
    return {"workload": "decode: B8 H16 D64 L1 M4096 clamp1000 bf16, head-major K/V cache (one new token per (b, h))",
            "us_per_call": t_us, "tokens_per_s": B * L / (t_us * 1e-6),
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                         "frac": gbs / hbm, "peak_source": "%s HBM copy" % kind,
                         "algorithmic_bytes_per_call": nbytes},
            "gpu_launches_per_call": 2}


def bench_layer(txl, device, stream, rank, args):
    """The attention-layer step over hidden states on the large workload, as
    txl_rel_attn_layer_fused runs it: the q|k|v projection of the segment (6144 x 3072 x 1024)
    writing K and V straight into the memory ring, the fused attention over [memory ++ segment]
    read from the ring, the output projection (6144 x 1024 x 1024), plus the position table, per
    step (the unfused step, with its separate push, is timed beside it).  Eight hidden-state sets (100 MB) rotate with the 25 MB K/V ring,
    the 50 MB workspace and 8 MB of weights, so a step does not find its inputs L2-warm.  The
    q|k|v product is also timed alone (same rotation) against the measured bf16 peak."""
    import torch
    B, H, D, L, M, C, dm = 16, 16, 64, 384, 384, 1000, 1024
    HD = H * D
    dt = torch.bfloat16
    g = torch.Generator(device=device).manual_seed(rank_seed(777, rank))
    n_rows = min(M + L, C + 1)
    W_R = (torch.randn(dm, HD, generator=g, device=device) * dm ** -0.5).to(dt)
    W_qkv = (torch.randn(dm, 3 * HD, generator=g, device=device) * dm ** -0.5).to(dt)
    W_o = (torch.randn(HD, dm, generator=g, device=device) * HD ** -0.5).to(dt)
    u = (0.02 * torch.randn(H, D, generator=g, device=device)).float()
    vb = (0.02 * torch.randn(H, D, generator=g, device=device)).float()
    r = torch.empty(n_rows, H, D, dtype=dt, device=device)
    nsets = 8
    hs = [torch.randn(B, L, dm, generator=g, device=device).to(dt) for _ in range(nsets)]
    ys = [torch.empty(B, L, dm, dtype=dt, device=device) for _ in range(2)]
    mem = txl.Memory.empty(B, M, H, D, device=device)
    ring = txl.Memory.empty(B, M + L, H, D, device=device)       # memory of M positions + the segment
    ws = torch.empty(txl.rel_attn_layer_workspace_size(B, L, H, D), dtype=torch.uint8, device=device)
    qkv = ws[: B * L * 3 * HD * 2].view(dt).view(B * L, 3 * HD)

    def step(i):
        txl.rel_pos_gen(W_R, r, n_rows, dm, H, D)
        txl.rel_attn_layer_fused(hs[i], ring, M, W_qkv, W_o, u, vb, r, n_rows, C, H, D, ys[i & 1], workspace=ws)

    def step_unfused(i):
        txl.rel_pos_gen(W_R, r, n_rows, dm, H, D)
        txl.rel_attn_layer(hs[i], mem, W_qkv, W_o, u, vb, r, n_rows, C, H, D, ys[i & 1], workspace=ws)

    def proj(i):
        txl.linear(hs[i].view(B * L, dm), W_qkv, qkv)

    def timed(fn, reps=10):
        with torch.cuda.stream(stream):
            for i in range(2 * nsets):
                fn(i % nsets)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for i in range(nsets):
                fn(i)
        with torch.cuda.stream(stream):
            graph.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(reps):
                graph.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / (nsets * reps)

    t_step = timed(step)
    t_unfused = timed(step_unfused)
    t_proj = timed(proj)
    # every position of the memory is valid once the warm-up has pushed two segments
    attn = 6 * D * B * H * (L * M + L * (L + 1) // 2)
    flops = 2 * B * L * dm * 4 * HD + attn + 2 * n_rows * dm * HD
    pflops = 2.0 * B * L * dm * 3 * HD
    peak, _, _, kind = _peaks()
    achieved = pflops / (t_proj * 1e-6) / 1e12
    return {"workload": "layer: B16 L384 M384 H16 D64 d_model1024 clamp1000 bf16 (hidden states in, y out)",
            "us_per_step": t_step, "tflops": flops / (t_step * 1e-6) / 1e12,
            "algorithmic_flops_per_step": flops, "gpu_launches_per_step": 4,
            "step": "txl_rel_attn_layer_fused: position table, q|k|v product writing K and V into the ring "
                    "(no push), attention from the ring, output product",
            "us_per_step_unfused": t_unfused, "gpu_launches_per_step_unfused": 5,
            "roofline": {"kernel": "txl_linear (linear_kernel, q|k|v 6144x3072x1024)", "bound": "tensor",
                         "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                         "peak_source": "%s bf16 burst" % kind, "us_per_launch": t_proj,
                         "algorithmic_flops_per_launch": pflops}}


def bwd_flops(B, H, D, L, M, n_rows, d_model):
    """Algorithmic flops of the backward of one call: per visible (query, key) pair the two score
    terms (4 D), dP (2 D), dq (4 D) and dr (2 D); per pair with a current-segment key also dk and
    dv (4 D; the memory is stop-gradient); and dW_R = R^T dr (2 n_rows d_model H D)."""
    pairs = B * H * (L * M + L * (L + 1) // 2)
    pairs_cur = B * H * (L * (L + 1) // 2)
    return 12 * D * pairs + 4 * D * pairs_cur, 2 * n_rows * d_model * H * D


def bench_backward(txl, device, stream, rank, args):
    """Gradients of one fused-attention call on the large workload.  The forward is run once,
    untimed, with its softmax statistics saved (txl_rel_attn_fwd_lse, as a training step's forward
    keeps them); then timed: txl_rel_attn_bwd_lse (the row dot products dO . out, then the tcgen05
    gradient kernel: bf16 operands, fp32 TMEM accumulators and gradients; the bias reduction) and the
    position table's txl_rel_pos_bwd, together and each alone; and, for comparison, txl_rel_attn_bwd
    without the saved statistics (it first retakes them with the fused forward kernel's statistics
    pass).  The attention backward is reported against the measured bf16 tensor peak."""
    import torch
    B, H, D, L, M, C, dm = 16, 16, 64, 384, 384, 1000, 1024
    dt = torch.bfloat16
    g = torch.Generator(device=device).manual_seed(rank_seed(31337, rank))
    n_rows = min(M + L, C + 1)
    W = (torch.randn(dm, H * D, generator=g, device=device) * dm ** -0.5).to(dt)
    r = torch.empty(n_rows, H, D, dtype=dt, device=device)
    txl.rel_pos_gen(W, r, n_rows, dm, H, D)
    u = (0.02 * torch.randn(H, D, generator=g, device=device)).float()
    vb = (0.02 * torch.randn(H, D, generator=g, device=device)).float()
    q = torch.randn(B, L, H, D, generator=g, device=device).to(dt)
    k = torch.randn(B, M + L, H, D, generator=g, device=device).to(dt)
    v = torch.randn(B, M + L, H, D, generator=g, device=device).to(dt)
    dO = torch.randn(B, L, H, D, generator=g, device=device).to(dt)
    out = torch.empty(B, L, H, D, dtype=dt, device=device)
    lse = torch.empty(B, L, H, dtype=torch.float32, device=device)
    mem = txl.Memory(k[:, :M], v[:, :M], 0, M)
    txl.rel_attn_fwd(q, mem, k[:, M:], v[:, M:], u, vb, r, n_rows, C, out, lse=lse)
    ws = torch.empty(16 * 1024 * 1024 * 8, dtype=torch.uint8, device=device)
    res = {}

    def attn():
        res["g"] = txl.rel_attn_bwd(q, mem, k[:, M:], v[:, M:], u, vb, r, n_rows, C, out, dO, workspace=ws, lse=lse)

    def attn_recompute():
        txl.rel_attn_bwd(q, mem, k[:, M:], v[:, M:], u, vb, r, n_rows, C, out, dO, workspace=ws)

    def pos():
        res["dW"] = txl.rel_pos_bwd(res["g"]["dr"], dm)

    def both():
        attn()
        pos()

    def timed(fn, reps=5):
        with torch.cuda.stream(stream):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(reps):
                fn()
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / reps

    t_us = timed(both)
    t_attn = timed(attn)
    t_pos = timed(pos)
    t_attn_rec = timed(attn_recompute)
    f_attn, f_pos = bwd_flops(B, H, D, L, M, n_rows, dm)
    bf16_peak, _, _, peak_src = _peaks()
    achieved = f_attn / (t_attn * 1e-6) / 1e12
    return {"workload": "backward: B16 H16 D64 d_model1024 L384 M384 clamp1000, bf16 inputs, fp32 gradients",
            "us_per_call": t_us, "us_attn_bwd": t_attn, "us_pos_bwd": t_pos,
            "us_attn_bwd_without_saved_lse": t_attn_rec,
            "algorithmic_flops_per_call": f_attn + f_pos, "tflops": (f_attn + f_pos) / (t_us * 1e-6) / 1e12,
            "roofline": {"kernel": "txl_rel_attn_bwd_lse (bwd_rowdot_kernel + bwd_umma_kernel, tcgen05 with TMEM accumulators)",
                         "traffic": _profile_traffic(os.path.join(ROOT, "transformer_xl_relative_gb300", "csrc",
                                                                  "txl_bwd_umma.cu"), "bwd_umma_kernel_large.json"),
                         "traffic_kernel": "bwd_umma_kernel (ncu, bytes per launch)",
                         "bound": "tensor", "achieved": achieved, "peak": bf16_peak, "unit": "TFLOP/s",
                         "frac": achieved / bf16_peak, "algorithmic_flops_per_launch": f_attn,
                         "peak_source": peak_src + " bf16 burst"}}


def bench_table(txl, device, stream, rank, args):
    """The learned-table variant (txl_rel_attn_table_fwd): bidirectional attention B16 L384 H16 D64,
    max_len 512, bf16 inputs, every key visible; on this workload the persistent tcgen05 kernel in its
    learned-table mode (bf16 products, fp32 accumulation in tensor memory).  Algorithmic flops 6 D per (query, key) pair (content 2 D,
    position 2 D, P.V 2 D) against the measured bf16 tensor peak."""
    import torch
    B, H, D, L, max_len = 16, 16, 64, 384, 512
    dt = torch.bfloat16
    g = torch.Generator(device=device).manual_seed(rank_seed(555, rank))
    q, k, v = (torch.randn(B, L, H, D, generator=g, device=device).to(dt) for _ in range(3))
    u = (0.02 * torch.randn(H, D, generator=g, device=device)).float()
    vb = (0.02 * torch.randn(H, D, generator=g, device=device)).float()
    rt = torch.randn(2 * max_len - 1, H, D, generator=g, device=device).to(dt)
    out = torch.empty(B, L, H, D, dtype=dt, device=device)

    def call():
        txl.rel_attn_table_fwd(q, k, v, u, vb, rt, max_len, out)

    with torch.cuda.stream(stream):
        for _ in range(3):
            call()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        call()
    reps = 20
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        graph.replay()
        e0.record(stream)
        for _ in range(reps):
            graph.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    t_us = e0.elapsed_time(e1) * 1e3 / reps
    flops = 6 * D * B * H * L * L
    bf16_peak, _, _, peak_src = _peaks()
    achieved = flops / (t_us * 1e-6) / 1e12
    return {"workload": "table variant: B16 L384 H16 D64 max_len512 bf16, bidirectional, no mask",
            "us_per_call": t_us, "algorithmic_flops_per_call": flops,
            "roofline": {"kernel": "txl_rel_attn_table_fwd (attn_persist_kernel, learned-table mode)", "bound": "tensor",
                         "achieved": achieved, "peak": bf16_peak, "unit": "TFLOP/s", "frac": achieved / bf16_peak,
                         "peak_source": peak_src + " bf16 burst"}}


def run_txl(args):
    import torch

    world, rank, local = _dist()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    device = torch.device("cuda", torch.cuda.current_device())
    import transformer_xl_relative_gb300 as txl
    import txl_inputs

    cfg = txl_inputs.CONFIGS[WORKLOAD]
    B, H, D, L, M, C = cfg.B, cfg.H, cfg.D, cfg.L, cfg.M, cfg.clamp_len
    dt = cfg.torch_dtype
    n_rows = cfg.n_rows
    NSETS = 4
    g = torch.Generator(device=device).manual_seed(rank_seed(cfg.seed, rank))
    sets = []
    for _ in range(NSETS):
        q = torch.randn(B, L, H, D, generator=g, device=device).to(dt)
        k = torch.randn(B, M + L, H, D, generator=g, device=device).to(dt)
        v = torch.randn(B, M + L, H, D, generator=g, device=device).to(dt)
        sets.append((q, k, v))
    u = (0.02 * torch.randn(H, D, generator=g, device=device)).float()
    vb = (0.02 * torch.randn(H, D, generator=g, device=device)).float()
    W = (torch.randn(cfg.d_model, H * D, generator=g, device=device) * cfg.d_model ** -0.5).to(dt)
    r = torch.empty(n_rows, H, D, dtype=dt, device=device)
    outs = [torch.empty(B, L, H, D, dtype=dt, device=device) for _ in range(NSETS)]
    ring = txl.Memory.empty(B, M, H, D, dtype=dt, device=device)
    mems = [txl.Memory.full(k[:, :M], v[:, :M]) for (_, k, v) in sets]

    def step(s):
        q, k, v = sets[s]
        txl.rel_pos_gen(W, r, n_rows, cfg.d_model, H, D)
        txl.rel_attn_fwd(q, mems[s], k[:, M:], v[:, M:], u, vb, r, n_rows, C, outs[s])
        txl.mem_push(ring, k[:, M:], v[:, M:])

    assert txl.rel_attn_path(sets[0][0], mems[0], sets[0][1][:, M:], sets[0][2][:, M:], r, outs[0]) == 1
    stream = torch.cuda.Stream(device=device)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for s in range(NSETS):           # warm-up outside capture (first-call attribute setup)
            step(s)
    torch.cuda.synchronize()
    # One CUDA graph per input set, each holding one whole step.  A step's position table does not
    # depend on the previous step's memory push, so each step's graph also computes the next
    # step's table on a side stream (into the other of two table buffers) while its own push
    # runs; every step still runs all three kernels.  Exactly W warm-up and K timed steps replay
    # the graphs in rotation.
    r_bufs = [r, torch.empty_like(r)]
    side = torch.cuda.Stream(device=device)

    def step_overlapped(s):
        q, k, v = sets[s]
        txl.rel_attn_fwd(q, mems[s], k[:, M:], v[:, M:], u, vb, r_bufs[s % 2], n_rows, C, outs[s])
        e_attn = torch.cuda.Event()
        e_attn.record(stream)
        side.wait_event(e_attn)
        with torch.cuda.stream(side):
            txl.rel_pos_gen(W, r_bufs[(s + 1) % 2], n_rows, cfg.d_model, H, D)
        e_pos = torch.cuda.Event()
        e_pos.record(side)
        txl.mem_push(ring, k[:, M:], v[:, M:])
        stream.wait_event(e_pos)

    with torch.cuda.stream(stream):
        txl.rel_pos_gen(W, r_bufs[0], n_rows, cfg.d_model, H, D)
        for s in range(NSETS):
            step_overlapped(s)
    torch.cuda.synchronize()
    graphs = []
    for s in range(NSETS):
        g_ = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_, stream=stream):
            step_overlapped(s)
        graphs.append(g_)
    attn_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(attn_graph, stream=stream):
        for s in range(NSETS):
            q, k, v = sets[s]
            txl.rel_attn_fwd(q, mems[s], k[:, M:], v[:, M:], u, vb, r, n_rows, C, outs[s])
    pos_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(pos_graph, stream=stream):
        for s in range(NSETS):
            txl.rel_pos_gen(W, r, n_rows, cfg.d_model, H, D)
    push_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(push_graph, stream=stream):
        for s in range(NSETS):
            txl.mem_push(ring, sets[s][1][:, M:], sets[s][2][:, M:])

    steps = max(1, args.steps)
    reps = max(1, math.ceil(steps / NSETS))
    sampler = ClockSampler(device.index if device.index is not None else 0)
    sampler.start()
    time.sleep(0.3)
    with torch.cuda.stream(stream):
        txl.rel_pos_gen(W, r_bufs[0], n_rows, cfg.d_model, H, D)
        for i in range(args.warmup):
            graphs[i % NSETS].replay()
    torch.cuda.synchronize()
    _barrier(world)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for i in range(steps):
            graphs[(args.warmup + i) % NSETS].replay()
        ev1.record(stream)
    torch.cuda.synchronize()
    _barrier(world)
    torch.cuda.synchronize()
    wall1 = time.time()
    t_step_ms = ev0.elapsed_time(ev1) / steps
    t_step_ms = _max_over_ranks(t_step_ms, world, device)

    # the fused attention kernel alone, same rotation, same stream
    with torch.cuda.stream(stream):
        attn_graph.replay()
    torch.cuda.synchronize()
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        a0.record(stream)
        for _ in range(reps):
            attn_graph.replay()
        a1.record(stream)
    torch.cuda.synchronize()
    t_attn_ms = a0.elapsed_time(a1) / (reps * NSETS)

    def graph_ms(g, reps_):
        with torch.cuda.stream(stream):
            g.replay()
        torch.cuda.synchronize()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            g0.record(stream)
            for _ in range(reps_):
                g.replay()
            g1.record(stream)
        torch.cuda.synchronize()
        return g0.elapsed_time(g1) / (reps_ * NSETS)

    t_pos_ms = graph_ms(pos_graph, max(1, reps // 4))
    t_push_ms = graph_ms(push_graph, max(1, reps // 4))
    sampler.stop()
    clocks = sampler.summary(wall0, wall1)

    # end to end through the public API, as a stream of segments: every step copies the new
    # segment's q, k, v [B, L, H, D] from pinned host memory, attends over the device-resident K/V
    # memory (the ring the previous steps pushed), pushes the segment, and copies the output back.
    # Copies run on their own streams, double-buffered, so step i+1's inputs move while step i
    # computes; the timed region spans every copy and kernel of the e2e_steps steps.
    e2e_steps = max(8, min(steps, 40))
    hq = [sets[i][0].cpu().pin_memory() for i in range(2)]
    hk = [sets[i][1][:, M:].cpu().pin_memory() for i in range(2)]
    hv = [sets[i][2][:, M:].cpu().pin_memory() for i in range(2)]
    ho = [torch.empty(B, L, H, D, dtype=dt).pin_memory() for _ in range(2)]
    dqb = [torch.empty(B, L, H, D, dtype=dt, device=device) for _ in range(2)]
    dkb = [torch.empty(B, L, H, D, dtype=dt, device=device) for _ in range(2)]
    dvb = [torch.empty(B, L, H, D, dtype=dt, device=device) for _ in range(2)]
    dob = [torch.empty(B, L, H, D, dtype=dt, device=device) for _ in range(2)]
    # one input stream per tensor so the three copies can use separate copy engines
    s_ins = [torch.cuda.Stream(device=device) for _ in range(3)]
    s_out = torch.cuda.Stream(device=device)
    e_in = [[torch.cuda.Event() for _ in range(3)] for _ in range(2)]   # inputs of buffer slot landed
    e_done = [torch.cuda.Event() for _ in range(2)]     # compute finished with the slot's inputs
    e_out = [torch.cuda.Event() for _ in range(2)]      # output of the slot copied back
    stream_ring = txl.Memory.empty(B, M, H, D, dtype=dt, device=device)

    def e2e_run(n):
        for i in range(n):
            sl = i % 2
            for c, (dst, src) in enumerate(((dqb[sl], hq[i % 2]), (dkb[sl], hk[i % 2]), (dvb[sl], hv[i % 2]))):
                with torch.cuda.stream(s_ins[c]):
                    if i >= 2:
                        s_ins[c].wait_event(e_done[sl])     # the slot's previous inputs are consumed
                    dst.copy_(src, non_blocking=True)
                    e_in[sl][c].record(s_ins[c])
            with torch.cuda.stream(stream):
                for c in range(3):
                    stream.wait_event(e_in[sl][c])
                if i >= 2:
                    stream.wait_event(e_out[sl])            # the slot's previous output is copied out
                txl.rel_pos_gen(W, r, n_rows, cfg.d_model, H, D)
                txl.rel_attn_fwd(dqb[sl], stream_ring, dkb[sl], dvb[sl], u, vb, r, n_rows, C, dob[sl])
                txl.mem_push(stream_ring, dkb[sl], dvb[sl])
                e_done[sl].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(e_done[sl])
                ho[sl].copy_(dob[sl], non_blocking=True)
                e_out[sl].record(s_out)

    e2e_run(4)                                          # warm-up; the memory is full from here on
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for si in s_ins:
        si.wait_event(e0)
    e2e_run(e2e_steps)
    s_done = torch.cuda.Event()
    s_done.record(s_out)
    stream.wait_event(s_done)
    e1.record(stream)
    torch.cuda.synchronize()
    t_e2e_ms = _max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world, device)
    h2d = 3 * B * L * H * D * 2
    d2h = B * L * H * D * 2

    decode = bench_decode(txl, device, stream, rank, args)
    layer = bench_layer(txl, device, stream, rank, args)
    backward = bench_backward(txl, device, stream, rank, args)
    table = bench_table(txl, device, stream, rank, args)
    configs = bench_configs(txl, device, stream, rank, args,
                            with_oracle=rank == 0 and world == 1 and not args.no_cpu_baseline)

    attn_flops, pos_flops = _flops(cfg)
    step_flops = attn_flops + pos_flops
    peak, peak_sust, _, peak_kind = _peaks()
    value = aggregate_value(world, step_flops, t_step_ms)
    achieved = attn_flops / (t_attn_ms * 1e-3) / 1e12
    kernel_src = os.path.join(ROOT, "transformer_xl_relative_gb300", "csrc", "txl_attn_persist.cu")
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": steps,
        "warmup": args.warmup,
        "ms_per_step": t_step_ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) q/k/v, N(0,0.02^2) u/v_bias, N(0,1/d_model) W_R)",
        "config": {"workload": WORKLOAD_NAME,
                   "global_batch": B * world, "seq_len": L, "mem_len": M,
                   "l2": "4 rotating input sets, 252 MB > 129 MB L2",
                   "parallelism": "dp%d: independent replicas, no collective on the data path" % world},
        "tokens_per_s": world * B * L / (t_step_ms * 1e-3),
        "attn_tflops": achieved,
        "kernel_us": {"rel_attn_fwd": 1e3 * t_attn_ms, "rel_pos_gen": 1e3 * t_pos_ms,
                      "mem_push": 1e3 * t_push_ms},
        "frac_of_bf16_peak_step": value / world / peak,
        "clocks": clocks,
        "e2e": {"value": world * step_flops / (t_e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": t_e2e_ms},
        "gpu_launches": 3 * steps,
        "decode": decode,
        "layer": layer,
        "backward": backward,
        "table": table,
        "configs": configs,
        "roofline": {"kernel": "txl_rel_attn_fwd (attn_persist_kernel)", "bound": "tensor",
                     "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "peak_source": "%s bf16 burst (MEASURED_PEAKS.json)" % peak_kind
                     if peak_kind == "measured" else "fallback 1.9 PFLOP/s",
                     "traffic": _profile_traffic(kernel_src),
                     "algorithmic_flops_per_launch": attn_flops},
    }
    # nominal GB300 figures (dense bf16 tensor rate; HBM3e bandwidth), beside the measured peaks
    line["nominal_peaks"] = {"bf16_dense_tflops": NOMINAL_BF16_TFLOPS, "hbm_gbs": NOMINAL_HBM_GBS,
                             "attn_frac_of_nominal_bf16": achieved / NOMINAL_BF16_TFLOPS,
                             "source": "NVIDIA GB300 nominal dense bf16 rate and HBM3e bandwidth"}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg)
        line["cpu_baseline"]["single_thread"] = cpu_baseline(cfg, target_s=1.0, threads=1)
        for key, base in row_baselines().items():
            line[key]["cpu_baseline"] = base
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def profile_leg(args):
    """A few calls of one workload's kernels and nothing else, for a profiler to capture:
    large / base / longmem (the fused attention), stream (8 segments: attention + push), layer (the
    fused layer step), decode, table (the learned-table variant), backward.  Prints the per-call device time of the last repetition."""
    import torch
    import transformer_xl_relative_gb300 as txl
    device = torch.device("cuda", 0)
    stream = torch.cuda.Stream(device=device)
    if args.profile_leg in ("base", "longmem", "stream"):
        res = bench_configs(txl, device, stream, 0, args, with_oracle=False, legs=(args.profile_leg,))[args.profile_leg]
    elif args.profile_leg == "layer":
        res = bench_layer(txl, device, stream, 0, args)
    elif args.profile_leg == "decode":
        res = bench_decode(txl, device, stream, 0, args)
    elif args.profile_leg == "table":
        res = bench_table(txl, device, stream, 0, args)
    elif args.profile_leg == "backward":
        res = bench_backward(txl, device, stream, 0, args)
    else:
        import txl_inputs
        cfg = txl_inputs.CONFIGS["large"]
        B, H, D, L, M, C = cfg.B, cfg.H, cfg.D, cfg.L, cfg.M, cfg.clamp_len
        g = torch.Generator(device=device).manual_seed(cfg.seed)
        q = torch.randn(B, L, H, D, generator=g, device=device).to(torch.bfloat16)
        k = torch.randn(B, M + L, H, D, generator=g, device=device).to(torch.bfloat16)
        v = torch.randn(B, M + L, H, D, generator=g, device=device).to(torch.bfloat16)
        u = (0.02 * torch.randn(H, D, generator=g, device=device)).float()
        vb = (0.02 * torch.randn(H, D, generator=g, device=device)).float()
        W = (torch.randn(cfg.d_model, H * D, generator=g, device=device) * cfg.d_model ** -0.5).to(torch.bfloat16)
        r = torch.empty(cfg.n_rows, H, D, dtype=torch.bfloat16, device=device)
        out = torch.empty_like(q)
        mem = txl.Memory.full(k[:, :M], v[:, :M])
        txl.rel_pos_gen(W, r, cfg.n_rows, cfg.d_model, H, D)
        res = {"us_per_call": _graph_us(stream, lambda i: txl.rel_attn_fwd(q, mem, k[:, M:], v[:, M:], u, vb, r,
                                                                         cfg.n_rows, C, out), 1, 3)}
    print(json.dumps({"profile_leg": args.profile_leg,
                      **{k_: v_ for k_, v_ in res.items() if isinstance(v_, (int, float, str))}}), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=40)
    ap.add_argument("--impl", choices=["txl", "reference"], default="txl")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-leg", choices=["large", "base", "longmem", "stream", "layer", "decode", "table",
                                              "backward"],
                    help="run only a few calls of this workload (for a profiler) and exit")
    args = ap.parse_args(argv)
    world = os.environ.get("WORLD_SIZE")
    if args.gpus > 1 and world is None:
        # one process per GPU: relaunch this command under torch.distributed.run
        cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", str(args.gpus),
               "--master-addr", "127.0.0.1", "--master-port", os.environ.get("MASTER_PORT", "29517"),
               os.path.abspath(__file__), *(argv if argv is not None else sys.argv[1:])]
        return subprocess.call(cmd)
    if world is not None and int(world) != args.gpus:
        sys.stderr.write("bench.py: --gpus %d but WORLD_SIZE=%s\n" % (args.gpus, world))
        return 2
    if args.impl == "reference":
        return run_reference(args)
    if args.profile_leg:
        return profile_leg(args)
    return run_txl(args)


if __name__ == "__main__":
    sys.exit(main())
