"""Seeded synthetic inputs for Transformer-XL relative attention.

This module only draws random numbers and lays them out; it holds none of the method's
arithmetic, and both the CUDA path and the fp64 oracle consume what it produces.

Distributions (the pages give no dataset for this path; these stand in for one):
  q, k, v  ~ N(0, 1)                     (projected activations)
  u, v_bias ~ N(0, 0.02^2)               ("TransformerXL 相对位置编码" §3.1 and §4.5: randn * 0.02)
  W_R      ~ N(0, 1/d_model) (variance)  (reading of "N(0, 1/d_model)": std d_model^-1/2)
  layer    : hidden states h ~ N(0, 1); W_q, W_k, W_v ~ N(0, 1/d_model) and W_o ~ N(0, 1/(H*D))
             (variance), so q, k, v and y come out with unit variance like the inputs above
Values are drawn on the CPU with ``torch.Generator().manual_seed(seed)`` in fp32 and then cast
to the compute dtype, so every consumer sees identical bits.
"""
from __future__ import annotations

import dataclasses

import torch


@dataclasses.dataclass(frozen=True)
class Config:
    name: str
    B: int
    H: int
    D: int
    d_model: int
    L: int
    M: int
    clamp_len: int
    dtype: str               # "f32" or "bf16"
    seed: int
    segments: int = 1        # >1: streaming through the FIFO memory
    head_stride: int = 0     # elements between heads in q/k/v/out (0: D, dense)
    ld_w: int = 0            # W_R row stride (0: H*D rounded up to a multiple of 8)

    @property
    def hs(self) -> int:
        return self.head_stride or self.D

    @property
    def ldw(self) -> int:
        return self.ld_w or (self.H * self.D + 7) // 8 * 8

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def n_rows(self) -> int:
        """Rows of the relative table r: distances 0..min(M+L-1, clamp_len)."""
        return min(self.M + self.L, self.clamp_len + 1)


# The five workloads.  The base shape has d_head = 41: its head stride is padded to 48 and the
# W_R row stride to 416 so that every row starts on a 16-byte boundary.
CONFIGS = {
    "tiny": Config("tiny", B=1, H=2, D=8, d_model=16, L=8, M=8, clamp_len=16, dtype="f32", seed=1000),
    "base": Config("base", B=32, H=10, D=41, d_model=410, L=150, M=150, clamp_len=1000, dtype="bf16",
                   seed=1001, head_stride=48, ld_w=416),
    "large": Config("large", B=16, H=16, D=64, d_model=1024, L=384, M=384, clamp_len=1000,
                    dtype="bf16", seed=1002),
    "longmem": Config("longmem", B=8, H=16, D=64, d_model=1024, L=128, M=1600, clamp_len=1000,
                      dtype="bf16", seed=1003),
    "stream": Config("stream", B=4, H=16, D=128, d_model=2048, L=512, M=2048, clamp_len=1000,
                     dtype="bf16", seed=1004, segments=8),
}


def _randn(gen: torch.Generator, shape, std: float = 1.0) -> torch.Tensor:
    return torch.randn(*shape, generator=gen, dtype=torch.float32) * std


def _padded(x: torch.Tensor, head_stride: int, dtype) -> torch.Tensor:
    """Place x [..., D] into zero storage [..., head_stride] and return the [..., :D] view."""
    D = x.shape[-1]
    if head_stride == D:
        return x.to(dtype).contiguous()
    store = torch.zeros(*x.shape[:-1], head_stride, dtype=dtype)
    store[..., :D] = x.to(dtype)
    return store[..., :D]


def make_params(cfg: Config, seed: int | None = None):
    """u, v_bias [H, D] fp32 and W_R [d_model, ldw] (first H*D columns used) in the compute dtype."""
    gen = torch.Generator().manual_seed(cfg.seed if seed is None else seed)
    u = _randn(gen, (cfg.H, cfg.D), 0.02)
    vb = _randn(gen, (cfg.H, cfg.D), 0.02)
    w = _randn(gen, (cfg.d_model, cfg.H * cfg.D), cfg.d_model ** -0.5)
    W = torch.zeros(cfg.d_model, cfg.ldw, dtype=cfg.torch_dtype)
    W[:, : cfg.H * cfg.D] = w.to(cfg.torch_dtype)
    return u, vb, W


def make_qkv(cfg: Config, seed: int, L: int | None = None, T: int | None = None):
    """q [B, L, H, D] and k, v [B, T, H, D] (views into head-stride-padded storage)."""
    L = cfg.L if L is None else L
    T = cfg.M + cfg.L if T is None else T
    gen = torch.Generator().manual_seed(seed)
    q = _randn(gen, (cfg.B, L, cfg.H, cfg.D))
    k = _randn(gen, (cfg.B, T, cfg.H, cfg.D))
    v = _randn(gen, (cfg.B, T, cfg.H, cfg.D))
    dt = cfg.torch_dtype
    return _padded(q, cfg.hs, dt), _padded(k, cfg.hs, dt), _padded(v, cfg.hs, dt)


def make_case(cfg: Config):
    """One call's inputs: q, k, v ([memory ++ current] keys/values), u, v_bias, W_R."""
    u, vb, W = make_params(cfg, cfg.seed + 10_000)
    q, k, v = make_qkv(cfg, cfg.seed)
    return dict(q=q, k=k, v=v, u=u, vb=vb, W_R=W)


def segment_seed(cfg: Config, s: int) -> int:
    return cfg.seed + 1 + 100 * s


def make_segment(cfg: Config, s: int):
    """Segment s of a stream: q, k, v [B, L, H, D]."""
    return make_qkv(cfg, segment_seed(cfg, s), L=cfg.L, T=cfg.L)


def custom(name="custom", B=1, H=2, D=16, d_model=32, L=16, M=16, clamp_len=1000, dtype="bf16",
           seed=7, segments=1, head_stride=0, ld_w=0) -> Config:
    return Config(name, B, H, D, d_model, L, M, clamp_len, dtype, seed, segments, head_stride, ld_w)


def make_layer(cfg: Config, segments: int = 1, seed: int | None = None):
    """Inputs of the attention-layer step: hidden states h [B, segments*L, d_model] and the
    weights W_qkv [d_model, 3*H*D] (columns W_q | W_k | W_v) and W_o [H*D, d_model], in the
    compute dtype, plus u, v_bias and W_R as make_params draws them."""
    gen = torch.Generator().manual_seed(cfg.seed + 20_000 if seed is None else seed)
    HD = cfg.H * cfg.D
    h = _randn(gen, (cfg.B, segments * cfg.L, cfg.d_model))
    W_qkv = _randn(gen, (cfg.d_model, 3 * HD), cfg.d_model ** -0.5)
    W_o = _randn(gen, (HD, cfg.d_model), HD ** -0.5)
    u, vb, W_R = make_params(cfg, cfg.seed + 10_000 if seed is None else seed + 1)
    dt = cfg.torch_dtype
    return dict(h=h.to(dt), W_qkv=W_qkv.to(dt), W_o=W_o.to(dt), u=u, vb=vb, W_R=W_R)


def make_matrix(rows: int, cols: int, seed: int, std: float = 1.0, dtype=torch.bfloat16) -> torch.Tensor:
    """A [rows, cols] N(0, std^2) matrix in `dtype` (operands of the projection products)."""
    gen = torch.Generator().manual_seed(seed)
    return _randn(gen, (rows, cols), std).to(dtype)
