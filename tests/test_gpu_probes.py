"""Bit-exact probes of the relative-shift remap, the clamp and the masks in the fused kernel.

Scores are built so that exactly one visible key (or an exactly known set of keys) carries a
logit about 2^8 above all others, which are exactly 0; every other exponent then underflows to
0 and the output is the value vector of the winner, bit for bit.  Values are binary codes of
the key index, so a wrong winner is visible in the output.

 * remap: q = 0, u = 0 (content term exactly 0), v_bias = e_0, r[delta*] = BIG e_0, r = 0
   elsewhere -> query i picks key M + i - delta* ("跨窗口的相对位置编码" §3, term (d)).
 * clamp: r[clamp_len] = BIG e_0 -> every key at distance >= clamp_len ties
   ("TransformerXL 相对位置编码" §2.4); the output is the exact mean over that key set.
 * masks: one key carries a BIG content term (u = e_1, k_j = BIG e_1); a future key or an
   invalid memory slot must never win ("TransformerXL 相对位置编码" §4.2-4.3).
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

BIG = 2048.0     # with c = log2(e)/sqrt(D) this is >= 180 in log2 units for D <= 128


@pytest.fixture(scope="module")
def txl():
    import transformer_xl_relative_gb300 as m
    return m


def codes(n, D):
    c = np.zeros((n, D), dtype=np.float32)
    for j in range(n):
        for d in range(min(D, 12)):
            c[j, d] = ((j + 1) >> d) & 1
    return c


class Probe:
    def __init__(self, B, H, D, L, M, valid, C, hs=0, wp=0):
        self.B, self.H, self.D, self.L, self.M, self.valid, self.C, self.wp = B, H, D, L, M, valid, C, wp
        self.hs = hs or D
        K = M + L
        self.code = codes(K, D)                                  # by logical key index
        dev = "cuda"
        self.q = torch.zeros(B, L, H, self.hs, dtype=torch.bfloat16, device=dev)[..., :D]
        self.kcur = torch.zeros(B, L, H, self.hs, dtype=torch.bfloat16, device=dev)[..., :D]
        self.vcur = torch.zeros(B, L, H, self.hs, dtype=torch.bfloat16, device=dev)[..., :D]
        self.kmem = torch.zeros(B, max(M, 1), H, self.hs, dtype=torch.bfloat16, device=dev)[:, :M, :, :D]
        self.vmem = torch.zeros(B, max(M, 1), H, self.hs, dtype=torch.bfloat16, device=dev)[:, :M, :, :D]
        cv = torch.from_numpy(self.code).to(torch.bfloat16).to(dev)
        for j in range(M):
            self.vmem[:, (wp + j) % M] = cv[j][None, None, :]
        self.vcur[:] = cv[M:][None, :, None, :]
        self.u = torch.zeros(H, D, dtype=torch.float32, device=dev)
        self.vb = torch.zeros(H, D, dtype=torch.float32, device=dev)
        self.n_rows = min(M + L, C + 1)
        self.r = torch.zeros(self.n_rows, H, (D + 7) // 8 * 8, dtype=torch.bfloat16, device=dev)

    def run(self, txl):
        mem = txl.Memory(self.kmem, self.vmem, self.wp, self.valid) if self.M else None
        out = torch.zeros(self.B, self.L, self.H, self.hs, dtype=torch.bfloat16, device="cuda")[..., :self.D]
        assert txl.rel_attn_path(self.q, mem, self.kcur, self.vcur, self.r, out) == 1
        txl.rel_attn_fwd(self.q, mem, self.kcur, self.vcur, self.u, self.vb, self.r, self.n_rows,
                         self.C, out)
        torch.cuda.synchronize()
        return out.float().cpu().numpy()

    def visible(self, i):
        return list(range(self.M - self.valid, self.M + i + 1))

    def check_row(self, out, i, winners):
        """winners: the exact key set sharing the top logit (one key -> bit-exact code)."""
        exp = self.code[winners].mean(axis=0)
        got = out[:, i]                                          # [B, H, D]
        if len(winners) == 1:
            assert np.array_equal(got, np.broadcast_to(exp, got.shape)), (i, winners)
        else:
            assert np.max(np.abs(got - exp)) <= 2.0 ** -8, (i, len(winners))


SHAPES = {
    "large": dict(B=1, H=2, D=64, L=384, M=384, valid=384, C=1000),
    "base": dict(B=1, H=2, D=41, L=150, M=150, valid=150, C=1000, hs=48),
    "longmem": dict(B=1, H=1, D=64, L=128, M=1600, valid=1600, C=1000),
    "stream_ring": dict(B=1, H=1, D=128, L=512, M=2048, valid=2048, C=1000, wp=1536),
    "partial": dict(B=1, H=1, D=64, L=200, M=300, valid=170, C=1000),
}


@pytest.mark.parametrize("shape", list(SHAPES))
def test_remap_picks_key_at_distance(txl, shape):
    s = SHAPES[shape]
    for dstar in [0, 1, 63, 64, 127, 128, 129, 255, 256, 383, 500, 767, s["C"] - 1]:
        p = Probe(**s)
        if dstar >= p.n_rows or dstar >= p.C:
            continue
        p.vb[:, 0] = 1.0
        p.r[dstar, :, 0] = BIG
        out = p.run(txl)
        for i in range(p.L):
            vis = p.visible(i)
            j = p.M + i - dstar
            p.check_row(out, i, [j] if j in vis else vis)


@pytest.mark.parametrize("shape,C", [("large", 700), ("large", 128), ("longmem", 1000),
                                     ("stream_ring", 1000), ("partial", 300), ("large", 0)])
def test_clamp_ties_every_far_key(txl, shape, C):
    s = dict(SHAPES[shape])
    s["C"] = C
    p = Probe(**s)
    p.vb[:, 0] = 1.0
    p.r[C, :, 0] = BIG
    out = p.run(txl)
    for i in range(p.L):
        vis = p.visible(i)
        far = [j for j in vis if p.M + i - j >= C]
        p.check_row(out, i, far if far else vis)


@pytest.mark.parametrize("shape", ["large", "base", "partial", "stream_ring"])
def test_future_key_never_wins(txl, shape):
    s = SHAPES[shape]
    for f in [0, 5, 127, 128, 200]:
        p = Probe(**s)
        if f >= p.L:
            continue
        p.u[:, 1] = 1.0
        p.kcur[:, f, :, 1] = BIG
        out = p.run(txl)
        for i in range(p.L):
            vis = p.visible(i)
            p.check_row(out, i, [p.M + f] if i >= f else vis)


def test_invalid_memory_never_wins(txl):
    s = SHAPES["partial"]
    p = Probe(**s)
    lo = p.M - p.valid
    p.u[:, 1] = 1.0
    for j in [0, lo - 1, lo // 2]:
        p.kmem[:, j, :, 1] = BIG
    out = p.run(txl)
    for i in range(p.L):
        p.check_row(out, i, p.visible(i))
