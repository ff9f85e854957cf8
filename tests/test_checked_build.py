"""The range-checked build of the library (libtxl_checked.so, -DTXL_CHECKED).

CPU: it compiles for sm_103a from the same sources and exports every function include/txl.h
declares; the normal build reports itself unchecked.
GPU: a child process with TXL_CHECKED=1 loads the checked library and runs the paths whose kernels
check their indices -- the persistent fused attention over a ring with a nonzero write pointer, the
fused layer step (keys read from the ring), the SIMT attention and the memory push -- with no
failed check and results bit-identical to the normal library's; the self-test then adds exactly
one failure, and clearing resets the counter."""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _build_module():
    import importlib.util
    spec = importlib.util.spec_from_file_location("txl_build", os.path.join(ROOT, "transformer_xl_relative_gb300", "_build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_checked_library_builds_and_exports_everything():
    from transformer_xl_relative_gb300 import native
    path = _build_module().build(checked=True)
    lib = ctypes.CDLL(path)
    for name in native.EXPORTS:
        assert hasattr(lib, name), name
    lib.txl_checked_build.restype = ctypes.c_int
    assert lib.txl_checked_build() == 1
    plain = ctypes.CDLL(_build_module().build())
    plain.txl_checked_build.restype = ctypes.c_int
    assert plain.txl_checked_build() == 0


# The paths run in both processes; the seeded inputs are the same there.
RUN = r'''
import sys, torch
sys.path.insert(0, ROOT)
import transformer_xl_relative_gb300 as txl
import txl_inputs

def run():
    outs = {}
    # persistent fused attention over a ring (write pointer 128, partly valid memory)
    cfg = txl_inputs.custom(B=2, H=2, D=64, d_model=128, L=200, M=256, clamp_len=300, dtype="bf16", seed=5)
    c = txl_inputs.make_case(cfg)
    q, k, v = (c[n].cuda() for n in ("q", "k", "v"))
    r = torch.empty(cfg.n_rows, 2, 64, dtype=torch.bfloat16, device="cuda")
    txl.rel_pos_gen(c["W_R"].cuda(), r, cfg.n_rows, 128, 2, 64)
    ring_k, ring_v = torch.zeros_like(k[:, :256]), torch.zeros_like(v[:, :256])
    slots = (128 + torch.arange(256)) % 256
    ring_k[:, slots], ring_v[:, slots] = k[:, :256], v[:, :256]
    mem = txl.Memory(ring_k, ring_v, 128, 200)
    o = torch.empty_like(q)
    txl.rel_attn_fwd(q, mem, k[:, 256:], v[:, 256:], c["u"].cuda(), c["vb"].cuda(), r, cfg.n_rows, 300, o)
    outs["fused"] = o
    # the memory push into that ring
    txl.mem_push(mem, k[:, 256:], v[:, 256:])
    outs["ring_k"], outs["ring_v"] = ring_k, ring_v
    # the SIMT attention (fp32)
    cf = txl_inputs.custom(B=1, H=2, D=16, d_model=32, L=20, M=12, clamp_len=9, dtype="f32", seed=6)
    cc = txl_inputs.make_case(cf)
    qf, kf, vf = (cc[n].cuda() for n in ("q", "k", "v"))
    rf = torch.empty(cf.n_rows, 2, 16, device="cuda")
    txl.rel_pos_gen(cc["W_R"].cuda(), rf, cf.n_rows, 32, 2, 16)
    of = torch.empty_like(qf)
    txl.rel_attn_fwd(qf, txl.Memory(kf[:, :12], vf[:, :12], 0, 12), kf[:, 12:], vf[:, 12:], cc["u"].cuda(),
                     cc["vb"].cuda(), rf, cf.n_rows, 9, of)
    outs["simt"] = of
    # two fused layer steps (every key read from a ring of 256 slots)
    cl = txl_inputs.custom(B=1, H=2, D=64, d_model=128, L=128, M=128, clamp_len=1000, dtype="bf16", seed=7)
    lay = txl_inputs.make_layer(cl, segments=2)
    rl = torch.empty(256, 2, 64, dtype=torch.bfloat16, device="cuda")
    txl.rel_pos_gen(lay["W_R"].cuda(), rl, 256, 128, 2, 64)
    lring = txl.Memory.empty(1, 256, 2, 64)
    h = lay["h"].cuda()
    for s in range(2):
        outs["layer%d" % s] = txl.rel_attn_layer_fused(h[:, 128 * s:128 * (s + 1)].contiguous(), lring, 128,
                                                       lay["W_qkv"].cuda(), lay["W_o"].cuda(), lay["u"].cuda(),
                                                       lay["vb"].cuda(), rl, 256, 1000, 2, 64)
    torch.cuda.synchronize()
    return {k_: t.cpu() for k_, t in outs.items()}
'''

CHILD = r'''
import ctypes, importlib.util, os, sys
ROOT = sys.argv[1]
spec = importlib.util.spec_from_file_location("checked_test", os.path.join(ROOT, "tests", "test_checked_build.py"))
T = importlib.util.module_from_spec(spec)
spec.loader.exec_module(T)
g = {"ROOT": ROOT}
exec(T.RUN, g)
run = g["run"]
import torch
from transformer_xl_relative_gb300 import native
lib = native.load()
assert lib.txl_checked_build() == 1, "not the checked library"
assert lib.txl_range_errors_clear() == 0
res = run()
n = ctypes.c_int(-1)
assert lib.txl_range_errors(ctypes.byref(n)) == 0
errors_after_paths = n.value
assert lib.txl_selftest_range_check(None) == 0
assert lib.txl_range_errors(ctypes.byref(n)) == 0
errors_after_selftest = n.value
assert lib.txl_range_errors_clear() == 0
assert lib.txl_range_errors(ctypes.byref(n)) == 0
torch.save({"outs": res, "counts": (errors_after_paths, errors_after_selftest, n.value)}, sys.argv[2])
'''


@pytest.mark.gpu
def test_checked_library_on_the_gpu(tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    _build_module().build(checked=True)
    out_file = str(tmp_path / "checked.pt")
    env = dict(os.environ, TXL_CHECKED="1")
    proc = subprocess.run([sys.executable, "-c", CHILD, ROOT, out_file], env=env, capture_output=True, text=True,
                          timeout=600)
    assert proc.returncode == 0, proc.stderr[-3000:]
    got = torch.load(out_file)
    assert got["counts"] == (0, 1, 0)
    g = {"ROOT": ROOT}
    exec(RUN, g)
    ref = g["run"]()                          # the normal library, in this process
    for name, t in ref.items():
        assert torch.equal(got["outs"][name], t), name
