"""CPU tests of the C ABI: the library builds, loads, exports every function include/txl.h
declares, and its host-side validation and kernel selection behave as documented.  Nothing here
launches a kernel (every call is rejected, or decides a path, before any CUDA work)."""
import ctypes
import importlib.util
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def native():
    spec = importlib.util.spec_from_file_location(
        "txl_build", os.path.join(ROOT, "transformer_xl_relative_gb300", "_build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build()
    from transformer_xl_relative_gb300 import native as n
    n.load()
    return n


def declared_functions():
    src = open(os.path.join(ROOT, "include", "txl.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(txl_[a-z0-9_]+)\s*\(", src)))


def test_header_lists_the_boundary():
    names = declared_functions()
    for fn in ("txl_rel_pos_gen", "txl_rel_attn_fwd", "txl_mem_push"):
        assert fn in names


def test_every_declared_function_is_exported(native):
    lib = native.load()
    for fn in declared_functions():
        assert hasattr(lib, fn), fn
    assert set(declared_functions()) == set(native.EXPORTS)


def test_status_strings_and_version(native):
    lib = native.load()
    assert lib.txl_status_str(0) == b"ok"
    assert lib.txl_status_str(5) == b"device wait timed out"
    assert lib.txl_version() >= 10000


def _view(ptr, sb, st, sh):
    return native_mod().TxlView(ptr, sb, st, sh)


def native_mod():
    from transformer_xl_relative_gb300 import native as n
    return n


FAKE = 1 << 40          # an aligned address that is never dereferenced (host-side checks only)


def _path(native, B=2, L=200, H=4, D=64, M=128, wp=0, valid=128, dtype=1, sh=None, misalign=0,
          ld_r=64):
    sh = sh or D
    V = native.TxlView
    q = V(FAKE + misalign, L * H * sh, H * sh, sh)
    kc = V(FAKE, (M + L) * H * sh, H * sh, sh)
    out = V(FAKE, L * H * sh, H * sh, sh)
    mem = native.TxlMem(FAKE, FAKE, (M + L) * H * sh, H * sh, sh, B, M, H, D, dtype, wp, valid)
    return native.load().txl_rel_attn_path(B, L, H, D, ctypes.byref(q), ctypes.byref(mem),
                                           ctypes.byref(kc), ctypes.byref(kc), FAKE, ld_r,
                                           ctypes.byref(out), dtype)


def test_path_selection(native):
    assert _path(native) == 1                                 # bf16, aligned: fused tcgen05
    assert _path(native, dtype=0) == 2                        # fp32: SIMT
    assert _path(native, D=41, sh=41, ld_r=48) == 2           # 82-byte rows: no TMA
    assert _path(native, D=41, sh=48, ld_r=48) == 1           # padded head stride: TMA
    assert _path(native, misalign=2) == 2                     # misaligned base
    assert _path(native, M=256, wp=128, valid=256) == 1       # ring aligned to 128
    assert _path(native, M=256, wp=64, valid=256) == 2        # ring not aligned
    assert _path(native, M=300, wp=128, valid=300) == 2       # ring length not a multiple
    assert _path(native, D=128, ld_r=128) == 1
    assert _path(native, D=130, ld_r=136) == -native.TXL_ERR_UNSUPPORTED
    assert _path(native, wp=128, valid=128) == -native.TXL_ERR_INVALID_ARG   # wp >= M


def _bwd_path(native, B=2, L=200, H=4, D=64, M=128, wp=0, valid=128, dtype=1, sh=None, out_off=0, grad_off=0,
              ld_r=64):
    sh = sh or D
    V = native.TxlView
    q = V(FAKE, L * H * sh, H * sh, sh)
    kc = V(FAKE, (M + L) * H * sh, H * sh, sh)
    out = V(FAKE + out_off, L * H * sh, H * sh, sh)
    mem = native.TxlMem(FAKE, FAKE, (M + L) * H * sh, H * sh, sh, B, M, H, D, dtype, wp, valid)
    return native.load().txl_rel_attn_bwd_path(B, L, H, D, ctypes.byref(q), ctypes.byref(mem), ctypes.byref(kc),
                                               ctypes.byref(kc), FAKE, ld_r, ctypes.byref(out), ctypes.byref(q),
                                               FAKE + grad_off, FAKE, FAKE, FAKE, dtype)


def test_backward_path_selection(native):
    assert _bwd_path(native) == 1                             # bf16, D 64, aligned: tcgen05 kernel
    assert _bwd_path(native, out_off=8) == 2                  # output off 16-byte alignment: mma.sync
    assert _bwd_path(native, grad_off=4) == 2                 # dq off 16-byte alignment: mma.sync
    assert _bwd_path(native, M=256, wp=128, valid=200) == 1   # ring aligned to 128
    assert _bwd_path(native, M=256, wp=64, valid=256) == 2    # ring the fused forward declines
    assert _bwd_path(native, dtype=0) == 3                    # fp32: SIMT
    assert _bwd_path(native, D=32, ld_r=32) == 3              # d_head 32: SIMT
    assert _bwd_path(native, wp=128, valid=128) == -native.TXL_ERR_INVALID_ARG   # wp >= M


def _table_path(native, B=2, L=300, H=4, D=64, max_len=512, dtype=1, sh=None, masked=False, ld_r=64):
    sh = sh or D
    V = native.TxlView
    x = V(FAKE, L * H * sh, H * sh, sh)
    return native.load().txl_rel_attn_table_path(B, L, H, D, max_len, ctypes.byref(x), ctypes.byref(x),
                                                 ctypes.byref(x), FAKE, ld_r, FAKE if masked else None,
                                                 ctypes.byref(x), dtype)


def test_table_path_selection(native):
    assert _table_path(native) == 1                               # bf16, L <= max_len: persistent tcgen05
    assert _table_path(native, masked=True) == 1                  # a key mask too
    assert _table_path(native, D=41, sh=48, ld_r=48) == 1         # padded heads, d_head <= 64
    assert _table_path(native, L=600) == 3                        # L > max_len: the mma.sync kernel
    assert _table_path(native, L=600, D=32, ld_r=32) == 2         # ... which wants d_head 64
    assert _table_path(native, dtype=0) == 2                      # fp32: CUDA cores
    assert _table_path(native, D=128, ld_r=128) == 2              # d_head above 64
    assert _table_path(native, D=130, ld_r=136) == -native.TXL_ERR_UNSUPPORTED
    assert _table_path(native, max_len=0) == -native.TXL_ERR_INVALID_ARG


def _decode_path(native, L=4, M=1024, wp=0, D=64, dtype=1):
    B, H = 2, 4
    V = native.TxlView
    q = V(FAKE, L * H * D, H * D, D)
    kc = V(FAKE, (M + L) * H * D, H * D, D)
    mem = native.TxlMem(FAKE, FAKE, (M + L) * H * D, H * D, D, B, M, H, D, dtype, wp, M)
    return native.load().txl_rel_attn_decode_path(B, L, H, D, ctypes.byref(q), ctypes.byref(mem), ctypes.byref(kc),
                                                  ctypes.byref(kc), FAKE, D, ctypes.byref(q), dtype)


def test_decode_path_selection(native):
    assert _decode_path(native) == 1                  # three or more queries: the fused kernel
    assert _decode_path(native, L=2) == 4             # one or two: the split-key decode kernels
    assert _decode_path(native, wp=100) == 4          # ring not aligned to 128
    assert _decode_path(native, dtype=0) == 4         # fp32
    assert _decode_path(native, D=128) == 4           # d_head above 64
    assert _decode_path(native, L=17) == -native.TXL_ERR_UNSUPPORTED


def test_rejections_before_any_launch(native):
    lib = native.load()
    V = native.TxlView
    q = V(FAKE, 1, 1, 1)
    nullv = V(None, 1, 1, 1)
    # null query view
    assert lib.txl_rel_attn_fwd(1, 8, 1, 8, 16, ctypes.byref(nullv), None, ctypes.byref(q),
                                ctypes.byref(q), FAKE, FAKE, FAKE, 8, 16, 0.0, ctypes.byref(q), 1,
                                None, 0, None, None) == native.TXL_ERR_INVALID_ARG
    # too few rows in r: min(M+L, clamp+1) = 8 > 4
    assert lib.txl_rel_attn_fwd(1, 8, 1, 8, 16, ctypes.byref(q), None, ctypes.byref(q),
                                ctypes.byref(q), FAKE, FAKE, FAKE, 8, 4, 0.0, ctypes.byref(q), 1,
                                None, 0, None, None) == native.TXL_ERR_INVALID_ARG
    # negative clamp
    assert lib.txl_rel_attn_fwd(1, 8, 1, 8, -1, ctypes.byref(q), None, ctypes.byref(q),
                                ctypes.byref(q), FAKE, FAKE, FAKE, 8, 16, 0.0, ctypes.byref(q), 1,
                                None, 0, None, None) == native.TXL_ERR_INVALID_ARG
    # d_head above 128
    assert lib.txl_rel_attn_fwd(1, 8, 1, 256, 16, ctypes.byref(q), None, ctypes.byref(q),
                                ctypes.byref(q), FAKE, FAKE, FAKE, 256, 16, 0.0, ctypes.byref(q), 1,
                                None, 0, None, None) == native.TXL_ERR_UNSUPPORTED
    # position table: odd d_model, misaligned bf16 W_R, d_model above the limit
    assert lib.txl_rel_pos_gen(8, 15, 2, 8, FAKE, 16, FAKE, 8, 1, None) == native.TXL_ERR_INVALID_ARG
    assert lib.txl_rel_pos_gen(8, 16, 2, 8, FAKE + 2, 16, FAKE, 8, 1, None) == native.TXL_ERR_ALIGNMENT
    assert lib.txl_rel_pos_gen(8, 16, 2, 8, FAKE, 20, FAKE, 8, 1, None) == native.TXL_ERR_ALIGNMENT
    assert lib.txl_rel_pos_gen(8, 8192, 2, 8, FAKE, 16, FAKE, 8, 1, None) == native.TXL_ERR_INVALID_ARG
    # memory push: write pointer outside the ring, and an empty segment (no work, no change)
    mem = native.TxlMem(FAKE, FAKE, 64, 8, 8, 1, 8, 1, 8, 1, 9, 0)
    assert lib.txl_mem_push(ctypes.byref(mem), ctypes.byref(q), ctypes.byref(q), 4, None) == \
        native.TXL_ERR_INVALID_ARG
    mem = native.TxlMem(FAKE, FAKE, 64, 8, 8, 1, 8, 1, 8, 1, 3, 5)
    assert lib.txl_mem_push(ctypes.byref(mem), ctypes.byref(q), ctypes.byref(q), 0, None) == native.TXL_OK
    assert (mem.wp, mem.valid) == (3, 5)
    # decode path: more than 16 queries, a missing or short workspace; the workspace formula
    ws = lib.txl_rel_attn_decode_workspace_size(2, 3, 4, 64, None)
    assert ws == 2 * 4 * 3 * 1 * (64 + 2) * 4
    mem = native.TxlMem(FAKE, FAKE, 64, 8, 8, 2, 700, 4, 64, 1, 0, 700)
    assert lib.txl_rel_attn_decode_workspace_size(2, 1, 4, 64, ctypes.byref(mem)) == 2 * 4 * 1 * 3 * 66 * 4
    assert lib.txl_rel_attn_decode_workspace_size(1, 17, 1, 8, None) == 0
    assert lib.txl_rel_attn_decode(1, 17, 1, 8, 16, ctypes.byref(q), None, ctypes.byref(q), ctypes.byref(q),
                                   FAKE, FAKE, FAKE, 8, 32, 0.0, ctypes.byref(q), 1, FAKE, 1 << 20,
                                   None) == native.TXL_ERR_UNSUPPORTED
    assert lib.txl_rel_attn_decode(1, 4, 1, 8, 16, ctypes.byref(q), None, ctypes.byref(q), ctypes.byref(q),
                                   FAKE, FAKE, FAKE, 8, 16, 0.0, ctypes.byref(q), 1, None, 0,
                                   None) == native.TXL_ERR_WORKSPACE
    assert lib.txl_rel_attn_decode(1, 4, 1, 8, 16, ctypes.byref(q), None, ctypes.byref(q), ctypes.byref(q),
                                   FAKE, FAKE, FAKE, 8, 16, 0.0, ctypes.byref(q), 1, FAKE, 16,
                                   None) == native.TXL_ERR_WORKSPACE
    # the entry point without a workspace refuses partial results beyond its 8 MiB scratch
    # (B*H*L*ceil((M+L)/256)*(D+2)*4 = 64*16*16*17*66*4 bytes here) before touching the GPU
    mem = native.TxlMem(FAKE, FAKE, 64, 8, 8, 64, 4096, 16, 64, 1, 0, 4096)
    assert lib.txl_rel_attn_decode_noalloc(64, 16, 16, 64, 1000, ctypes.byref(q), ctypes.byref(mem),
                                           ctypes.byref(q), ctypes.byref(q), FAKE, FAKE, FAKE, 64, 4112,
                                           0.0, ctypes.byref(q), 1, None) == native.TXL_ERR_WORKSPACE
    # projections: fp32 is not provided, K must be positive, rows must hold their columns, X and W
    # need 16-byte rows; an empty product is a no-op
    assert lib.txl_linear(8, 8, 8, FAKE, 8, FAKE, 8, FAKE, 8, 0, None, None) == native.TXL_ERR_UNSUPPORTED
    assert lib.txl_linear(8, 8, 0, FAKE, 8, FAKE, 8, FAKE, 8, 1, None, None) == native.TXL_ERR_INVALID_ARG
    assert lib.txl_linear(8, 16, 8, FAKE, 8, FAKE, 8, FAKE, 16, 1, None, None) == native.TXL_ERR_INVALID_ARG
    assert lib.txl_linear(8, 8, 8, FAKE + 2, 8, FAKE, 8, FAKE, 8, 1, None, None) == native.TXL_ERR_ALIGNMENT
    assert lib.txl_linear(8, 8, 12, FAKE, 12, FAKE, 8, FAKE, 8, 1, None, None) == native.TXL_ERR_ALIGNMENT
    assert lib.txl_linear(0, 8, 8, FAKE, 8, FAKE, 8, FAKE, 8, 1, None, None) == native.TXL_OK
    # layer step: workspace formula, a missing or short workspace, H*D or d_model not a multiple
    # of 8, a memory of another shape; all rejected before any launch and the memory unchanged
    assert lib.txl_rel_attn_layer_workspace_size(2, 3, 4, 64) == 2 * 3 * 4 * 64 * 8
    assert lib.txl_rel_attn_layer_workspace_size(0, 3, 4, 64) == 0
    mem = native.TxlMem(FAKE, FAKE, 64, 8, 8, 2, 8, 4, 64, 1, 0, 0)
    lay = lambda B, H, D, dm, ws, n: lib.txl_rel_attn_layer(  # noqa: E731
        B, 8, H, D, dm, 16, FAKE, dm, ctypes.byref(mem), FAKE, FAKE, FAKE, FAKE, FAKE, D, 16, 0.0, FAKE, dm,
        ws, n, None, None)
    assert lay(2, 4, 64, 128, None, 0) == native.TXL_ERR_WORKSPACE
    assert lay(2, 4, 64, 128, FAKE, 16) == native.TXL_ERR_WORKSPACE
    assert lay(2, 4, 6, 128, FAKE, 1 << 30) == native.TXL_ERR_INVALID_ARG    # D differs from the memory's
    assert lay(2, 1, 6, 128, FAKE, 1 << 30) == native.TXL_ERR_INVALID_ARG
    assert lay(2, 4, 64, 100, FAKE, 1 << 30) == native.TXL_ERR_ALIGNMENT
    assert lay(3, 4, 64, 128, FAKE, 1 << 30) == native.TXL_ERR_INVALID_ARG   # memory of B = 2
    assert (mem.wp, mem.valid) == (0, 0)
    # self-test limits
    assert lib.txl_selftest_wait_timeout(FAKE, 0, None) == native.TXL_ERR_INVALID_ARG
    assert lib.txl_selftest_wait_timeout(None, 10, None) == native.TXL_ERR_INVALID_ARG


def test_gradient_entry_points_reject_before_any_launch(native):
    """The saved-statistics forward, the two backward entry points and dW_R validate on the host:
    every call below returns its status before any CUDA work."""
    lib = native.load()
    V = native.TxlView
    B, L, H, D = 2, 8, 1, 64
    q = V(FAKE, L * H * D, H * D, D)
    nullv = V(None, 1, 1, 1)
    bq = ctypes.byref(q)

    def fwd_lse(lse, dtype=1, D=D, n_rows=16):
        return lib.txl_rel_attn_fwd_lse(B, L, H, D, 16, bq, None, bq, bq, FAKE, FAKE, FAKE, D, n_rows, 0.0, bq,
                                        lse, dtype, None, 0, None, None)

    assert fwd_lse(None) == native.TXL_ERR_INVALID_ARG               # no statistics buffer
    assert fwd_lse(FAKE + 2) == native.TXL_ERR_ALIGNMENT             # statistics not 4-byte aligned
    assert fwd_lse(FAKE, n_rows=4) == native.TXL_ERR_INVALID_ARG     # min(M + L, clamp + 1) = 8 rows of r
    assert fwd_lse(FAKE, dtype=0) == native.TXL_ERR_UNSUPPORTED      # fp32: only the fused bf16 kernel saves them
    assert fwd_lse(FAKE, D=128) == native.TXL_ERR_UNSUPPORTED        # d_head above 64

    need = lib.txl_rel_attn_bwd_workspace_size(B, L, H, D)
    rows = B * L * H
    assert need == rows * 2 * 4 + rows * D * 2 * 4                   # lse, D_i, and two fp32 [rows][D] parts
    assert lib.txl_rel_attn_bwd_workspace_size(0, L, H, D) == 0

    def bwd_lse(lse=None, dq=FAKE, d_out=q, ws=FAKE, ws_bytes=need, n_rows=16):
        return lib.txl_rel_attn_bwd_lse(B, L, H, D, 16, bq, None, bq, bq, FAKE, FAKE, FAKE, D, n_rows, 0.0, bq,
                                        ctypes.byref(d_out), lse, dq, FAKE, FAKE, FAKE, FAKE, FAKE, 1, ws,
                                        ws_bytes, None)

    assert bwd_lse(lse=FAKE + 2) == native.TXL_ERR_ALIGNMENT
    assert bwd_lse(dq=None) == native.TXL_ERR_INVALID_ARG
    assert bwd_lse(d_out=nullv) == native.TXL_ERR_INVALID_ARG
    assert bwd_lse(n_rows=4) == native.TXL_ERR_INVALID_ARG
    assert bwd_lse(ws=None, ws_bytes=0) == native.TXL_ERR_WORKSPACE
    assert bwd_lse(ws_bytes=need - 16) == native.TXL_ERR_WORKSPACE
    assert bwd_lse(ws=FAKE + 4) == native.TXL_ERR_ALIGNMENT          # workspace not 16-byte aligned
    # the entry point without statistics applies the same checks
    assert lib.txl_rel_attn_bwd(B, L, H, D, 16, bq, None, bq, bq, FAKE, FAKE, FAKE, D, 16, 0.0, bq, bq,
                                FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, None, 0, None) == native.TXL_ERR_WORKSPACE

    # dW_R: d_model even and at least 2, a destination, a row stride holding H * D columns, dr when
    # there are rows
    assert lib.txl_rel_pos_bwd(16, 15, 2, 8, FAKE, FAKE, 16, None) == native.TXL_ERR_INVALID_ARG
    assert lib.txl_rel_pos_bwd(16, 0, 2, 8, FAKE, FAKE, 16, None) == native.TXL_ERR_INVALID_ARG
    assert lib.txl_rel_pos_bwd(16, 16, 2, 8, FAKE, FAKE, 15, None) == native.TXL_ERR_INVALID_ARG
    assert lib.txl_rel_pos_bwd(16, 16, 2, 8, FAKE, None, 16, None) == native.TXL_ERR_INVALID_ARG
    assert lib.txl_rel_pos_bwd(16, 16, 2, 8, None, FAKE, 16, None) == native.TXL_ERR_INVALID_ARG


def test_empty_batch_is_a_no_op(native):
    lib = native.load()
    q = native.TxlView(FAKE, 1, 1, 1)
    assert lib.txl_rel_attn_fwd(0, 8, 1, 8, 16, ctypes.byref(q), None, ctypes.byref(q),
                                ctypes.byref(q), FAKE, FAKE, FAKE, 8, 16, 0.0, ctypes.byref(q), 1,
                                None, 0, None, None) == native.TXL_OK
    assert lib.txl_rel_pos_gen(0, 16, 2, 8, FAKE, 16, FAKE, 8, 1, None) == native.TXL_OK
