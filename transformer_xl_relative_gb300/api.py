"""Python binding of libtxl.so over torch CUDA tensors.

Argument marshalling only: every function converts tensors to pointers and element strides and
calls the C ABI of the same name; all computation happens in the library's CUDA kernels.  Torch
provides device memory and streams.  Tensors are [B, T, H, D] views whose last dimension is
contiguous; r is [n_rows, H, ld_r].
"""
from __future__ import annotations

import ctypes

import torch

from . import native
from .native import TxlMem, TxlView, check

_DTYPES = {torch.float32: native.TXL_F32, torch.bfloat16: native.TXL_BF16}


def _lib():
    return native.load()


def dtype_code(t: torch.Tensor) -> int:
    try:
        return _DTYPES[t.dtype]
    except KeyError:
        raise TypeError("libtxl computes in float32 or bfloat16, got %s" % t.dtype) from None


def view(t: torch.Tensor) -> TxlView:
    """[B, T, H, D] tensor with contiguous D -> txl_view."""
    if t.dim() != 4:
        raise ValueError("expected a [B, T, H, D] tensor, got shape %s" % (tuple(t.shape),))
    if t.shape[-1] > 1 and t.stride(-1) != 1:
        raise ValueError("the last (d) dimension must be contiguous")
    if not t.is_cuda:
        raise ValueError("tensors must live on a CUDA device")
    return TxlView(t.data_ptr(), t.stride(0), t.stride(1), t.stride(2))


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


class Memory:
    """K/V memory of M positions per batch entry (FIFO ring, or a plain contiguous memory).

    ``k`` and ``v`` are [B, M, H, D] tensors (same strides).  ``wp``/``valid`` follow txl_mem:
    logical memory key j lives in slot (wp + j) mod M and is valid iff j >= M - valid.
    """

    def __init__(self, k: torch.Tensor, v: torch.Tensor, wp: int = 0, valid: int = 0):
        if k.shape != v.shape or k.stride() != v.stride() or k.dtype != v.dtype:
            raise ValueError("k and v must share shape, strides and dtype")
        self.k, self.v = k, v
        B, M, H, D = k.shape
        self._c = TxlMem(k.data_ptr() if M else None, v.data_ptr() if M else None,
                         k.stride(0), k.stride(1), k.stride(2), B, M, H, D, dtype_code(k), wp, valid)

    @classmethod
    def empty(cls, B, M, H, D, dtype=torch.bfloat16, device="cuda", head_stride=None):
        hs = head_stride or D
        store = torch.zeros(B, M, H, hs, dtype=dtype, device=device)
        store2 = torch.zeros(B, M, H, hs, dtype=dtype, device=device)
        return cls(store[..., :D], store2[..., :D], 0, 0)

    @classmethod
    def full(cls, k: torch.Tensor, v: torch.Tensor):
        """A contiguous memory, oldest position first, every slot valid."""
        return cls(k, v, 0, k.shape[1])

    @property
    def M(self) -> int:
        return self._c.M

    @property
    def wp(self) -> int:
        return self._c.wp

    @property
    def valid(self) -> int:
        return self._c.valid

    def state(self):
        """Host ring state (wp, valid): with the buffers, everything needed to resume."""
        return self._c.wp, self._c.valid

    def restore(self, wp: int, valid: int) -> None:
        self._c.wp, self._c.valid = int(wp), int(valid)

    @property
    def c_struct(self) -> TxlMem:
        return self._c


def rel_pos_gen(W_R: torch.Tensor, r: torch.Tensor, n_rows: int, d_model: int, n_head: int,
                d_head: int, stream=None) -> torch.Tensor:
    """r[delta, h, d] = sum_m R_delta[m] W_R[m, h*d_head + d] for delta < n_rows (txl_rel_pos_gen)."""
    if W_R.dim() != 2 or W_R.stride(1) != 1 or r.dim() != 3 or r.stride(2) != 1:
        raise ValueError("W_R must be [d_model, ld_w] and r [n_rows, H, ld_r] with unit last stride")
    if r.stride(1) * n_head != r.stride(0) and r.shape[0] > 1:
        raise ValueError("r rows must be n_head * ld_r elements apart")
    st = _lib().txl_rel_pos_gen(n_rows, d_model, n_head, d_head, W_R.data_ptr(), W_R.stride(0),
                                r.data_ptr(), r.stride(1), dtype_code(W_R), _stream(stream))
    check(st, "txl_rel_pos_gen")
    return r


def _attn_args(q, mem, k_cur, v_cur, r, out):
    B, L, H, D = q.shape
    memc = ctypes.byref(mem.c_struct) if mem is not None else None
    return (B, L, H, D), memc, view(q), view(k_cur), view(v_cur), view(out)


def rel_attn_fwd(q: torch.Tensor, mem: Memory | None, k_cur: torch.Tensor, v_cur: torch.Tensor,
                 u: torch.Tensor, v_bias: torch.Tensor, r: torch.Tensor, n_rows: int,
                 clamp_len: int, out: torch.Tensor, scale: float = 0.0,
                 err_flag: torch.Tensor | None = None, stream=None, lse: torch.Tensor | None = None) -> torch.Tensor:
    """One relative-attention call over [memory ++ current] (txl_rel_attn_fwd).  With `lse` (fp32
    [B, L, H]) the call also saves every row's log-sum-exp for rel_attn_bwd (txl_rel_attn_fwd_lse)."""
    (B, L, H, D), memc, vq, vk, vv, vo = _attn_args(q, mem, k_cur, v_cur, r, out)
    if u.dtype != torch.float32 or v_bias.dtype != torch.float32:
        raise TypeError("u and v_bias are fp32 [H, D]")
    if not (u.is_contiguous() and v_bias.is_contiguous()):
        raise ValueError("u and v_bias must be contiguous [H, D]")
    ef = err_flag.data_ptr() if err_flag is not None else None
    if lse is not None:
        _check_lse(lse, B, L, H)
        st = _lib().txl_rel_attn_fwd_lse(
            B, L, H, D, int(clamp_len), ctypes.byref(vq), memc, ctypes.byref(vk), ctypes.byref(vv),
            u.data_ptr(), v_bias.data_ptr(), r.data_ptr(), r.stride(1), int(n_rows), float(scale),
            ctypes.byref(vo), lse.data_ptr(), dtype_code(q), None, 0, ef, _stream(stream))
        check(st, "txl_rel_attn_fwd_lse")
        return out
    st = _lib().txl_rel_attn_fwd(
        B, L, H, D, int(clamp_len), ctypes.byref(vq), memc, ctypes.byref(vk), ctypes.byref(vv),
        u.data_ptr(), v_bias.data_ptr(), r.data_ptr(), r.stride(1), int(n_rows), float(scale),
        ctypes.byref(vo), dtype_code(q), None, 0, ef, _stream(stream))
    check(st, "txl_rel_attn_fwd")
    return out


def _check_lse(lse: torch.Tensor, B: int, L: int, H: int) -> None:
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, L, H) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 [B, L, H] tensor")


def rel_attn_decode_workspace_size(q: torch.Tensor, mem: Memory | None) -> int:
    """Bytes of workspace rel_attn_decode needs (txl_rel_attn_decode_workspace_size)."""
    B, L, H, D = q.shape
    memc = ctypes.byref(mem.c_struct) if mem is not None else None
    return int(_lib().txl_rel_attn_decode_workspace_size(B, L, H, D, memc))


def rel_attn_decode(q: torch.Tensor, mem: Memory | None, k_cur: torch.Tensor, v_cur: torch.Tensor,
                    u: torch.Tensor, v_bias: torch.Tensor, r: torch.Tensor, n_rows: int,
                    clamp_len: int, out: torch.Tensor, scale: float = 0.0,
                    workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Attention of 1..16 queries per (b, h) over a long memory, keys split across CTAs
    (txl_rel_attn_decode).  Without `workspace`, a device buffer of the required size is taken
    from torch's allocator for the call."""
    (B, L, H, D), memc, vq, vk, vv, vo = _attn_args(q, mem, k_cur, v_cur, r, out)
    if u.dtype != torch.float32 or v_bias.dtype != torch.float32:
        raise TypeError("u and v_bias are fp32 [H, D]")
    if not (u.is_contiguous() and v_bias.is_contiguous()):
        raise ValueError("u and v_bias must be contiguous [H, D]")
    need = rel_attn_decode_workspace_size(q, mem)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    nbytes = workspace.numel() * workspace.element_size()
    st = _lib().txl_rel_attn_decode(
        B, L, H, D, int(clamp_len), ctypes.byref(vq), memc, ctypes.byref(vk), ctypes.byref(vv),
        u.data_ptr(), v_bias.data_ptr(), r.data_ptr(), r.stride(1), int(n_rows), float(scale),
        ctypes.byref(vo), dtype_code(q), workspace.data_ptr(), nbytes, _stream(stream))
    check(st, "txl_rel_attn_decode")
    return out


def rel_attn_path(q, mem, k_cur, v_cur, r, out) -> int:
    """1 = fused tcgen05 kernel, 2 = SIMT kernel (txl_rel_attn_path)."""
    (B, L, H, D), memc, vq, vk, vv, vo = _attn_args(q, mem, k_cur, v_cur, r, out)
    return _lib().txl_rel_attn_path(B, L, H, D, ctypes.byref(vq), memc, ctypes.byref(vk),
                                    ctypes.byref(vv), r.data_ptr(), r.stride(1), ctypes.byref(vo),
                                    dtype_code(q))


def rel_attn_decode_path(q, mem, k_cur, v_cur, r, out) -> int:
    """1 = fused tcgen05 kernel, 4 = split-key decode kernels (txl_rel_attn_decode_path)."""
    (B, L, H, D), memc, vq, vk, vv, vo = _attn_args(q, mem, k_cur, v_cur, r, out)
    return _lib().txl_rel_attn_decode_path(B, L, H, D, ctypes.byref(vq), memc, ctypes.byref(vk),
                                           ctypes.byref(vv), r.data_ptr(), r.stride(1), ctypes.byref(vo),
                                           dtype_code(q))


def rel_attn_bwd_path(q, mem, k_cur, v_cur, r, out, d_out, g: dict) -> int:
    """1 = tcgen05 gradient kernel, 2 = mma.sync, 3 = SIMT (txl_rel_attn_bwd_path), for the gradient
    buffers g (as rel_attn_bwd returns them: dq, dk_cur, dv_cur, dr)."""
    (B, L, H, D), memc, vq, vk, vv, vo = _attn_args(q, mem, k_cur, v_cur, r, out)
    vg = view(d_out)
    return _lib().txl_rel_attn_bwd_path(B, L, H, D, ctypes.byref(vq), memc, ctypes.byref(vk), ctypes.byref(vv),
                                        r.data_ptr(), r.stride(1), ctypes.byref(vo), ctypes.byref(vg),
                                        g["dq"].data_ptr(), g["dk_cur"].data_ptr(), g["dv_cur"].data_ptr(),
                                        g["dr"].data_ptr(), dtype_code(q))


def mem_push(mem: Memory, k_new: torch.Tensor, v_new: torch.Tensor, stream=None) -> Memory:
    """Append k_new/v_new [B, L, H, D] to the FIFO memory (txl_mem_push)."""
    vk, vv = view(k_new), view(v_new)
    st = _lib().txl_mem_push(ctypes.byref(mem.c_struct), ctypes.byref(vk), ctypes.byref(vv),
                             k_new.shape[1], _stream(stream))
    check(st, "txl_mem_push")
    return mem


def _rows2d(t: torch.Tensor, what: str):
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError("%s must be a 2-D tensor with unit column stride" % what)
    return t.data_ptr(), t.stride(0)


def linear(X: torch.Tensor, W: torch.Tensor, Y: torch.Tensor | None = None,
           err_flag: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Y = X W for bf16 X [m, k] and W [k, n] (txl_linear); Y [m, n] is allocated if not given."""
    m, k = X.shape
    k2, n = W.shape
    if k2 != k:
        raise ValueError("inner dimensions differ")
    if Y is None:
        Y = torch.empty(m, n, dtype=X.dtype, device=X.device)
    px, ldx = _rows2d(X, "X")
    pw, ldw = _rows2d(W, "W")
    py, ldy = _rows2d(Y, "Y")
    st = _lib().txl_linear(m, n, k, px, ldx, pw, ldw, py, ldy, dtype_code(X),
                           err_flag.data_ptr() if err_flag is not None else None, _stream(stream))
    check(st, "txl_linear")
    return Y


def rel_attn_layer_workspace_size(B: int, L: int, H: int, D: int) -> int:
    """Bytes of workspace rel_attn_layer needs (txl_rel_attn_layer_workspace_size)."""
    return int(_lib().txl_rel_attn_layer_workspace_size(B, L, H, D))


def rel_attn_layer(h: torch.Tensor, mem: Memory | None, W_qkv: torch.Tensor, W_o: torch.Tensor,
                   u: torch.Tensor, v_bias: torch.Tensor, r: torch.Tensor, n_rows: int, clamp_len: int,
                   n_head: int, d_head: int, y: torch.Tensor | None = None, scale: float = 0.0,
                   workspace: torch.Tensor | None = None, err_flag: torch.Tensor | None = None,
                   stream=None) -> torch.Tensor:
    """One attention-layer step over hidden states h [B, L, d_model] (txl_rel_attn_layer): the
    projections, the relative attention over [memory ++ segment], the output projection, and the
    push of the segment's keys and values into `mem`.  Returns y [B, L, d_model]."""
    B, L, d_model = h.shape
    if h.stride(2) != 1 or (B > 1 and h.stride(0) != L * h.stride(1)):
        raise ValueError("h must be [B, L, d_model] with rows b*L + t evenly spaced")
    if u.dtype != torch.float32 or v_bias.dtype != torch.float32:
        raise TypeError("u and v_bias are fp32 [H, D]")
    if not (u.is_contiguous() and v_bias.is_contiguous() and W_qkv.is_contiguous() and W_o.is_contiguous()):
        raise ValueError("u, v_bias, W_qkv and W_o must be contiguous")
    if y is None:
        y = torch.empty(B, L, d_model, dtype=h.dtype, device=h.device)
    if y.stride(2) != 1 or (B > 1 and y.stride(0) != L * y.stride(1)):
        raise ValueError("y must be [B, L, d_model] with rows b*L + t evenly spaced")
    need = rel_attn_layer_workspace_size(B, L, n_head, d_head)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=h.device)
    nbytes = workspace.numel() * workspace.element_size()
    memc = ctypes.byref(mem.c_struct) if mem is not None else None
    st = _lib().txl_rel_attn_layer(
        B, L, n_head, d_head, d_model, int(clamp_len), h.data_ptr(), h.stride(1), memc, W_qkv.data_ptr(),
        W_o.data_ptr(), u.data_ptr(), v_bias.data_ptr(), r.data_ptr(), r.stride(1), int(n_rows), float(scale),
        y.data_ptr(), y.stride(1), workspace.data_ptr(), nbytes,
        err_flag.data_ptr() if err_flag is not None else None, _stream(stream))
    check(st, "txl_rel_attn_layer")
    return y


def rel_attn_layer_fused_workspace_size(B: int, L: int, H: int, D: int) -> int:
    """Bytes of workspace rel_attn_layer_fused needs (txl_rel_attn_layer_fused_workspace_size)."""
    return int(_lib().txl_rel_attn_layer_fused_workspace_size(B, L, H, D))


def rel_attn_layer_fused(h: torch.Tensor, mem: Memory, mem_len: int, W_qkv: torch.Tensor, W_o: torch.Tensor,
                         u: torch.Tensor, v_bias: torch.Tensor, r: torch.Tensor, n_rows: int, clamp_len: int,
                         n_head: int, d_head: int, y: torch.Tensor | None = None, scale: float = 0.0,
                         workspace: torch.Tensor | None = None, err_flag: torch.Tensor | None = None,
                         stream=None) -> torch.Tensor:
    """The layer step of rel_attn_layer with the memory push folded into the projection
    (txl_rel_attn_layer_fused): `mem` is a ring of at least mem_len + L slots (Memory.empty(B,
    slots, H, D)) holding a memory of mem_len positions.  Returns y [B, L, d_model]."""
    B, L, d_model = h.shape
    if h.stride(2) != 1 or (B > 1 and h.stride(0) != L * h.stride(1)):
        raise ValueError("h must be [B, L, d_model] with rows b*L + t evenly spaced")
    if u.dtype != torch.float32 or v_bias.dtype != torch.float32:
        raise TypeError("u and v_bias are fp32 [H, D]")
    if not (u.is_contiguous() and v_bias.is_contiguous() and W_qkv.is_contiguous() and W_o.is_contiguous()):
        raise ValueError("u, v_bias, W_qkv and W_o must be contiguous")
    if y is None:
        y = torch.empty(B, L, d_model, dtype=h.dtype, device=h.device)
    if y.stride(2) != 1 or (B > 1 and y.stride(0) != L * y.stride(1)):
        raise ValueError("y must be [B, L, d_model] with rows b*L + t evenly spaced")
    need = rel_attn_layer_fused_workspace_size(B, L, n_head, d_head)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=h.device)
    nbytes = workspace.numel() * workspace.element_size()
    st = _lib().txl_rel_attn_layer_fused(
        B, L, n_head, d_head, d_model, int(clamp_len), h.data_ptr(), h.stride(1), ctypes.byref(mem.c_struct),
        int(mem_len), W_qkv.data_ptr(), W_o.data_ptr(), u.data_ptr(), v_bias.data_ptr(), r.data_ptr(), r.stride(1),
        int(n_rows), float(scale), y.data_ptr(), y.stride(1), workspace.data_ptr(), nbytes,
        err_flag.data_ptr() if err_flag is not None else None, _stream(stream))
    check(st, "txl_rel_attn_layer_fused")
    return y


def rel_attn_bwd(q: torch.Tensor, mem: Memory | None, k_cur: torch.Tensor, v_cur: torch.Tensor,
                 u: torch.Tensor, v_bias: torch.Tensor, r: torch.Tensor, n_rows: int, clamp_len: int,
                 out: torch.Tensor, d_out: torch.Tensor, scale: float = 0.0,
                 workspace: torch.Tensor | None = None, stream=None, lse: torch.Tensor | None = None) -> dict:
    """Gradients of one rel_attn_fwd call for the upstream gradient d_out (txl_rel_attn_bwd; with
    `lse`, the statistics rel_attn_fwd saved for this call, txl_rel_attn_bwd_lse).
    Returns fp32 tensors dq, dk_cur, dv_cur [B, L, H, D], du, dv_bias [H, D], dr [n_rows, H, D]."""
    (B, L, H, D), memc, vq, vk, vv, vo = _attn_args(q, mem, k_cur, v_cur, r, out)
    vg = view(d_out)
    if u.dtype != torch.float32 or v_bias.dtype != torch.float32:
        raise TypeError("u and v_bias are fp32 [H, D]")
    f32 = dict(dtype=torch.float32, device=q.device)
    g = {"dq": torch.empty(B, L, H, D, **f32), "dk_cur": torch.empty(B, L, H, D, **f32),
         "dv_cur": torch.empty(B, L, H, D, **f32), "du": torch.empty(H, D, **f32),
         "dv_bias": torch.empty(H, D, **f32), "dr": torch.empty(n_rows, H, D, **f32)}
    need = int(_lib().txl_rel_attn_bwd_workspace_size(B, L, H, D))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if lse is not None:
        _check_lse(lse, B, L, H)
    st = _lib().txl_rel_attn_bwd_lse(
        B, L, H, D, int(clamp_len), ctypes.byref(vq), memc, ctypes.byref(vk), ctypes.byref(vv),
        u.data_ptr(), v_bias.data_ptr(), r.data_ptr(), r.stride(1), int(n_rows), float(scale),
        ctypes.byref(vo), ctypes.byref(vg), lse.data_ptr() if lse is not None else None,
        g["dq"].data_ptr(), g["dk_cur"].data_ptr(), g["dv_cur"].data_ptr(),
        g["du"].data_ptr(), g["dv_bias"].data_ptr(), g["dr"].data_ptr(), dtype_code(q), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _stream(stream))
    check(st, "txl_rel_attn_bwd_lse" if lse is not None else "txl_rel_attn_bwd")
    return g


def rel_pos_bwd(dr: torch.Tensor, d_model: int, dW_R: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """dW_R [d_model, H*D] = sum_delta R_delta^T dr[delta] for fp32 dr [n_rows, H, D] (txl_rel_pos_bwd)."""
    n_rows, H, D = dr.shape
    if not dr.is_contiguous() or dr.dtype != torch.float32:
        raise ValueError("dr must be a contiguous fp32 [n_rows, H, D] tensor")
    if dW_R is None:
        dW_R = torch.empty(d_model, H * D, dtype=torch.float32, device=dr.device)
    st = _lib().txl_rel_pos_bwd(n_rows, d_model, H, D, dr.data_ptr(), dW_R.data_ptr(), dW_R.stride(0),
                                _stream(stream))
    check(st, "txl_rel_pos_bwd")
    return dW_R


def rel_attn_table_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, u: torch.Tensor,
                       v_bias: torch.Tensor, r_table: torch.Tensor, max_len: int, out: torch.Tensor,
                       key_mask: torch.Tensor | None = None, scale: float = 0.0, stream=None) -> torch.Tensor:
    """The learned-table variant (txl_rel_attn_table_fwd): bidirectional attention over q, k, v
    [B, L, H, D] with the position vector of a pair read from r_table [2 max_len - 1, H, ld_r] at
    clamp(i - j + max_len - 1); key_mask [B, L] uint8 (0 = masked) or None."""
    B, L, H, D = q.shape
    if u.dtype != torch.float32 or v_bias.dtype != torch.float32:
        raise TypeError("u and v_bias are fp32 [H, D]")
    if key_mask is not None and (key_mask.dtype != torch.uint8 or not key_mask.is_contiguous()):
        raise TypeError("key_mask must be a contiguous uint8 [B, L] tensor")
    vq, vk, vv, vo = view(q), view(k), view(v), view(out)
    st = _lib().txl_rel_attn_table_fwd(
        B, L, H, D, int(max_len), ctypes.byref(vq), ctypes.byref(vk), ctypes.byref(vv), u.data_ptr(),
        v_bias.data_ptr(), r_table.data_ptr(), r_table.stride(1),
        key_mask.data_ptr() if key_mask is not None else None, float(scale), ctypes.byref(vo), dtype_code(q),
        _stream(stream))
    check(st, "txl_rel_attn_table_fwd")
    return out


def rel_attn_table_path(q, k, v, r_table, max_len: int, out, key_mask=None) -> int:
    """1 = persistent tcgen05 kernel, 3 = mma.sync tensor-core kernel, 2 = CUDA-core kernel
    (txl_rel_attn_table_path)."""
    B, L, H, D = q.shape
    vq, vk, vv, vo = view(q), view(k), view(v), view(out)
    return _lib().txl_rel_attn_table_path(
        B, L, H, D, int(max_len), ctypes.byref(vq), ctypes.byref(vk), ctypes.byref(vv), r_table.data_ptr(),
        r_table.stride(1), key_mask.data_ptr() if key_mask is not None else None, ctypes.byref(vo), dtype_code(q))


def selftest_wait_timeout(err_flag: torch.Tensor, timeout_us: int, stream=None) -> None:
    st = _lib().txl_selftest_wait_timeout(err_flag.data_ptr(), int(timeout_us), _stream(stream))
    check(st, "txl_selftest_wait_timeout")


def version() -> int:
    return _lib().txl_version()
