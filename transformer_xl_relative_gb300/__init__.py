"""Transformer-XL relative multi-head attention over [memory ++ current segment] for GB300.

The computation lives in libtxl.so (CUDA, sm_103a; C ABI in include/txl.h).  This package is its
Python binding: torch supplies device memory and streams, the library supplies every kernel.
Importing the package loads the library and fails loudly if it has not been built.
"""
from . import native
from .api import (  # noqa: F401
    Memory,
    linear,
    mem_push,
    rel_attn_bwd,
    rel_attn_bwd_path,
    rel_attn_decode,
    rel_attn_decode_path,
    rel_attn_decode_workspace_size,
    rel_attn_fwd,
    rel_attn_layer,
    rel_attn_layer_workspace_size,
    rel_attn_layer_fused,
    rel_attn_layer_fused_workspace_size,
    rel_attn_path,
    rel_attn_table_fwd,
    rel_attn_table_path,
    rel_pos_bwd,
    rel_pos_gen,
    selftest_wait_timeout,
    version,
)
from .native import TxlError  # noqa: F401

native.load()
