"""fp64 CPU oracle for Transformer-XL relative attention.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` are the only callers.  The product path (the CUDA library and its Python
binding) never imports this package, and this package never imports the product path.
"""
from .oracle import (  # noqa: F401
    build,
    library,
    sinusoid,
    rel_table,
    score_terms,
    rel_attn,
    stream_attn,
    ring_push,
    ring_logical,
    attn_flops,
    linear,
    rel_layer,
    stream_layer,
    layer_flops,
    rel_attn_bwd,
    rel_attn_lse,
    table_attn,
)
