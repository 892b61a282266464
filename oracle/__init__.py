"""CPU oracle of the single-GPU MoE layer -- TEST INFRASTRUCTURE ONLY.

Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference leg
may import this package.  The CUDA library and its Python binding never do.

The arithmetic lives in moe_oracle.c (plain C, double precision, naive loops);
this package compiles it with gcc, loads it with ctypes and composes the layer
from its steps in the order the Primus MoE blog's Figure 7 dataflow lists them:
route -> permute -> FC1/SwiGLU/FC2 per expert -> combine, and the backward by
dispatch/combine duality.
"""

from .layer import (  # noqa: F401
    build,
    bf16,
    route,
    layer_fwd,
    layer_bwd,
    layer_sampled,
    permute,
    combine,
    combine_bwd,
    unpermute_reduce,
    ffn_fwd_rows,
    ffn_bwd_rows,
    ffn_bwd_rows_dispatch,
    e4m3,
    e4m3_code,
    mx_quantize_rows,
    mx_quantize_cols,
    ffn_fwd_rows_mx,
    ffn_bwd_rows_mx,
    ffn_wgrad_rows_mx,
    HostSource,
    TorchSource,
    threads,
)
