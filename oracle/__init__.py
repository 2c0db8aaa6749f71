"""CPU oracle for the Sparse-Flash-MLA Softmax-L1Norm forward (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg import this package.  The product path (``softmax_l1_norm_gb300``) never
does, and this package imports nothing from it.
"""
from .smla_oracle import (  # noqa: F401
    decode_half,
    token_geometry,
    slot_key_positions,
    slot_valid,
    simple_softmax,
    reduce_sum_g_mean,
    softmax_l1_norm,
    softmax_l1_norm_rows,
    softmax_lse,
)
