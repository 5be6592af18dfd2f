"""fp64 CPU oracle for the FMHA backward pass (test infrastructure only).

Only tests, the smoke check and the CPU-baseline legs of the benchmark may
import this package; the product path never does.
"""
from .attn_ref import (  # noqa: F401
    MASK_CAUSAL_BOTTOM_RIGHT,
    MASK_CAUSAL_TOP_LEFT,
    MASK_NONE,
    MASK_WINDOW,
    attn_backward,
    attn_forward,
    dkv_rows,
    dq_rows,
    visible,
    visible_pairs,
)
