"""CPU oracle for the speculative-decoding verify-and-sample step.

TEST INFRASTRUCTURE ONLY. This package is the plain, slow, float64 statement of
what the CUDA library computes, written from the pages and pinned by the
`-m "not gpu"` tests. Only tests/, __graft_entry__.smoke() and bench.py's
CPU-baseline leg may import it. It shares no code with the CUDA path and never
imports the library package.

Every function here is pinned (see tests/test_oracle_*.py); nothing is marked
"parity unpinned". lm_head holds the logits of the fused LM-head step (h . W^T)
and feeds them to the same verify.
"""
from . import lm_head
from .philox import philox4, philox4x32_10, to_uniform, uniforms
from .sampler import (BOUNDARY, SeqResult, Truncated, accept_margin, accepts, descending_order, draft_sample,
                      inverse_cdf, residual_weights, sample_row, truncate, truncated_probs, verify_batch,
                      verify_sequence)

__all__ = [
    "lm_head",
    "philox4", "philox4x32_10", "to_uniform", "uniforms",
    "BOUNDARY", "SeqResult", "Truncated", "accept_margin", "accepts", "descending_order", "draft_sample",
    "inverse_cdf", "residual_weights", "sample_row", "truncate", "truncated_probs", "verify_batch",
    "verify_sequence",
]
