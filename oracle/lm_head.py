"""Float64 oracle of the fused LM-head + verify step: logits from hidden states.

TEST INFRASTRUCTURE: only tests/, the smoke check and bench.py's CPU-baseline
leg may import or run this module. The library never calls it, and it shares
no code, header, table or constant with the CUDA path.

What it computes, and where the pages say so (page titles as cited):

* Every decode step ends with the output projection: the logit row of a
  position is z = h . W^T, the position's final hidden state h [d] against the
  LM-head weight W [V, d]; choosing the next token reads that row. "Apple
  Silikon İçin Cihaz Üstü Çıkarımı Optimize Etme" (perplexity.coolkeypoint.com)
  names both halves, and in its section on the limits of further optimisation
  reports that fusing the output projection with token selection was tried
  there (no end-to-end gain on that machine).
* The verify step that consumes the K+1 target rows (and K draft rows) is
  oracle.sampler.verify_batch, unchanged.

Readings where the pages are silent:
* The logits are the exact dot products of the given inputs. In float64 every
  product of two bf16 values is exact (8 + 8 significant bits), and the sums
  carry a relative error near 2^-53, far below any decision margin checked.
* A kernel that accumulates the d products in fp32, in any order, differs from
  these logits by at most logit_error_bound per logit. Parity lets a token
  differ only where a decision margin (a draw, a nucleus cut, an argmax gap)
  lies within that perturbation.
* Draft logits come either as rows or from the draft's own hidden states and
  LM-head weight. An MTP head that shares the target's W passes the same W.
"""
from __future__ import annotations

import numpy as np

from .sampler import verify_batch

# fp32 unit roundoff, doubled to cover accumulators that truncate instead of
# rounding to nearest
FP32_U = 2.0 ** -23


def lm_head_logits(h, W) -> np.ndarray:
    """z[..., v] = sum_j h[..., j] * W[v, j] in float64.

    h: [..., d] hidden states; W: [V, d] LM-head weight (one row per token).
    """
    h = np.asarray(h, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    if W.ndim != 2 or h.shape[-1] != W.shape[1]:
        raise ValueError(f"hidden size {h.shape[-1]} does not match LM-head weight {W.shape}")
    return h @ W.T


def logit_error_bound(h, W, u: float = FP32_U) -> np.ndarray:
    """Largest |z_acc - z| for a sum of the d exact products accumulated with
    unit roundoff u in any order: gamma_(d-1) * sum_j |h_j W_vj|, gamma_n =
    n u / (1 - n u) (the standard bound for recursive summation in any order,
    Higham, "Accuracy and Stability of Numerical Algorithms", section 4.2).
    """
    h = np.asarray(h, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    n = max(h.shape[-1] - 1, 0)
    gamma = n * u / (1.0 - n * u)
    return gamma * (np.abs(h) @ np.abs(W).T)


def verify_from_hidden(h_target, W_target, draft, draft_tokens, temperature, top_k, top_p,
                       seed: int, offset: int):
    """The verify step on logits computed from hidden states.

    h_target: [B, K+1, d] target hidden states; W_target: [V, d].
    draft: [B, K, V] draft logits, or a pair (h_draft [B, K, d'], W_draft [V, d']),
    or None when every temperature is 0 (greedy reads no draft row).
    Returns oracle.sampler.verify_batch's per-sequence results.
    """
    zt = lm_head_logits(h_target, W_target)
    if isinstance(draft, tuple):
        zd = lm_head_logits(*draft)
    else:
        zd = None if draft is None else np.asarray(draft, dtype=np.float64)
    if zd is not None and zd.shape[-1] != zt.shape[-1]:
        raise ValueError("draft and target vocabularies differ")
    return verify_batch(zt, zd, draft_tokens, temperature, top_k, top_p, seed, offset)
