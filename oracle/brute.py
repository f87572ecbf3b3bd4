"""Literal numpy fp64 forms for tiny shapes -- TEST INFRASTRUCTURE ONLY.

Independent of ``bsa_oracle.c``: it materialises the full N x N token mask,
fills the disallowed scores with -inf and takes a full-row softmax, which is
the naive masked attention of "Sparse Attention Kernels vs Full Attention
Performance" (section "How Sparse Attention Kernels Actually Speed Up
Inference": build a boolean mask, ``scores.masked_fill(mask, -inf)``,
softmax, times V).  The token windows follow "Flash MSA Sparse Attention vs
Full Attention" (section "The Mechanics": ``Mask[i][j] = 1 if |i - j| <= W``
and the causal form ``j >= i - W and j <= i`` of its pseudocode).
"""

from __future__ import annotations

import numpy as np


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def token_window_mask(N: int, W: int, causal: bool) -> np.ndarray:
    """Allowed[q, k]: |q - k| <= W, and k <= q when causal."""
    q = np.arange(N)[:, None]
    k = np.arange(N)[None, :]
    m = np.abs(q - k) <= W
    if causal:
        m &= k <= q
    return m


def block_mask_from_csr(row_ptr: np.ndarray, col_idx: np.ndarray, nb: int, r0: int = 0) -> np.ndarray:
    """nb x nb boolean block mask of the rows r0 .. r0+nb-1 of a CSR."""
    bm = np.zeros((nb, nb), dtype=bool)
    for i in range(nb):
        for e in range(int(row_ptr[r0 + i]), int(row_ptr[r0 + i + 1])):
            bm[i, int(col_idx[e])] = True
    return bm


def expand_block_mask(bm: np.ndarray, block: int, causal: bool, noncausal_rows=None) -> np.ndarray:
    """Token mask A[q, k] = BM[q // block, k // block] and (not causal or k <= q);
    query blocks listed in ``noncausal_rows`` keep every key of their blocks
    (global query rows of a causal model)."""
    a = np.kron(bm.astype(np.uint8), np.ones((block, block), dtype=np.uint8)).astype(bool)
    if causal:
        n = a.shape[0]
        cut = np.arange(n)[None, :] <= np.arange(n)[:, None]
        if noncausal_rows is not None:
            for i in noncausal_rows:
                cut[i * block:(i + 1) * block, :] = True
        a &= cut
    return a


def masked_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, allowed: np.ndarray,
                     scale: float):
    """Full-row masked softmax attention for one head, all fp64.

    q, k, v: [N, D] fp64; allowed: [N, N] bool.  Returns (O [N, D], LSE [N]).
    Rows with no allowed key give O = 0 and LSE = -inf.
    """
    s = (q @ k.T) * scale
    s = np.where(allowed, s, -np.inf)
    m = s.max(axis=1, keepdims=True)
    empty = ~np.isfinite(m[:, 0])
    m = np.where(np.isfinite(m), m, 0.0)
    p = np.exp(s - m)
    l = p.sum(axis=1, keepdims=True)
    safe_l = np.where(l > 0, l, 1.0)
    o = (p @ v) / safe_l
    lse = (m + np.log(safe_l))[:, 0]
    o[empty] = 0.0
    lse[empty] = -np.inf
    return o, lse
