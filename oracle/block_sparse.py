"""fp64 oracle for block-sparse attention.  Test infrastructure only (see the
package docstring).

Source: [FA-notes] §4.4 "块稀疏 FlashAttention": attention may skip most
blocks because not every position needs every other one; the method keeps
FlashAttention's IO behaviour and is approximate with respect to dense
attention (the sparsity pattern drops score blocks).

Readings where the page leaves the step open (listed with the other
readings of the pages):
  * The sparsity pattern is a 0/1 block mask over (query block, key block)
    pairs; a 0 block masks all of its scores (they are -inf before the
    softmax), a 1 block keeps them.  What is computed is then the plain
    definition of attention with that mask: the result is exact for the
    masked problem.
  * Blocks are ``block`` x ``block`` (128 x 128, the tile of the kernels)
    and the mask combines with the causal mask and key padding by AND.
  * A row left with no visible key gets O_i = 0 and LSE_i = -inf, as every
    empty row does.
  * The mask is either shared by all (batch, head) pairs or given per pair.
"""
from __future__ import annotations

import numpy as np

from .attention import NEG_INF, to_f64


def expand_block_mask(block_mask, n_q: int, n_k: int, block: int = 128) -> np.ndarray:
    """Boolean [n_q, n_k] element mask of a [ceil(n_q/block), ceil(n_k/block)]
    block mask: element (i, j) takes block (i // block, j // block)."""
    bm = np.asarray(block_mask).astype(bool)
    return bm[np.arange(n_q) // block][:, np.arange(n_k) // block]


def block_sparse_forward(Q, K, V, block_mask, causal=False, scale=None, kv_lens=None, block=128,
                         rows=None):
    """Attention over [B, H, N, d] inputs whose scores outside the kept blocks
    are masked.  ``block_mask`` is [nqb, nkb] (shared) or [B, H, nqb, nkb].
    Returns O [B, H, R, d] and LSE [B, H, R] for the query ``rows`` (all N by
    default)."""
    Q, K, V = to_f64(Q), to_f64(K), to_f64(V)
    B, H, N, d = Q.shape
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    bm = np.asarray(block_mask)
    rows = np.arange(N) if rows is None else np.asarray(rows)
    O = np.zeros((B, H, len(rows), V.shape[3]))
    LSE = np.full((B, H, len(rows)), NEG_INF)
    j = np.arange(N)[None, :]
    for b in range(B):
        L = N if kv_lens is None else int(kv_lens[b])
        for h in range(H):
            m = bm if bm.ndim == 2 else bm[b, h]
            vis = expand_block_mask(m, N, N, block)[rows]
            if causal:
                vis &= j <= rows[:, None]
            vis &= j < L
            S = scale * (Q[b, h][rows] @ K[b, h].T)
            for r in range(len(rows)):
                if not vis[r].any():
                    continue
                s = S[r, vis[r]]
                mx = s.max()
                w = np.exp(s - mx)
                l = w.sum()
                O[b, h, r] = (w @ V[b, h][vis[r]]) / l
                LSE[b, h, r] = mx + np.log(l)
    return O, LSE
