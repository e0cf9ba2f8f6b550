"""fp64 oracle: standard (materialised) attention, its analytic backward, and
the pages' two streaming formulations.  Test infrastructure only (see the
package docstring); nothing in the library's product path imports this.

Notation follows [FA-notes] §2.1: Q, K, V in R^{N x d};
S = scale * Q K^T, P = softmax(S) row-wise over the valid keys, O = P V.
The stored row statistic is LSE_i = m_i + ln(l_i) (natural log, scaled-logit
units), the single number that replaces the pair (m, l) of [FA-notes] §3.3.

Valid keys of query row i in batch b (readings of the pages' masking remarks,
[FA-notes] §3.4 and [S12] exercise 2):
    A(i) = { j : (not causal or j <= i) and j < L_b },   L_b = N without padding.
Causal masking is top-left aligned on a square matrix.  A row with empty A(i)
returns O_i = 0 and LSE_i = -inf (the pages name the hazard, not the output).
"""
from __future__ import annotations

import numpy as np

NEG_INF = -np.inf


def to_f64(x) -> np.ndarray:
    """Exact widening of a (bf16/fp32/...) torch tensor or array to fp64 numpy."""
    try:
        import torch

        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu").to(torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


def valid_key_mask(n_q: int, n_k: int, causal: bool, kv_len: int | None = None,
                   rows=None) -> np.ndarray:
    """Boolean [len(rows), n_k]: True where key j is visible to query row i."""
    rows = np.arange(n_q) if rows is None else np.asarray(rows)
    j = np.arange(n_k)[None, :]
    m = np.ones((len(rows), n_k), dtype=bool)
    if causal:
        m &= j <= rows[:, None]
    if kv_len is not None:
        m &= j < int(kv_len)
    return m


def _softmax_rows(S: np.ndarray, mask: np.ndarray):
    """Row softmax over the masked-in entries of S ([FA-notes] §2.1, step 2).

    Returns P (0 where masked), row max m and row sum l = sum exp(S - m).
    Rows without any valid key get P = 0, m = -inf, l = 0.
    """
    Sm = np.where(mask, S, NEG_INF)
    m = Sm.max(axis=1)
    has = np.isfinite(m)
    m_safe = np.where(has, m, 0.0)
    E = np.where(mask, np.exp(Sm - m_safe[:, None]), 0.0)
    l = E.sum(axis=1)
    P = np.divide(E, l[:, None], out=np.zeros_like(E), where=l[:, None] > 0)
    return P, m, l


def _head_iter(B, H):
    for b in range(B):
        for h in range(H):
            yield b, h


def attention_probs(Q, K, causal=False, scale=None, kv_lens=None):
    """Materialised P = softmax(scale * Q K^T) per (b, h): [B, H, N, N] fp64.

    [FA-notes] §2.1 (standard attention, steps 1-2).
    """
    Q, K = to_f64(Q), to_f64(K)
    B, H, N, d = Q.shape
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    out = np.zeros((B, H, N, K.shape[2]))
    for b, h in _head_iter(B, H):
        L = None if kv_lens is None else int(kv_lens[b])
        S = scale * (Q[b, h] @ K[b, h].T)
        P, _, _ = _softmax_rows(S, valid_key_mask(N, K.shape[2], causal, L))
        out[b, h] = P
    return out


def attention_forward_rows(Q, K, V, rows, causal=False, scale=None, kv_lens=None,
                           heads=None):
    """O and LSE for the selected query ``rows`` of the selected ``heads``.

    Each row is the standard-attention definition ([FA-notes] §2.1) evaluated
    for that row alone; used where the full N x N matrix does not fit.
    Returns O [len(heads), len(rows), d], LSE [len(heads), len(rows)].
    """
    Q, K, V = to_f64(Q), to_f64(K), to_f64(V)
    B, H, N, d = Q.shape
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    rows = np.asarray(rows)
    heads = [(b, h) for b, h in _head_iter(B, H)] if heads is None else list(heads)
    O = np.zeros((len(heads), len(rows), V.shape[3]))
    LSE = np.zeros((len(heads), len(rows)))
    for t, (b, h) in enumerate(heads):
        L = None if kv_lens is None else int(kv_lens[b])
        S = scale * (Q[b, h][rows] @ K[b, h].T)
        P, m, l = _softmax_rows(S, valid_key_mask(N, K.shape[2], causal, L, rows=rows))
        O[t] = P @ V[b, h]
        with np.errstate(divide="ignore"):
            LSE[t] = np.where(l > 0, m + np.log(np.where(l > 0, l, 1.0)), NEG_INF)
    return O, LSE


def attention_forward(Q, K, V, causal=False, scale=None, kv_lens=None, row_chunk=2048):
    """Standard attention forward: O [B,H,N,d] and LSE [B,H,N] in fp64.

    [FA-notes] §2.1: S = QK^T (times ``scale``), P = softmax(S), O = PV;
    LSE_i = m_i + ln l_i keeps the row statistics of [FA-notes] §3.3.
    Rows are evaluated in chunks of ``row_chunk`` only to bound memory; every
    row's arithmetic is the plain definition.
    """
    Q, K, V = to_f64(Q), to_f64(K), to_f64(V)
    B, H, N, d = Q.shape
    O = np.zeros((B, H, N, V.shape[3]))
    LSE = np.zeros((B, H, N))
    for b, h in _head_iter(B, H):
        for r0 in range(0, N, row_chunk):
            rows = np.arange(r0, min(N, r0 + row_chunk))
            o, lse = attention_forward_rows(Q, K, V, rows, causal, scale, kv_lens, heads=[(b, h)])
            O[b, h, rows] = o[0]
            LSE[b, h, rows] = lse[0]
    return O, LSE


def attention_backward(Q, K, V, dO, causal=False, scale=None, kv_lens=None,
                       return_aux=False):
    """Analytic gradient of sum(dO * O) for O = softmax(scale Q K^T) V.

    The pages prescribe recomputing S and P from O and (m, l) instead of
    storing them ([FA-notes] §3.3; [IO-explained], recomputation) but print no
    formulas; this is the plain derivation by the chain rule:
        dV = P^T dO,   dP = dO V^T,   D_i = sum_j P_ij dP_ij (= sum_c dO_ic O_ic),
        dS = P * (dP - D),   dQ = scale * dS K,   dK = scale * dS^T Q.
    Masked entries have P = 0 and contribute nothing.
    """
    Q, K, V, dO = to_f64(Q), to_f64(K), to_f64(V), to_f64(dO)
    B, H, N, d = Q.shape
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    dQ = np.zeros_like(Q)
    dK = np.zeros_like(K)
    dV = np.zeros_like(V)
    Dall = np.zeros((B, H, N))
    for b, h in _head_iter(B, H):
        L = None if kv_lens is None else int(kv_lens[b])
        S = scale * (Q[b, h] @ K[b, h].T)
        P, _, _ = _softmax_rows(S, valid_key_mask(N, K.shape[2], causal, L))
        dV[b, h] = P.T @ dO[b, h]
        dP = dO[b, h] @ V[b, h].T
        D = (P * dP).sum(axis=1)
        dS = P * (dP - D[:, None])
        dQ[b, h] = scale * (dS @ K[b, h])
        dK[b, h] = scale * (dS.T @ Q[b, h])
        Dall[b, h] = D
    if return_aux:
        return dQ, dK, dV, Dall
    return dQ, dK, dV


def attention_backward_rows(Q, K, V, dO, rows, causal=False, scale=None, kv_lens=None, heads=None):
    """The backward restricted to the selected query ``rows``: the same chain
    rule as ``attention_backward``, evaluated for those rows alone.

    Returns dQ of the rows [len(heads), len(rows), d] and the rows' share of
    dK and dV [len(heads), N_k, d] (the sum over the selected rows of
    scale * dS_ij Q_i and P_ij dO_i).  Summing the shares over a partition of
    all rows gives ``attention_backward``'s dK and dV.  D_i is taken as
    sum_j P_ij dP_ij, which equals rowsum(dO_i * O_i).
    """
    Q, K, V, dO = to_f64(Q), to_f64(K), to_f64(V), to_f64(dO)
    B, H, N, d = Q.shape
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    rows = np.asarray(rows)
    heads = [(b, h) for b, h in _head_iter(B, H)] if heads is None else list(heads)
    n_k = K.shape[2]
    dQ = np.zeros((len(heads), len(rows), d))
    dK = np.zeros((len(heads), n_k, d))
    dV = np.zeros((len(heads), n_k, V.shape[3]))
    for t, (b, h) in enumerate(heads):
        L = None if kv_lens is None else int(kv_lens[b])
        S = scale * (Q[b, h][rows] @ K[b, h].T)
        P, _, _ = _softmax_rows(S, valid_key_mask(N, n_k, causal, L, rows=rows))
        dP = dO[b, h][rows] @ V[b, h].T
        D = (P * dP).sum(axis=1)
        dS = P * (dP - D[:, None])
        dQ[t] = scale * (dS @ K[b, h])
        dK[t] = scale * (dS.T @ Q[b, h][rows])
        dV[t] = P.T @ dO[b, h][rows]
    return dQ, dK, dV


def streaming_row_forward(q, K, V, tile, scale, key_mask=None, nan_guard=True):
    """One query row by the online-softmax loop of [S12] ("核心思路"):
    running max m, running sum l, unnormalised accumulator o; each key tile
    updates m_new = max(m, max s), alpha = exp(m - m_new), p = exp(s - m_new),
    l = alpha l + sum p, o = alpha o + p V; the result is o / l.

    ``key_mask`` (bool [n_k]) drops keys by setting their logit to -inf, as the
    masked variant of [S12] exercise 2 does.  With ``nan_guard`` a tile whose
    running max is still -inf subtracts 0 instead (the fix [S12] asks for
    after "exp(-inf - -inf) 是 NaN"); without it the hazard is reproduced.
    Returns (o / l, m, l); an empty row returns (0, -inf, 0) when guarded.
    """
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    n_k = K.shape[0]
    m, l = NEG_INF, 0.0
    o = np.zeros(V.shape[1])
    for start in range(0, n_k, tile):
        stop = min(n_k, start + tile)
        s = scale * (K[start:stop] @ q)
        if key_mask is not None:
            s = np.where(key_mask[start:stop], s, NEG_INF)
        m_new = max(m, s.max())
        sub = 0.0 if (nan_guard and m_new == NEG_INF) else m_new
        with np.errstate(invalid="ignore"):
            alpha = np.exp(m - sub)
            p = np.exp(s - sub)
        l = alpha * l + p.sum()
        o = alpha * o + p @ V[start:stop]
        m = m_new
    if nan_guard and l == 0.0:
        return np.zeros_like(o), m, l
    with np.errstate(invalid="ignore", divide="ignore"):
        return o / l, m, l


def algorithm1_forward(Q, K, V, Br, Bc, scale=1.0, causal=False):
    """[FA-notes] §3.2 Algorithm 1 for one head, in its own loop order:
    K/V blocks outer (j), Q blocks inner (i); O, l, m kept "in HBM" (arrays
    here) and updated after every (i, j) with the per-step normalisation
        m_new = max(m_i, m~_ij),
        l_new = e^{m_i - m_new} l_i + e^{m~_ij - m_new} l~_ij,
        O_i   = diag(l_new)^{-1} [diag(l_i) e^{m_i - m_new} O_i
                                  + e^{m~_ij - m_new} P~_ij V_j].
    The printed algorithm has no scale (scale = 1); ``scale`` multiplies S.
    Causal masking (j > i -> -inf) is an addition for the exercise; a fully
    masked (i, j) block is skipped so no exp(-inf - -inf) arises.
    Returns O [N, d], l [N], m [N].
    """
    Q, K, V = (np.asarray(x, dtype=np.float64) for x in (Q, K, V))
    N, d = Q.shape
    O = np.zeros((N, V.shape[1]))
    l = np.zeros(N)
    m = np.full(N, NEG_INF)
    for c0 in range(0, K.shape[0], Bc):
        Kj, Vj = K[c0:c0 + Bc], V[c0:c0 + Bc]
        cols = np.arange(c0, c0 + Kj.shape[0])
        for r0 in range(0, N, Br):
            rows = np.arange(r0, min(N, r0 + Br))
            S = scale * (Q[rows] @ Kj.T)
            if causal:
                S = np.where(cols[None, :] <= rows[:, None], S, NEG_INF)
            mt = S.max(axis=1)
            live = np.isfinite(mt)
            if not live.any():
                continue
            r = rows[live]
            S, mt = S[live], mt[live]
            Pt = np.exp(S - mt[:, None])
            lt = Pt.sum(axis=1)
            m_new = np.maximum(m[r], mt)
            a_old = np.exp(m[r] - m_new)
            a_new = np.exp(mt - m_new)
            l_new = a_old * l[r] + a_new * lt
            O[r] = ((l[r] * a_old)[:, None] * O[r] + a_new[:, None] * (Pt @ Vj)) / l_new[:, None]
            l[r] = l_new
            m[r] = m_new
    return O, l, m


def merge_states(ms, ls, os_):
    """Merge partial softmax states (m_s, l_s, o_s) over the leading axis.

    [FA-notes] §3.1 merge rule m = max_s m_s, l = sum_s e^{m_s - m} l_s,
    applied to the unnormalised accumulators o as well ([S12] flash-decoding:
    "the merge rule is the rescale you already wrote").  States with
    l_s = 0 (empty splits) are skipped.  Returns (o / l, m, l).
    """
    ms = np.asarray(ms, dtype=np.float64)
    ls = np.asarray(ls, dtype=np.float64)
    os_ = np.asarray(os_, dtype=np.float64)
    keep = ls > 0
    if not keep.any():
        return np.zeros(os_.shape[1:]), NEG_INF, 0.0
    ms, ls, os_ = ms[keep], ls[keep], os_[keep]
    m = ms.max()
    w = np.exp(ms - m)
    l = (w * ls).sum()
    o = (w[:, None] * os_).sum(axis=0)
    return o / l, m, l


def attention_forward_varlen(Q, K, V, cu_seqlens, causal=False, scale=None):
    """Attention over a packed ragged batch: Q, K, V are [total, H, d] with
    sequence s occupying rows cu_seqlens[s] .. cu_seqlens[s+1]-1; every
    sequence is an independent attention problem ([FA-notes] §2.1 applied per
    sequence; causal masking is top-left within each sequence).
    Returns O [total, H, d] and LSE [H, total]."""
    Q, K, V = to_f64(Q), to_f64(K), to_f64(V)
    cu = np.asarray(cu_seqlens.cpu().numpy() if hasattr(cu_seqlens, "cpu") else cu_seqlens, dtype=np.int64)
    total, H, d = Q.shape
    O = np.zeros((total, H, V.shape[2]))
    LSE = np.full((H, total), NEG_INF)
    for s in range(len(cu) - 1):
        a, b = int(cu[s]), int(cu[s + 1])
        if b <= a:
            continue
        # [L, H, d] -> [1, H, L, d]
        q, k, v = (x[a:b].transpose(1, 0, 2)[None] for x in (Q, K, V))
        o, lse = attention_forward(q, k, v, causal=causal, scale=scale)
        O[a:b] = o[0].transpose(1, 0, 2)
        LSE[:, a:b] = lse[0]
    return O, LSE


def attention_backward_varlen(Q, K, V, dO, cu_seqlens, causal=False, scale=None):
    """Gradients of sum(dO * O) for the packed ragged batch of
    attention_forward_varlen: attention_backward applied to each sequence
    (sequences do not interact).  Q, K, V, dO [total, H, d] -> dQ, dK, dV."""
    Q, K, V, dO = to_f64(Q), to_f64(K), to_f64(V), to_f64(dO)
    cu = np.asarray(cu_seqlens.cpu().numpy() if hasattr(cu_seqlens, "cpu") else cu_seqlens, dtype=np.int64)
    dQ, dK, dV = np.zeros_like(Q), np.zeros_like(K), np.zeros_like(V)
    for s in range(len(cu) - 1):
        a, b = int(cu[s]), int(cu[s + 1])
        if b <= a:
            continue
        q, k, v, g = (x[a:b].transpose(1, 0, 2)[None] for x in (Q, K, V, dO))
        gq, gk, gv = attention_backward(q, k, v, g, causal=causal, scale=scale)
        dQ[a:b], dK[a:b], dV[a:b] = (x[0].transpose(1, 0, 2) for x in (gq, gk, gv))
    return dQ, dK, dV
