"""fp64 oracle for paged (chunked) prefill: a packed batch of query chunks
attending to the keys and values of a paged KV cache.  Test infrastructure
only (see the package docstring).

Sources:
  [S12] "除了快，它还解锁了什么", PagedAttention bullet: because the kernel
        already streams over key tiles, the tiles need not be contiguous; each
        can be fetched through the block table.  "实现": key t of a sequence
        lives at cache[block_table[t // block_size], t % block_size].
  [S12] grouped-query heads: a group of query heads shares one KV head.

Readings where the pages leave the step open (each is listed with the other
readings of the pages):
  * A chunk of q_len queries is the LAST q_len tokens of a sequence whose
    context (cached prefix + the chunk itself) has kv_len tokens, so query i
    of the chunk sits at absolute position kv_len - q_len + i.  Causal masking
    is therefore bottom-right aligned: key j is visible to query i when
    j <= kv_len - q_len + i.  With q_len = kv_len this is the square,
    top-left causal mask of plain attention; with q_len = 1 it is decode.
  * If q_len > kv_len the first rows see no key at all; such a row returns
    O_i = 0 and LSE_i = -inf, as every empty row does.
  * Query head h reads KV head h // (Hq // Hkv), as in decode.

Layouts: q [total_q, Hq, d] with chunk b in rows cu_seqlens_q[b] ..
cu_seqlens_q[b+1]-1; k_cache / v_cache [num_blocks, block_size, Hkv, d];
block_table int32 [B, max_blocks]; seq_lens_k int32 [B] (kv_len of each
sequence).  Returns O [total_q, Hq, d] and LSE [Hq, total_q] (natural log).
"""
from __future__ import annotations

import numpy as np

from .attention import NEG_INF, to_f64
from .decode import gather_paged_keys


def _np_int(x):
    return np.asarray(x.cpu().numpy() if hasattr(x, "cpu") else x, dtype=np.int64)


def chunk_key_mask(q_len: int, kv_len: int, causal: bool) -> np.ndarray:
    """Boolean [q_len, kv_len]: key j visible to chunk query i (the
    bottom-right causal reading above; all keys when not causal)."""
    i = np.arange(q_len)[:, None]
    j = np.arange(kv_len)[None, :]
    m = np.ones((q_len, kv_len), dtype=bool)
    if causal:
        m &= j <= (kv_len - q_len) + i
    return m


def paged_prefill(q, k_cache, v_cache, block_table, cu_seqlens_q, seq_lens_k, block_size,
                  causal=True, scale=None):
    """Attention of each chunk's queries over its sequence's gathered keys, by
    the plain definition: S = scale * q K^T, a softmax over each row's visible
    keys, O = P V."""
    q = to_f64(q)
    kc, vc = to_f64(k_cache), to_f64(v_cache)
    bt, cu, sl = _np_int(block_table), _np_int(cu_seqlens_q), _np_int(seq_lens_k)
    total_q, Hq, d = q.shape
    Hkv = kc.shape[2]
    grp = Hq // Hkv
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    O = np.zeros((total_q, Hq, vc.shape[3]))
    LSE = np.full((Hq, total_q), NEG_INF)
    for b in range(len(cu) - 1):
        a, e = int(cu[b]), int(cu[b + 1])
        q_len, kv_len = e - a, int(sl[b])
        if q_len <= 0 or kv_len <= 0:
            continue
        mask = chunk_key_mask(q_len, kv_len, causal)
        for h in range(Hq):
            g = h // grp
            Kb = gather_paged_keys(kc, bt[b], kv_len, block_size, g)
            Vb = gather_paged_keys(vc, bt[b], kv_len, block_size, g)
            S = scale * (q[a:e, h] @ Kb.T)
            for i in range(q_len):
                vis = mask[i]
                if not vis.any():
                    continue
                s = S[i, vis]
                m = s.max()
                w = np.exp(s - m)
                l = w.sum()
                O[a + i, h] = (w @ Vb[vis]) / l
                LSE[h, a + i] = m + np.log(l)
    return O, LSE


def paged_prefill_rows(q, k_cache, v_cache, block_table, cu_seqlens_q, seq_lens_k, block_size, b, rows,
                       heads, causal=True, scale=None):
    """O [len(heads), len(rows), d] and LSE [len(heads), len(rows)] of chunk
    b's query ``rows`` for the given query heads: the same definition as
    paged_prefill, evaluated only where the full problem is too large."""
    bt, cu, sl = _np_int(block_table), _np_int(cu_seqlens_q), _np_int(seq_lens_k)
    a, e = int(cu[b]), int(cu[b + 1])
    q_len, kv_len = e - a, int(sl[b])
    d = q.shape[2]
    Hq, Hkv = q.shape[1], k_cache.shape[2]
    grp = Hq // Hkv
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    rows = np.asarray(rows)
    mask = chunk_key_mask(q_len, kv_len, causal)[rows]
    O = np.zeros((len(heads), len(rows), v_cache.shape[3]))
    LSE = np.full((len(heads), len(rows)), NEG_INF)
    # the same block-table gather as gather_paged_keys, done before widening
    # so that only this sequence's rows are converted to fp64
    tok = np.arange(kv_len)
    phys = bt[b][tok // block_size]
    for t, h in enumerate(heads):
        g = h // grp
        Kb = to_f64(k_cache[phys, tok % block_size, g])
        Vb = to_f64(v_cache[phys, tok % block_size, g])
        qh = to_f64(q[a:e, h])[rows]
        S = scale * (qh @ Kb.T)
        for r in range(len(rows)):
            vis = mask[r]
            if not vis.any():
                continue
            s = S[r, vis]
            m = s.max()
            w = np.exp(s - m)
            l = w.sum()
            O[t, r] = (w @ Vb[vis]) / l
            LSE[t, r] = m + np.log(l)
    return O, LSE
