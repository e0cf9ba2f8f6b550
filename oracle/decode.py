"""fp64 oracle for paged, split-KV, grouped-query decode.  Test infrastructure
only (see the package docstring).

[S12] "实现" gives the paged loop: for each logical block t of a sequence,
``physical = block_table[t]``, ``n = min(block_size, seq_len - t*block_size)``
(stop when n <= 0), keys/values are ``cache[physical, :n]``, and the same
online-softmax recurrence runs over them.  [S12] flash-decoding splits the
keys across workers and merges their (m, l, o) states with the same rescale;
grouped-query attention lets each query group share one KV head.

Layouts: q [B, Hq, d]; k_cache / v_cache [num_blocks, block_size, Hkv, d];
block_table int32 [B, max_blocks]; seq_lens int32 [B].  Query head h reads KV
head g = h // (Hq // Hkv) (consecutive query heads share a KV head; the pages
say only that a group shares one head).
"""
from __future__ import annotations

import numpy as np

from .attention import NEG_INF, to_f64, streaming_row_forward, merge_states


def _np_int(x):
    return np.asarray(x.cpu().numpy() if hasattr(x, "cpu") else x, dtype=np.int64)


def gather_paged_keys(cache, block_table_row, seq_len, block_size, g):
    """Keys (or values) t = 0..seq_len-1 of KV head g, gathered through the
    block table: row t lives at cache[block_table[t // bs], t % bs, g, :]."""
    cache = to_f64(cache) if not isinstance(cache, np.ndarray) else cache
    t = np.arange(int(seq_len))
    phys = np.asarray(block_table_row, dtype=np.int64)[t // block_size]
    return cache[phys, t % block_size, g, :]


def paged_decode(q, k_cache, v_cache, block_table, seq_lens, block_size, scale=None):
    """Decode attention by the plain definition: gather the sequence's keys and
    values, then one softmax over all of them.  Returns o [B, Hq, d] and
    lse [B, Hq] (natural log of sum exp of scaled logits); an empty sequence
    gives o = 0, lse = -inf."""
    q = to_f64(q)
    kc, vc = to_f64(k_cache), to_f64(v_cache)
    bt, sl = _np_int(block_table), _np_int(seq_lens)
    B, Hq, d = q.shape
    Hkv = kc.shape[2]
    grp = Hq // Hkv
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    o = np.zeros((B, Hq, vc.shape[3]))
    lse = np.full((B, Hq), NEG_INF)
    for b in range(B):
        L = int(sl[b])
        if L <= 0:
            continue
        for h in range(Hq):
            g = h // grp
            Kb = gather_paged_keys(kc, bt[b], L, block_size, g)
            Vb = gather_paged_keys(vc, bt[b], L, block_size, g)
            s = scale * (Kb @ q[b, h])
            m = s.max()
            e = np.exp(s - m)
            l = e.sum()
            o[b, h] = (e @ Vb) / l
            lse[b, h] = m + np.log(l)
    return o, lse


def paged_decode_streaming(q, k_cache, v_cache, block_table, seq_lens, block_size,
                           scale=None):
    """The [S12] paged loop verbatim in structure: one logical block at a time,
    online softmax across blocks.  Returns o [B, Hq, d]."""
    q = to_f64(q)
    kc, vc = to_f64(k_cache), to_f64(v_cache)
    bt, sl = _np_int(block_table), _np_int(seq_lens)
    B, Hq, d = q.shape
    Hkv = kc.shape[2]
    grp = Hq // Hkv
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    o_out = np.zeros((B, Hq, vc.shape[3]))
    for b in range(B):
        L = int(sl[b])
        for h in range(Hq):
            g = h // grp
            m, l, o = NEG_INF, 0.0, np.zeros(vc.shape[3])
            for logical in range(bt.shape[1]):
                n = min(block_size, L - logical * block_size)
                if n <= 0:
                    break
                phys = bt[b, logical]
                kb = kc[phys, :n, g, :]
                vb = vc[phys, :n, g, :]
                s = scale * (kb @ q[b, h])
                m_new = max(m, s.max())
                alpha = np.exp(m - m_new)
                p = np.exp(s - m_new)
                l, o, m = alpha * l + p.sum(), alpha * o + p @ vb, m_new
            if l > 0:
                o_out[b, h] = o / l
    return o_out


def split_ranges(n_blocks: int, num_splits: int):
    """Contiguous, balanced block ranges [lo, hi) for ``num_splits`` workers
    (some may be empty when n_blocks < num_splits)."""
    return [((s * n_blocks) // num_splits, ((s + 1) * n_blocks) // num_splits)
            for s in range(num_splits)]


def split_paged_decode(q, k_cache, v_cache, block_table, seq_lens, block_size,
                       num_splits, scale=None, return_partials=False):
    """Flash-decoding ([S12], "除了快…" and exercise 1): the logical blocks of a
    sequence are cut into ``num_splits`` contiguous chunks; each chunk runs the
    streaming recurrence independently and yields an unnormalised state
    (m_s, l_s, o_s); the states are merged by ``merge_states``.
    Returns o [B, Hq, d], lse [B, Hq] (and the partials if asked)."""
    q = to_f64(q)
    kc, vc = to_f64(k_cache), to_f64(v_cache)
    bt, sl = _np_int(block_table), _np_int(seq_lens)
    B, Hq, d = q.shape
    Hkv = kc.shape[2]
    dv = vc.shape[3]
    grp = Hq // Hkv
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    o = np.zeros((B, Hq, dv))
    lse = np.full((B, Hq), NEG_INF)
    parts_m = np.full((B, Hq, num_splits), NEG_INF)
    parts_l = np.zeros((B, Hq, num_splits))
    parts_o = np.zeros((B, Hq, num_splits, dv))
    for b in range(B):
        L = int(sl[b])
        nb = (L + block_size - 1) // block_size if L > 0 else 0
        for s, (lo, hi) in enumerate(split_ranges(nb, num_splits)):
            if hi <= lo:
                continue
            t0, t1 = lo * block_size, min(L, hi * block_size)
            for h in range(Hq):
                g = h // grp
                Kb = gather_paged_keys(kc, bt[b], L, block_size, g)[t0:t1]
                Vb = gather_paged_keys(vc, bt[b], L, block_size, g)[t0:t1]
                on, m_s, l_s = streaming_row_forward(q[b, h], Kb, Vb, tile=block_size, scale=scale)
                parts_m[b, h, s] = m_s
                parts_l[b, h, s] = l_s
                parts_o[b, h, s] = on * l_s  # back to the unnormalised accumulator
        for h in range(Hq):
            ob, m, l = merge_states(parts_m[b, h], parts_l[b, h], parts_o[b, h])
            o[b, h] = ob
            lse[b, h] = m + np.log(l) if l > 0 else NEG_INF
    if return_partials:
        return o, lse, (parts_m, parts_l, parts_o)
    return o, lse
