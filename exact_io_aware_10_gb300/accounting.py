"""Algorithmic FLOP and byte counts used for throughput and roofline figures.

Conventions (matmul work only; exp, masking and reductions are not counted):
  forward   4 * B * H * N^2 * d     (QK^T and PV, 2 N^2 d each), halved when causal
  backward  2.5 x the forward       (five N^2 d products instead of two)
  key padding: the effective forward count is 4 * H * N * d * sum_b L_b
  packed ragged batch: the sum of the forward count of every sequence,
            4 * H * d * sum_s L_s^2, halved when causal
  block-sparse: 4 * H * d per visible (query, key) pair of the kept blocks
            (counted per block: the pairs of a block that lie inside N and,
            when causal, on or below the diagonal)
  paged chunked prefill: 4 * Hq * d per visible (query, key) pair, counted
            exactly: a causal chunk of q rows after a prefix of p keys has
            q * p + q (q + 1) / 2 pairs; non-causal q * (p + q)
  decode    bytes = K and V of every visible key, read once per KV head
            (sum_b L_b * Hkv * d * 2 B * 2) + q + o + lse + the block-table
            entries and sequence lengths read.
Compulsory forward bytes are Q, K, V, O (2 B each) + LSE (4 B); backward bytes
are Q, K, V, O, dO, dQ, dK, dV (2 B each) + LSE and D = rowsum(dO * O) (4 B
each per row).
"""
from __future__ import annotations


def fwd_flops(B, H, N, d, causal=False):
    f = 4.0 * B * H * N * N * d
    return f * 0.5 if causal else f


def bwd_flops(B, H, N, d, causal=False):
    return 2.5 * fwd_flops(B, H, N, d, causal)


def fwd_flops_padded(H, N, d, kv_lens):
    return 4.0 * H * N * d * float(sum(int(x) for x in kv_lens))


def varlen_fwd_flops(lengths, H, d, causal=False):
    return sum(fwd_flops(1, H, int(n), d, causal) for n in lengths)


def paged_prefill_flops(q_lens, kv_lens, Hq, d, causal=True):
    pairs = 0
    for q, k in zip(q_lens, kv_lens):
        q, k = int(q), int(k)
        if not causal:
            pairs += q * k
            continue
        for_rows = 0
        p = k - q  # keys before the chunk's first query (negative: rows with no key)
        if p >= 0:
            for_rows = q * p + q * (q + 1) // 2
        else:
            r = q + p  # rows that see at least one key: r rows seeing 1..r keys
            for_rows = max(r, 0) * (max(r, 0) + 1) // 2
        pairs += for_rows
    return 4.0 * Hq * d * pairs


def block_sparse_flops(block_mask, B, H, N, d, causal=True, block=128):
    """block_mask: [nb, nb] (shared) or [B, H, nb, nb] array-like of 0/1."""
    import numpy as np

    m = np.asarray(block_mask).astype(bool)
    nb = m.shape[-1]
    qi = np.arange(nb)
    rows = np.minimum(block, N - qi * block)  # valid rows (and keys) per block
    pairs = rows[:, None] * rows[None, :]
    if causal:
        diag = rows * (rows + 1) // 2
        pairs = np.where(qi[:, None] > qi[None, :], pairs, 0)
        pairs[qi, qi] = diag
    per_mask = (m * pairs).reshape(-1, nb, nb).sum(axis=(1, 2))
    total = per_mask.sum() * (B * H if m.ndim == 2 else 1)
    return 4.0 * d * float(total)


def fwd_bytes(B, H, N, d):
    return 8.0 * B * H * N * d + 4.0 * B * H * N


def bwd_bytes(B, H, N, d):
    # Q, K, V, O, dO read and dQ, dK, dV written (bf16), LSE and D (fp32) --
    # compulsory only
    return 2.0 * B * H * N * d * 8 + 8.0 * B * H * N


def decode_bytes(seq_lens, Hq, Hkv, d, block_size=16, with_lse=True):
    L = [int(x) for x in seq_lens]
    B = len(L)
    kv = sum(L) * Hkv * d * 2.0 * 2
    qo = 2.0 * B * Hq * d * 2
    lse = 4.0 * B * Hq if with_lse else 0.0
    table = 4.0 * sum((x + block_size - 1) // block_size for x in L) + 4.0 * B
    return kv + qo + lse + table
