"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module draws random numbers and lays them out; it holds none of the
attention arithmetic.  Every tensor is produced on the CPU with a seeded
``torch.Generator`` (values drawn in fp32, rounded to bf16 round-to-nearest-even),
so both sides read bit-identical inputs.

Workload recipes (shapes follow the attention configurations this library is
measured on; the pages' benchmark suites -- MLPerf BERT-large, OpenWebText GPT-2,
Long Range Arena -- are stood in for by these synthetic tensors):

* ``dense``      Q, K, V, dO ~ N(0, std^2), layout [B, H, N, d].
* ``padded``     ``dense`` plus per-sequence key lengths L_b ~ U{lo..hi}.
* ``boosted``    ``dense`` with std 0.5 plus a max-shift stressor: per (b, h) a
                 random unit direction u; each Q row and each K row is picked
                 with probability 0.1 and gets c*u added, c = sqrt(8*sqrt(d)),
                 so about 1% of (query, key) pairs gain ~+8 in scaled logit.
* ``varlen``     a packed ragged batch: sequence lengths L_s ~ U{lo..hi}
                 (or given), Q, K, V, dO ~ N(0, std^2) in layout [total, H, d]
                 with sequence s in rows cu_seqlens[s] .. cu_seqlens[s+1]-1.
* ``paged_prefill``  query chunks of lengths q_len_b packed [total_q, Hq, d]
                 (cu_seqlens_q) over a ``paged`` cache whose sequences hold
                 kv_len_b >= q_len_b tokens (cached prefix + the chunk).
* ``block_mask`` 0/1 masks over 128 x 128 score blocks: ``butterfly`` keeps
                 block (i, j) when i == j or i XOR j is a power of two (the
                 fixed butterfly pattern family block-sparse FlashAttention
                 was measured with) plus the w nearest key blocks before i;
                 ``random`` keeps each block with probability p (diagonal
                 always kept).
* ``paged``      decode queries [B, Hq, d], a paged KV cache
                 [num_blocks, block_size, Hkv, d], context lengths
                 L_b ~ U{lo..hi}, and a block table whose physical ids are a
                 seeded random permutation (entries past a row's blocks are -1).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

__all__ = [
    "AttentionInputs",
    "PagedInputs",
    "dense_inputs",
    "padded_lengths",
    "boosted_inputs",
    "paged_inputs",
    "block_mask",
    "VarlenInputs",
    "PagedPrefillInputs",
    "paged_prefill_inputs",
    "varlen_lengths",
    "varlen_inputs",
    "paged_layout",
    "device_normal_bf16",
    "config_seed",
]


def config_seed(seed: int, config_id: int) -> int:
    """Per-configuration RNG stream id derived from (seed, config id)."""
    return int(seed) * 1_000_003 + int(config_id) * 7919 + 17


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def _normal_bf16(shape, g, std=1.0):
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        x = x * std
    return x.to(torch.bfloat16)


@dataclass
class AttentionInputs:
    Q: torch.Tensor  # [B, H, N, d] bf16 (CPU)
    K: torch.Tensor
    V: torch.Tensor
    dO: torch.Tensor
    kv_lens: torch.Tensor | None  # int32 [B] or None

    @property
    def shape(self):
        return tuple(self.Q.shape)


def dense_inputs(B, H, N, d, seed=0, std=1.0, kv_lens=None) -> AttentionInputs:
    """Q, K, V, dO i.i.d. N(0, std^2) rounded to bf16, layout [B, H, N, d]."""
    g = _gen(seed)
    Q = _normal_bf16((B, H, N, d), g, std)
    K = _normal_bf16((B, H, N, d), g, std)
    V = _normal_bf16((B, H, N, d), g, std)
    dO = _normal_bf16((B, H, N, d), g, 1.0)
    return AttentionInputs(Q, K, V, dO, kv_lens)


def padded_lengths(B, lo, hi, seed=0) -> torch.Tensor:
    """Per-sequence valid key lengths, uniform integers in [lo, hi], int32 [B]."""
    g = _gen(seed + 101)
    return torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int64).to(torch.int32)


@dataclass
class VarlenInputs:
    Q: torch.Tensor  # [total, H, d] bf16 (CPU)
    K: torch.Tensor
    V: torch.Tensor
    dO: torch.Tensor
    cu_seqlens: torch.Tensor  # int32 [num_seqs + 1], starts at 0, ends at total
    max_seqlen: int

    @property
    def lengths(self):
        return (self.cu_seqlens[1:] - self.cu_seqlens[:-1]).tolist()


def varlen_lengths(num_seqs, lo, hi, seed=0) -> list:
    """Sequence lengths of a ragged batch, uniform integers in [lo, hi]."""
    g = _gen(seed + 211)
    return torch.randint(lo, hi + 1, (num_seqs,), generator=g, dtype=torch.int64).tolist()


def varlen_inputs(lengths, H, d, seed=0, std=1.0) -> VarlenInputs:
    """Packed [total, H, d] Q, K, V, dO for sequences of the given lengths."""
    lengths = [int(x) for x in lengths]
    if any(x < 0 for x in lengths) or not lengths:
        raise ValueError("lengths must be a non-empty list of non-negative ints")
    cu = torch.zeros(len(lengths) + 1, dtype=torch.int64)
    cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0)
    total = int(cu[-1])
    g = _gen(seed)
    Q = _normal_bf16((total, H, d), g, std)
    K = _normal_bf16((total, H, d), g, std)
    V = _normal_bf16((total, H, d), g, std)
    dO = _normal_bf16((total, H, d), g, 1.0)
    return VarlenInputs(Q, K, V, dO, cu.to(torch.int32), max(lengths))


def boosted_inputs(B, H, N, d, seed=0, std=0.5, pick_prob=0.1, boost=8.0) -> AttentionInputs:
    """``dense`` inputs (std 0.5) with ~1% of (q, k) pairs boosted by ~``boost``
    in scaled logit, to exercise max-shift rescaling in a streaming softmax."""
    g = _gen(seed)
    Qf = torch.randn(B, H, N, d, generator=g, dtype=torch.float32) * std
    Kf = torch.randn(B, H, N, d, generator=g, dtype=torch.float32) * std
    V = _normal_bf16((B, H, N, d), g, std)
    dO = _normal_bf16((B, H, N, d), g, 1.0)
    u = torch.randn(B, H, 1, d, generator=g, dtype=torch.float32)
    u = u / u.norm(dim=-1, keepdim=True)
    c = math.sqrt(boost * math.sqrt(d))
    qpick = (torch.rand(B, H, N, 1, generator=g) < pick_prob).to(torch.float32)
    kpick = (torch.rand(B, H, N, 1, generator=g) < pick_prob).to(torch.float32)
    Q = (Qf + qpick * c * u).to(torch.bfloat16)
    K = (Kf + kpick * c * u).to(torch.bfloat16)
    return AttentionInputs(Q, K, V, dO, None)


@dataclass
class PagedInputs:
    q: torch.Tensor            # [B, Hq, d] bf16
    k_cache: torch.Tensor      # [num_blocks, block_size, Hkv, d] bf16
    v_cache: torch.Tensor      # [num_blocks, block_size, Hkv, d] bf16
    block_table: torch.Tensor  # [B, max_blocks] int32, -1 past each row's blocks
    seq_lens: torch.Tensor     # [B] int32
    block_size: int

    @property
    def num_blocks(self):
        return int(self.k_cache.shape[0])

    @property
    def max_blocks(self):
        return int(self.block_table.shape[1])


def paged_layout(B, L_lo, L_hi, block_size=16, seed=0, max_blocks=None, seq_lens=None, spare_blocks=0,
                 g=None):
    """Context lengths and block table of a paged KV cache (CPU int32).

    L_b ~ U{L_lo..L_hi} unless ``seq_lens`` is given; physical block ids are a
    seeded random permutation of [0, NB), NB = sum_b ceil(L_b / block_size)
    (+ ``spare_blocks`` never referenced); entries past a row's blocks are -1.
    Returns (seq_lens, block_table, NB, generator).
    """
    g = _gen(seed) if g is None else g
    if seq_lens is None:
        seq_lens = torch.randint(L_lo, L_hi + 1, (B,), generator=g, dtype=torch.int64)
    seq_lens = torch.as_tensor(seq_lens, dtype=torch.int64).reshape(-1)
    B = int(seq_lens.numel())
    nblk = [(int(L) + block_size - 1) // block_size for L in seq_lens.tolist()]
    NB = sum(nblk) + int(spare_blocks)
    if max_blocks is None:
        max_blocks = max(1, max(nblk) if nblk else 1)
    perm = torch.randperm(NB, generator=g).to(torch.int32)
    table = torch.full((B, max_blocks), -1, dtype=torch.int32)
    pos = 0
    for b, n in enumerate(nblk):
        table[b, :n] = perm[pos:pos + n]
        pos += n
    return seq_lens.to(torch.int32), table, NB, g


def paged_inputs(B, Hq, Hkv, d, L_lo, L_hi, block_size=16, seed=0, max_blocks=None,
                 seq_lens=None, std=1.0, spare_blocks=0) -> PagedInputs:
    """Paged decode inputs on the CPU (layout from ``paged_layout``; q and the
    K/V caches ~ N(0, std^2) in bf16)."""
    seq_lens, table, NB, g = paged_layout(B, L_lo, L_hi, block_size, seed, max_blocks, seq_lens, spare_blocks)
    B = int(seq_lens.numel())
    q = _normal_bf16((B, Hq, d), g, std)
    k_cache = _normal_bf16((max(NB, 1), block_size, Hkv, d), g, std)
    v_cache = _normal_bf16((max(NB, 1), block_size, Hkv, d), g, std)
    return PagedInputs(q, k_cache, v_cache, table, seq_lens, block_size)


@dataclass
class PagedPrefillInputs:
    q: torch.Tensor  # [total_q, Hq, d] bf16 (CPU)
    k_cache: torch.Tensor  # [num_blocks, block_size, Hkv, d] bf16
    v_cache: torch.Tensor
    block_table: torch.Tensor  # int32 [B, max_blocks], -1 past a sequence's blocks
    cu_seqlens_q: torch.Tensor  # int32 [B + 1]
    seq_lens_k: torch.Tensor  # int32 [B]
    block_size: int

    @property
    def q_lens(self):
        return (self.cu_seqlens_q[1:] - self.cu_seqlens_q[:-1]).tolist()

    @property
    def max_seqlen_q(self):
        return max(self.q_lens)


def paged_prefill_inputs(q_lens, kv_lens, Hq, Hkv, d, block_size=16, seed=0, std=1.0, max_blocks=None,
                         spare_blocks=0) -> PagedPrefillInputs:
    """Chunked-prefill inputs on the CPU: a ``paged_layout`` cache for context
    lengths kv_lens, and packed query chunks of lengths q_lens."""
    q_lens = [int(x) for x in q_lens]
    if len(q_lens) != len(kv_lens) or not q_lens or min(q_lens) < 0:
        raise ValueError("q_lens and kv_lens must be equal-length lists of non-negative ints")
    seq_lens, table, NB, g = paged_layout(len(q_lens), 0, 0, block_size, seed, max_blocks, list(kv_lens),
                                          spare_blocks)
    cu = torch.zeros(len(q_lens) + 1, dtype=torch.int64)
    cu[1:] = torch.cumsum(torch.tensor(q_lens, dtype=torch.int64), 0)
    q = _normal_bf16((int(cu[-1]), Hq, d), g, std)
    k_cache = _normal_bf16((max(NB, 1), block_size, Hkv, d), g, std)
    v_cache = _normal_bf16((max(NB, 1), block_size, Hkv, d), g, std)
    return PagedPrefillInputs(q, k_cache, v_cache, table, cu.to(torch.int32), seq_lens, block_size)


def block_mask(nb, pattern="butterfly", window=2, p=0.25, seed=0, heads=None) -> torch.Tensor:
    """uint8 block mask [nb, nb] (or [*heads, nb, nb] for per-head random masks)."""
    if pattern == "butterfly":
        i = torch.arange(nb)[:, None]
        j = torch.arange(nb)[None, :]
        x = i ^ j
        keep = (x == 0) | ((x & (x - 1)) == 0) | ((i - j >= 0) & (i - j <= window))
        return keep.to(torch.uint8)
    if pattern == "random":
        g = _gen(seed + 307)
        shape = (nb, nb) if heads is None else (*heads, nb, nb)
        keep = torch.rand(shape, generator=g) < p
        keep[..., torch.arange(nb), torch.arange(nb)] = True
        return keep.to(torch.uint8)
    raise ValueError(f"unknown pattern {pattern!r}")


def device_normal_bf16(shape, seed, device, std=1.0):
    """N(0, std^2) bf16 tensor drawn on the device with a seeded generator
    (benchmark-sized inputs that would be slow to draw on the host)."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)
