"""Pins of the block-sparse oracle against what the page and the mathematics
fix: an all-ones mask is dense attention, a block-diagonal mask is attention
on each block by itself, an empty mask row gives empty rows, torch's fp64
scaled-dot-product attention with the expanded boolean mask (a library
routine), and a scalar brute-force loop."""
import math

import numpy as np
import pytest
import torch

import oracle


def _rand(shape, seed, std=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * std


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("padded", [False, True])
def test_all_ones_mask_is_dense_attention(causal, padded):
    B, H, N, d, blk = 2, 2, 21, 8, 4
    Q, K, V = (_rand((B, H, N, d), s) for s in (1, 2, 3))
    kv = np.array([21, 9]) if padded else None
    nb = -(-N // blk)
    O, L = oracle.block_sparse_forward(Q, K, V, np.ones((nb, nb), np.uint8), causal=causal, kv_lens=kv, block=blk)
    Oref, Lref = oracle.attention_forward(Q, K, V, causal=causal, kv_lens=kv)
    np.testing.assert_allclose(O, Oref, atol=1e-14)
    np.testing.assert_allclose(L, Lref, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_block_diagonal_mask_is_attention_within_each_block(causal):
    B, H, N, d, blk = 1, 2, 20, 4, 5
    Q, K, V = (_rand((B, H, N, d), s) for s in (4, 5, 6))
    nb = N // blk
    O, L = oracle.block_sparse_forward(Q, K, V, np.eye(nb, dtype=np.uint8), causal=causal, block=blk)
    for c in range(nb):
        sl = slice(c * blk, (c + 1) * blk)
        Oc, Lc = oracle.attention_forward(Q[:, :, sl], K[:, :, sl], V[:, :, sl], causal=causal)
        np.testing.assert_allclose(O[:, :, sl], Oc, atol=1e-14)
        np.testing.assert_allclose(L[:, :, sl], Lc, atol=1e-13)


def test_empty_mask_row_gives_empty_rows():
    B, H, N, d, blk = 1, 1, 12, 4, 4
    Q, K, V = (_rand((B, H, N, d), s) for s in (7, 8, 9))
    m = np.ones((3, 3), np.uint8)
    m[1] = 0
    O, L = oracle.block_sparse_forward(Q, K, V, m, block=blk)
    assert np.all(O[0, 0, 4:8] == 0) and np.all(np.isneginf(L[0, 0, 4:8]))
    assert np.all(np.isfinite(L[0, 0, :4])) and np.all(np.isfinite(L[0, 0, 8:]))


@pytest.mark.parametrize("causal", [False, True])
def test_matches_library_attention_with_the_expanded_mask(causal):
    B, H, N, d, blk = 2, 3, 30, 8, 8
    Q, K, V = (_rand((B, H, N, d), s) for s in (10, 11, 12))
    nb = -(-N // blk)
    rng = np.random.default_rng(13)
    m = (rng.random((B, H, nb, nb)) < 0.5).astype(np.uint8)
    m[..., np.arange(nb), np.arange(nb)] = 1  # every row keeps its diagonal block
    O, L = oracle.block_sparse_forward(Q, K, V, m, causal=causal, block=blk)
    allowed = np.stack([np.stack([oracle.expand_block_mask(m[b, h], N, N, blk) for h in range(H)])
                        for b in range(B)])
    if causal:
        allowed &= np.tril(np.ones((N, N), bool))
    t = [torch.from_numpy(x) for x in (Q, K, V)]
    ref = torch.nn.functional.scaled_dot_product_attention(*t, attn_mask=torch.from_numpy(allowed))
    np.testing.assert_allclose(O, ref.numpy(), atol=1e-12)
    S = np.einsum("bhid,bhjd->bhij", Q, K) / math.sqrt(d)
    S = np.where(allowed, S, -np.inf)
    lse = torch.logsumexp(torch.from_numpy(S), dim=-1).numpy()
    np.testing.assert_allclose(L, lse, atol=1e-12)


def test_brute_force_tiny_per_head_mask():
    B, H, N, d, blk, scale = 1, 2, 6, 3, 2, 0.4
    Q, K, V = (_rand((B, H, N, d), s) for s in (14, 15, 16))
    m = np.array([[[[1, 0, 1], [0, 1, 0], [1, 1, 0]], [[0, 0, 1], [1, 0, 0], [0, 1, 1]]]], np.uint8)
    O, L = oracle.block_sparse_forward(Q, K, V, m, causal=True, scale=scale, block=blk)
    for h in range(H):
        for i in range(N):
            keys = [j for j in range(N) if m[0, h, i // blk, j // blk] and j <= i]
            if not keys:
                assert np.all(O[0, h, i] == 0) and np.isneginf(L[0, h, i])
                continue
            lg = [scale * sum(Q[0, h, i, c] * K[0, h, j, c] for c in range(d)) for j in keys]
            mx = max(lg)
            w = [math.exp(x - mx) for x in lg]
            for c in range(d):
                assert abs(O[0, h, i, c] - sum(wk * V[0, h, j, c] for wk, j in zip(w, keys)) / sum(w)) < 1e-13
            assert abs(L[0, h, i] - (mx + math.log(sum(w)))) < 1e-13


def test_row_subset_equals_full():
    B, H, N, d, blk = 1, 1, 16, 4, 4
    Q, K, V = (_rand((B, H, N, d), s) for s in (17, 18, 19))
    m = np.array([[1, 0, 0, 1], [0, 1, 1, 0], [1, 1, 1, 1], [0, 0, 0, 1]], np.uint8)
    O, L = oracle.block_sparse_forward(Q, K, V, m, causal=True, block=blk)
    rows = np.array([0, 5, 11, 15])
    Or, Lr = oracle.block_sparse_forward(Q, K, V, m, causal=True, block=blk, rows=rows)
    np.testing.assert_array_equal(Or, O[:, :, rows])
    np.testing.assert_array_equal(Lr, L[:, :, rows])
