"""The algorithmic FLOP and byte counts behind the reported throughputs,
checked against brute-force counts of the (query, key) pairs each mask
admits, so a miscount cannot inflate a TFLOP/s figure."""
import numpy as np
import pytest

import oracle
from exact_io_aware_10_gb300 import accounting as acc


def _pairs(mask):
    return int(np.count_nonzero(mask))


@pytest.mark.parametrize("N", [1, 7, 64])
def test_dense_forward_counts(N):
    # 4 d flops per (query, key) pair; causal is counted as half the square
    H, d = 3, 8
    assert acc.fwd_flops(2, H, N, d, False) == 4 * d * 2 * H * _pairs(oracle.valid_key_mask(N, N, False))
    assert acc.fwd_flops(2, H, N, d, True) == 0.5 * acc.fwd_flops(2, H, N, d, False)
    assert acc.bwd_flops(2, H, N, d, True) == 2.5 * acc.fwd_flops(2, H, N, d, True)


def test_varlen_counts_are_per_sequence():
    lens = [0, 1, 5, 40]
    assert acc.varlen_fwd_flops(lens, 2, 8, False) == sum(4 * 8 * 2 * n * n for n in lens)
    assert acc.varlen_fwd_flops(lens, 2, 8, True) == 0.5 * acc.varlen_fwd_flops(lens, 2, 8, False)


@pytest.mark.parametrize("q,k", [(5, 40), (17, 17), (200, 100), (1, 1), (0, 5), (3, 0), (129, 1000)])
@pytest.mark.parametrize("causal", [False, True])
def test_paged_prefill_counts_visible_pairs_exactly(q, k, causal):
    pairs = _pairs(oracle.chunk_key_mask(q, k, causal)) if q and k else 0
    assert acc.paged_prefill_flops([q], [k], 1, 1, causal) == 4 * pairs
    assert acc.paged_prefill_flops([q, q], [k, k], 4, 16, causal) == 2 * 4 * 4 * 16 * pairs


def test_decode_bytes_count_each_key_once_per_kv_head():
    sl = [1, 16, 17]
    b = acc.decode_bytes(sl, 8, 2, 64, 16, with_lse=False)
    kv = sum(sl) * 2 * 64 * 2 * 2
    assert b >= kv and b - kv < 64 * 1024


@pytest.mark.parametrize("N", [128, 300, 512])
@pytest.mark.parametrize("causal", [False, True])
def test_block_sparse_counts_visible_pairs(N, causal):
    nb = (N + 127) // 128
    m = np.random.default_rng(N).random((nb, nb)) < 0.5
    vis = oracle.expand_block_mask(m, N, N, 128)
    if causal:
        vis &= np.tril(np.ones((N, N), bool))
    assert acc.block_sparse_flops(m, 2, 3, N, 8, causal) == 4 * 8 * 2 * 3 * _pairs(vis)
    per = np.stack([np.stack([m, ~m]), np.stack([m, m])])  # [B=2, H=2] per-head masks
    want = sum(_pairs(oracle.expand_block_mask(per[b, h], N, N, 128) & (np.tril(np.ones((N, N), bool))
                                                                      if causal else True))
               for b in range(2) for h in range(2))
    assert acc.block_sparse_flops(per, 2, 2, N, 8, causal) == 4 * 8 * want


def test_key_padding_effective_count_is_every_row_times_its_valid_keys():
    N, H, d = 40, 3, 8
    kv = [40, 7, 0, 23]
    pairs = sum(_pairs(oracle.valid_key_mask(N, N, False, L)) for L in kv)
    assert acc.fwd_flops_padded(H, N, d, kv) == 4 * d * H * pairs


def test_compulsory_bytes_are_the_tensors_each_call_must_touch():
    B, H, N, d = 2, 3, 50, 64
    bf16 = B * H * N * d * 2
    row = B * H * N * 4
    assert acc.fwd_bytes(B, H, N, d) == 4 * bf16 + row  # Q, K, V, O + LSE
    assert acc.bwd_bytes(B, H, N, d) == 8 * bf16 + 2 * row  # Q, K, V, O, dO, dQ, dK, dV + LSE, D
