"""Pins of the paged (chunked) prefill oracle against what the pages and the
mathematics fix, independent of the oracle's own formula: single-query
chunks are decode, each causal row is decode over its visible prefix, a chunk
covering the whole sequence is plain causal attention, a brute-force loop on
tiny inputs, invariance under moving physical blocks, and empty rows."""
import math

import numpy as np
import pytest

import oracle
from exact_io_aware_10_gb300 import workloads as wl


def _inputs(q_lens, kv_lens, Hq=4, Hkv=2, d=8, bs=16, seed=0):
    return wl.paged_prefill_inputs(q_lens, kv_lens, Hq, Hkv, d, block_size=bs, seed=seed)


def _run(P, causal=True, scale=None):
    return oracle.paged_prefill(P.q, P.k_cache, P.v_cache, P.block_table, P.cu_seqlens_q, P.seq_lens_k,
                                P.block_size, causal=causal, scale=scale)


@pytest.mark.parametrize("causal", [False, True])
def test_single_query_chunk_is_decode(causal):
    # q_len = 1 puts the query at the last position: it sees every key, which
    # is the decode problem (S12 "实现"), whichever mask is asked for
    P = _inputs([1, 1, 1], [1, 33, 70], seed=1)
    O, L = _run(P, causal)
    o, lse = oracle.paged_decode(P.q, P.k_cache, P.v_cache, P.block_table, P.seq_lens_k, P.block_size)
    np.testing.assert_allclose(O, o, atol=1e-14)
    np.testing.assert_allclose(L, lse.T, atol=1e-13)


def test_each_causal_row_is_decode_over_its_prefix():
    # row i of a chunk of q_len queries over kv_len keys sees keys
    # 0 .. kv_len - q_len + i: decode with that many keys
    q_lens, kv_lens = [5, 17, 3], [40, 17, 33]
    P = _inputs(q_lens, kv_lens, seed=2)
    O, L = _run(P, True)
    cu = P.cu_seqlens_q.tolist()
    for b, (ql, kl) in enumerate(zip(q_lens, kv_lens)):
        for i in range(ql):
            q = P.q[cu[b] + i][None]
            sl = np.array([kl - ql + i + 1])
            o, lse = oracle.paged_decode(q, P.k_cache, P.v_cache, P.block_table[b:b + 1], sl, P.block_size)
            np.testing.assert_allclose(O[cu[b] + i], o[0], atol=1e-14)
            np.testing.assert_allclose(L[:, cu[b] + i], lse[0], atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_whole_sequence_chunk_is_plain_attention(causal):
    # q_len = kv_len: the queries are the whole sequence and the mask is the
    # square top-left one of plain attention (FA notes §2.1)
    Hq = Hkv = 3
    n, bs, d = 37, 8, 8
    P = _inputs([n], [n], Hq=Hq, Hkv=Hkv, d=d, bs=bs, seed=3)
    O, L = _run(P, causal)
    kc, vc = oracle.to_f64(P.k_cache), oracle.to_f64(P.v_cache)
    bt = P.block_table[0].numpy()
    K = np.stack([oracle.gather_paged_keys(kc, bt, n, bs, g) for g in range(Hkv)])[None]
    V = np.stack([oracle.gather_paged_keys(vc, bt, n, bs, g) for g in range(Hkv)])[None]
    Q = oracle.to_f64(P.q).transpose(1, 0, 2)[None]
    Oref, Lref = oracle.attention_forward(Q, K, V, causal=causal)
    np.testing.assert_allclose(O, Oref[0].transpose(1, 0, 2), atol=1e-14)
    np.testing.assert_allclose(L, Lref[0], atol=1e-13)


def test_brute_force_tiny():
    # scalar loops over the definition with math.exp, GQA group of 2,
    # block size 2, custom scale
    q_lens, kv_lens = [2, 3], [3, 5]
    Hq, Hkv, d, bs, scale = 4, 2, 3, 2, 0.7
    P = _inputs(q_lens, kv_lens, Hq=Hq, Hkv=Hkv, d=d, bs=bs, seed=4)
    O, L = _run(P, True, scale=scale)
    q, kc, vc = (oracle.to_f64(t) for t in (P.q, P.k_cache, P.v_cache))
    bt = P.block_table.numpy()
    cu = P.cu_seqlens_q.tolist()
    for b in range(2):
        ql, kl = q_lens[b], kv_lens[b]
        for i in range(ql):
            for h in range(Hq):
                g = h // (Hq // Hkv)
                keys = range(0, kl - ql + i + 1)
                logits = []
                for j in keys:
                    row = kc[bt[b][j // bs], j % bs, g]
                    logits.append(scale * sum(q[cu[b] + i, h, c] * row[c] for c in range(d)))
                mx = max(logits)
                w = [math.exp(x - mx) for x in logits]
                tot = sum(w)
                for c in range(d):
                    val = sum(w[k] * vc[bt[b][j // bs], j % bs, g, c] for k, j in enumerate(keys)) / tot
                    assert abs(O[cu[b] + i, h, c] - val) < 1e-13
                assert abs(L[h, cu[b] + i] - (mx + math.log(tot))) < 1e-13


def test_moving_physical_blocks_is_bit_identical():
    P = _inputs([4, 9], [50, 30], seed=5)
    O1, L1 = _run(P)
    NB = P.k_cache.shape[0]
    perm = np.random.default_rng(7).permutation(NB)
    inv = np.argsort(perm)
    bt = P.block_table.numpy()
    bt2 = np.where(bt >= 0, inv[np.maximum(bt, 0)], -1)
    O2, L2 = oracle.paged_prefill(P.q, oracle.to_f64(P.k_cache)[perm], oracle.to_f64(P.v_cache)[perm], bt2,
                                  P.cu_seqlens_q, P.seq_lens_k, P.block_size)
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)


def test_rows_before_the_context_are_empty():
    # q_len > kv_len: the first q_len - kv_len rows see no key (O = 0,
    # LSE = -inf) and the rest see the same keys as a q_len = kv_len chunk
    P = _inputs([7], [4], seed=6)
    O, L = _run(P, True)
    assert np.all(O[:3] == 0) and np.all(np.isneginf(L[:, :3]))
    assert np.all(np.isfinite(L[:, 3:]))
    sub = wl.PagedPrefillInputs(P.q[3:], P.k_cache, P.v_cache, P.block_table, P.cu_seqlens_q.clone(),
                                P.seq_lens_k, P.block_size)
    sub.cu_seqlens_q[1] = 4
    O2, L2 = _run(sub, True)
    np.testing.assert_array_equal(O[3:], O2)
    np.testing.assert_array_equal(L[:, 3:], L2)


def test_empty_chunks_and_contexts():
    P = _inputs([0, 3, 0], [10, 3, 0], seed=8)
    O, L = _run(P, True)
    assert O.shape[0] == 3 and np.all(np.isfinite(L))


def test_rows_helper_equals_full_oracle():
    P = _inputs([6, 20], [30, 45], Hq=4, Hkv=1, seed=9)
    O, L = _run(P, True)
    rows = np.array([0, 3, 19])
    Or, Lr = oracle.paged_prefill_rows(P.q, P.k_cache, P.v_cache, P.block_table, P.cu_seqlens_q, P.seq_lens_k,
                                       P.block_size, 1, rows, [0, 3], causal=True)
    a = int(P.cu_seqlens_q[1])
    for t, h in enumerate([0, 3]):
        np.testing.assert_array_equal(Or[t], O[a + rows, h])
        np.testing.assert_array_equal(Lr[t], L[h, a + rows])
