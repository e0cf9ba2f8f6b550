"""Pins for the fp64 oracle: each test checks it against something the pages or
the mathematics fix (closed forms, invariants, finite differences, the pages'
worked numbers, a textbook library routine), never against a re-typed copy of
its own formulas.  CPU only."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle.decode import split_ranges
from exact_io_aware_10_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed, std=1.0):
    g = np.random.default_rng(seed)
    return g.standard_normal(shape) * std


# ---------------------------------------------------------------- forward pins


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("padded", [False, True])
def test_rows_of_P_sum_to_one(causal, padded):
    Q, K = _rand((2, 3, 37, 8), 1), _rand((2, 3, 37, 8), 2)
    kv = np.array([37, 20]) if padded else None
    P = oracle.attention_probs(Q, K, causal=causal, kv_lens=kv)
    s = P.sum(-1)
    assert np.abs(s - 1).max() <= 1e-14
    assert (P >= 0).all()
    if causal:
        assert np.all(np.triu(P[0, 0], 1) == 0)
    if padded:
        assert np.all(P[1, :, :, 20:] == 0)


def test_single_key_returns_its_value():
    Q, K, V = _rand((1, 2, 1, 5), 3), _rand((1, 2, 1, 5), 4), _rand((1, 2, 1, 5), 5)
    O, L = oracle.attention_forward(Q, K, V, scale=0.7)
    np.testing.assert_allclose(O, V, rtol=0, atol=1e-15)
    np.testing.assert_allclose(L, 0.7 * (Q * K).sum(-1), rtol=1e-15, atol=1e-15)


@pytest.mark.parametrize("causal", [False, True])
def test_identical_keys_give_mean_of_values(causal):
    N, d = 9, 4
    Q = _rand((1, 1, N, d), 6)
    k = _rand((d,), 7)
    K = np.broadcast_to(k, (1, 1, N, d)).copy()
    V = _rand((1, 1, N, d), 8)
    O, L = oracle.attention_forward(Q, K, V, causal=causal, scale=0.5)
    for i in range(N):
        n = i + 1 if causal else N
        np.testing.assert_allclose(O[0, 0, i], V[0, 0, :n].mean(0), atol=1e-14)
        np.testing.assert_allclose(L[0, 0, i], 0.5 * Q[0, 0, i] @ k + math.log(n), atol=1e-13)


def test_causal_row0_returns_v0():
    Q, K, V = (_rand((2, 2, 11, 6), s) for s in (9, 10, 11))
    O, L = oracle.attention_forward(Q, K, V, causal=True)
    np.testing.assert_allclose(O[:, :, 0], V[:, :, 0], atol=1e-15)
    np.testing.assert_allclose(L[:, :, 0], (Q[:, :, 0] * K[:, :, 0]).sum(-1) / math.sqrt(6), atol=1e-14)


def test_hand_computed_d1_cases():
    # d = 1, scale = 1.  Q = [1, 2], K = [0, 1], V = [1, 3]:
    # row 0 logits (0, 1): O = (1 + 3e)/(1 + e), LSE = ln(1 + e)
    # row 1 logits (0, 2): O = (1 + 3e^2)/(1 + e^2), LSE = ln(1 + e^2)
    e = math.e
    Q = np.array([1.0, 2.0]).reshape(1, 1, 2, 1)
    K = np.array([0.0, 1.0]).reshape(1, 1, 2, 1)
    V = np.array([1.0, 3.0]).reshape(1, 1, 2, 1)
    O, L = oracle.attention_forward(Q, K, V, scale=1.0)
    np.testing.assert_allclose(O.ravel(), [(1 + 3 * e) / (1 + e), (1 + 3 * e * e) / (1 + e * e)], rtol=1e-15)
    np.testing.assert_allclose(L.ravel(), [math.log(1 + e), math.log(1 + e * e)], rtol=1e-15)
    # causal: row 0 sees key 0 only, row 1 as before
    O, L = oracle.attention_forward(Q, K, V, causal=True, scale=1.0)
    np.testing.assert_allclose(O.ravel(), [1.0, (1 + 3 * e * e) / (1 + e * e)], rtol=1e-15)
    np.testing.assert_allclose(L.ravel(), [0.0, math.log(1 + e * e)], atol=1e-15)
    # 3 keys, q = 1: logits (-1, 0, 1), V = (0, 1, 2): O = (1*1 + 2e)/(1/e + 1 + e)
    Q = np.ones((1, 1, 1, 1))
    K = np.array([-1.0, 0.0, 1.0]).reshape(1, 1, 3, 1)
    V = np.array([0.0, 1.0, 2.0]).reshape(1, 1, 3, 1)
    O, L = oracle.attention_forward(Q[:, :, :1], K, V, scale=1.0)
    np.testing.assert_allclose(O.ravel(), [(1 + 2 * e) / (1 / e + 1 + e)], rtol=1e-15)
    np.testing.assert_allclose(L.ravel(), [math.log(1 / e + 1 + e)], rtol=1e-15)


def test_shift_invariance():
    # an extra coordinate with q_extra = c and k_extra = 1 adds c to every
    # logit of the row (scale 1): O is unchanged, LSE moves by exactly c.
    Q, K, V = _rand((1, 2, 13, 5), 12), _rand((1, 2, 13, 5), 13), _rand((1, 2, 13, 5), 14)
    c = 3.25
    Q2 = np.concatenate([Q, np.full((1, 2, 13, 1), c)], -1)
    K2 = np.concatenate([K, np.ones((1, 2, 13, 1))], -1)
    for causal in (False, True):
        O1, L1 = oracle.attention_forward(Q, K, V, causal=causal, scale=1.0)
        O2, L2 = oracle.attention_forward(Q2, K2, V, causal=causal, scale=1.0)
        np.testing.assert_allclose(O2, O1, atol=1e-13)
        np.testing.assert_allclose(L2, L1 + c, atol=1e-13)


def test_key_value_permutation_invariance():
    Q, K, V = _rand((1, 1, 10, 4), 15), _rand((1, 1, 12, 4), 16), _rand((1, 1, 12, 4), 17)
    perm = np.random.default_rng(0).permutation(12)
    O1, L1 = oracle.attention_forward(Q, K, V)
    O2, L2 = oracle.attention_forward(Q, K[:, :, perm], V[:, :, perm])
    np.testing.assert_allclose(O2, O1, atol=1e-14)
    np.testing.assert_allclose(L2, L1, atol=1e-14)


def test_empty_rows_are_zero_with_minus_inf_lse():
    Q, K, V = (_rand((2, 1, 5, 3), s) for s in (18, 19, 20))
    O, L = oracle.attention_forward(Q, K, V, kv_lens=np.array([0, 2]))
    assert np.all(O[0] == 0) and np.all(np.isneginf(L[0]))
    assert np.all(np.isfinite(L[1]))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("padded", [False, True])
def test_forward_matches_textbook_library_attention(causal, padded):
    # torch's scaled_dot_product_attention in float64 on the CPU is an
    # independent implementation of the textbook definition.
    B, H, N, d = 2, 2, 33, 16
    Q, K, V = (torch.from_numpy(_rand((B, H, N, d), s)) for s in (21, 22, 23))
    kv = np.array([33, 17]) if padded else None
    O, L = oracle.attention_forward(Q, K, V, causal=causal, kv_lens=kv)
    mask = torch.ones(B, 1, N, N, dtype=torch.bool)
    if causal:
        mask &= torch.ones(N, N, dtype=torch.bool).tril()
    if padded:
        for b in range(B):
            mask[b, :, :, int(kv[b]):] = False
    ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask)
    np.testing.assert_allclose(O, ref.numpy(), atol=1e-13)
    # LSE against logsumexp of the masked logit matrix
    S = (Q @ K.transpose(-1, -2)) / math.sqrt(d)
    S = S.masked_fill(~mask, float("-inf"))
    np.testing.assert_allclose(L, torch.logsumexp(S, -1).numpy(), atol=1e-13)


# ---------------------------------------------------------------- streaming / tiled pins


@pytest.mark.parametrize("N", [1, 7, 16, 33])
def test_streaming_loop_equals_materialised_for_every_tile(N):
    d = 5
    Q, K, V = _rand((1, 1, N, d), 24), _rand((1, 1, N, d), 25), _rand((1, 1, N, d), 26)
    O, L = oracle.attention_forward(Q, K, V, causal=False)
    Oc, Lc = oracle.attention_forward(Q, K, V, causal=True)
    for tile in range(1, N + 1):
        for i in range(N):
            o, m, l = oracle.streaming_row_forward(Q[0, 0, i], K[0, 0], V[0, 0], tile, 1 / math.sqrt(d))
            assert np.abs(o - O[0, 0, i]).max() <= 1e-13
            assert abs(m + math.log(l) - L[0, 0, i]) <= 1e-13
            mask = np.arange(N) <= i
            o, m, l = oracle.streaming_row_forward(Q[0, 0, i], K[0, 0], V[0, 0], tile, 1 / math.sqrt(d), key_mask=mask)
            assert np.abs(o - Oc[0, 0, i]).max() <= 1e-13
            assert abs(m + math.log(l) - Lc[0, 0, i]) <= 1e-13


@pytest.mark.parametrize("N", [1, 5, 24, 40])
@pytest.mark.parametrize("causal", [False, True])
def test_algorithm1_equals_materialised_for_every_block_size(N, causal):
    d = 4
    Q, K, V = _rand((N, d), 27), _rand((N, d), 28), _rand((N, d), 29)
    O, L = oracle.attention_forward(Q[None, None], K[None, None], V[None, None], causal=causal, scale=1.0)
    for Bc in range(1, N + 1):
        for Br in sorted({1, 2, 3, max(1, N // 2), N}):
            Oa, l, m = oracle.algorithm1_forward(Q, K, V, Br, Bc, scale=1.0, causal=causal)
            assert np.abs(Oa - O[0, 0]).max() <= 1e-13
            assert np.abs(m + np.log(l) - L[0, 0]).max() <= 1e-13


def test_fully_masked_first_tile_nan_hazard_and_guard():
    # [S12]: if the first tile is entirely masked, the running max is still
    # -inf and exp(-inf - -inf) is NaN; the guard removes it.
    N, d = 12, 4
    q, K, V = _rand((d,), 30), _rand((N, d), 31), _rand((N, d), 32)
    mask = np.arange(N) >= 4  # the first tile of 4 keys is fully masked
    o_bad, _, _ = oracle.streaming_row_forward(q, K, V, 4, 0.5, key_mask=mask, nan_guard=False)
    assert np.isnan(o_bad).all()
    o, m, l = oracle.streaming_row_forward(q, K, V, 4, 0.5, key_mask=mask, nan_guard=True)
    s = 0.5 * K[4:] @ q
    p = np.exp(s - s.max())
    np.testing.assert_allclose(o, (p / p.sum()) @ V[4:], atol=1e-14)
    o, m, l = oracle.streaming_row_forward(q, K, V, 4, 0.5, key_mask=np.zeros(N, bool), nan_guard=True)
    assert np.all(o == 0) and m == -np.inf and l == 0


def test_merge_of_split_states_equals_single_pass():
    N, d = 50, 6
    q, K, V = _rand((d,), 33), _rand((N, d), 34), _rand((N, d), 35)
    o_ref, m_ref, l_ref = oracle.streaming_row_forward(q, K, V, N, 0.4)
    for S in list(range(1, 17)) + [4]:
        ms, ls, os_ = [], [], []
        for lo, hi in split_ranges(N, S):
            if hi <= lo:
                ms.append(-np.inf), ls.append(0.0), os_.append(np.zeros(d))
                continue
            o, m, l = oracle.streaming_row_forward(q, K[lo:hi], V[lo:hi], 3, 0.4)
            ms.append(m), ls.append(l), os_.append(o * l)
        o, m, l = oracle.merge_states(ms, ls, os_)
        assert np.abs(o - o_ref).max() <= 1e-13
        assert abs((m + math.log(l)) - (m_ref + math.log(l_ref))) <= 1e-13


# ---------------------------------------------------------------- backward pins


def _loss(Q, K, V, dO, causal, scale, kv):
    O, _ = oracle.attention_forward(Q, K, V, causal=causal, scale=scale, kv_lens=kv)
    return float((O * dO).sum())


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("padded", [False, True])
def test_backward_matches_central_finite_differences(causal, padded):
    B, H, N, d = 1, 1, 9, 4
    Q, K, V, dO = (_rand((B, H, N, d), s) for s in (36, 37, 38, 39))
    kv = np.array([6]) if padded else None
    scale = 0.6
    dQ, dK, dV = oracle.attention_backward(Q, K, V, dO, causal=causal, scale=scale, kv_lens=kv)
    h = 1e-6
    for X, G in ((Q, dQ), (K, dK), (V, dV)):
        num = np.zeros_like(X)
        it = np.nditer(X, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            x0 = X[idx]
            X[idx] = x0 + h
            fp = _loss(Q, K, V, dO, causal, scale, kv)
            X[idx] = x0 - h
            fm = _loss(Q, K, V, dO, causal, scale, kv)
            X[idx] = x0
            num[idx] = (fp - fm) / (2 * h)
        err = np.linalg.norm(num - G) / max(np.linalg.norm(G), 1e-30)
        assert err <= 1e-6, err


def test_backward_matches_textbook_library_autograd():
    B, H, N, d = 2, 2, 21, 8
    for causal in (False, True):
        Q, K, V, dO = (torch.from_numpy(_rand((B, H, N, d), s)) for s in (40, 41, 42, 43))
        dQ, dK, dV = oracle.attention_backward(Q, K, V, dO, causal=causal)
        q, k, v = (t.clone().requires_grad_(True) for t in (Q, K, V))
        out = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=causal)
        out.backward(dO)
        np.testing.assert_allclose(dQ, q.grad.numpy(), atol=1e-12)
        np.testing.assert_allclose(dK, k.grad.numpy(), atol=1e-12)
        np.testing.assert_allclose(dV, v.grad.numpy(), atol=1e-12)


def test_rowsum_identity_and_padded_keys_get_no_gradient():
    B, H, N, d = 2, 1, 15, 4
    Q, K, V, dO = (_rand((B, H, N, d), s) for s in (44, 45, 46, 47))
    kv = np.array([15, 9])
    dQ, dK, dV, D = oracle.attention_backward(Q, K, V, dO, causal=True, kv_lens=kv, return_aux=True)
    O, _ = oracle.attention_forward(Q, K, V, causal=True, kv_lens=kv)
    np.testing.assert_allclose(D, (dO * O).sum(-1), atol=1e-12)
    assert np.all(dK[1, :, 9:] == 0) and np.all(dV[1, :, 9:] == 0)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_rows_match_finite_differences_of_the_rows_loss(causal):
    # the loss restricted to the selected rows, sum_{i in rows} dO_i . O_i: its
    # gradient is dQ on those rows (zero elsewhere) and the rows' share of dK, dV
    B, H, N, d = 1, 1, 8, 3
    Q, K, V, dO = (_rand((B, H, N, d), s) for s in (48, 49, 50, 51))
    rows = np.array([0, 3, 7])
    kv = np.array([6])
    scale = 0.7
    gq, gk, gv = oracle.attention_backward_rows(Q, K, V, dO, rows, causal=causal, scale=scale, kv_lens=kv)
    mask = np.zeros((N, 1))
    mask[rows] = 1.0

    def loss():
        O, _ = oracle.attention_forward(Q, K, V, causal=causal, scale=scale, kv_lens=kv)
        return float((O[0, 0] * dO[0, 0] * mask).sum())

    h = 1e-6
    for X, G in ((Q, None), (K, gk[0]), (V, gv[0])):
        num = np.zeros((N, d))
        for i in range(N):
            for c in range(d):
                x0 = X[0, 0, i, c]
                X[0, 0, i, c] = x0 + h
                fp = loss()
                X[0, 0, i, c] = x0 - h
                fm = loss()
                X[0, 0, i, c] = x0
                num[i, c] = (fp - fm) / (2 * h)
        if G is None:  # Q: only the selected rows carry gradient
            assert np.abs(np.delete(num, rows, axis=0)).max() <= 1e-8
            num, G = num[rows], gq[0]
        err = np.linalg.norm(num - G) / max(np.linalg.norm(G), 1e-30)
        assert err <= 1e-6, err


def test_backward_rows_over_a_partition_sum_to_the_full_backward():
    B, H, N, d = 2, 2, 37, 8
    Q, K, V, dO = (_rand((B, H, N, d), s) for s in (52, 53, 54, 55))
    kv = np.array([37, 20])
    for causal in (False, True):
        dQ, dK, dV = oracle.attention_backward(Q, K, V, dO, causal=causal, kv_lens=kv)
        parts = [np.arange(0, 10), np.arange(10, 11), np.arange(11, 37)]
        acc_k, acc_v = np.zeros_like(dK), np.zeros_like(dV)
        heads = [(b, h) for b in range(B) for h in range(H)]
        for rows in parts:
            gq, gk, gv = oracle.attention_backward_rows(Q, K, V, dO, rows, causal=causal, kv_lens=kv, heads=heads)
            for t, (b, h) in enumerate(heads):
                np.testing.assert_allclose(gq[t], dQ[b, h, rows], atol=1e-12)
                acc_k[b, h] += gk[t]
                acc_v[b, h] += gv[t]
        np.testing.assert_allclose(acc_k, dK, atol=1e-12)
        np.testing.assert_allclose(acc_v, dV, atol=1e-12)


# ---------------------------------------------------------------- paged decode pins


def _paged(B=3, Hq=8, Hkv=2, d=8, lo=1, hi=70, bs=16, seed=0, seq_lens=None):
    return wl.paged_inputs(B, Hq, Hkv, d, lo, hi, block_size=bs, seed=seed, seq_lens=seq_lens)


def test_paged_identity_table_equals_causal_prefill_last_row():
    B, Hq, Hkv, d, bs = 1, 4, 4, 8, 16
    L = 45
    N = 48
    Q, K, V = _rand((1, Hq, N, d), 48), _rand((1, Hq, N, d), 49), _rand((1, Hq, N, d), 50)
    nb = N // bs
    kc = K[0].transpose(1, 0, 2).reshape(nb, bs, Hkv, d)
    vc = V[0].transpose(1, 0, 2).reshape(nb, bs, Hkv, d)
    table = np.arange(nb, dtype=np.int32)[None]
    q = Q[0, :, L - 1]
    o, lse = oracle.paged_decode(q[None], kc, vc, table, np.array([L]), bs)
    O, LS = oracle.attention_forward(Q, K, V, causal=True)
    np.testing.assert_allclose(o[0], O[0, :, L - 1], atol=1e-14)
    np.testing.assert_allclose(lse[0], LS[0, :, L - 1], atol=1e-13)


def test_paged_physical_permutation_is_bit_identical():
    P = _paged()
    o1, l1 = oracle.paged_decode(P.q, P.k_cache, P.v_cache, P.block_table, P.seq_lens, P.block_size)
    perm = np.random.default_rng(3).permutation(P.num_blocks)
    inv = np.argsort(perm)
    kc = oracle.to_f64(P.k_cache)[perm]
    vc = oracle.to_f64(P.v_cache)[perm]
    bt = P.block_table.numpy().copy()
    bt = np.where(bt >= 0, inv[np.maximum(bt, 0)], -1)
    o2, l2 = oracle.paged_decode(P.q, kc, vc, bt, P.seq_lens, P.block_size)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_paged_mha_reduces_to_single_query_attention():
    P = _paged(Hq=4, Hkv=4)
    o, lse = oracle.paged_decode(P.q, P.k_cache, P.v_cache, P.block_table, P.seq_lens, P.block_size)
    kc, vc, q = oracle.to_f64(P.k_cache), oracle.to_f64(P.v_cache), oracle.to_f64(P.q)
    for b in range(q.shape[0]):
        L = int(P.seq_lens[b])
        for h in range(4):
            Kb = oracle.gather_paged_keys(kc, P.block_table[b].numpy(), L, 16, h)
            Vb = oracle.gather_paged_keys(vc, P.block_table[b].numpy(), L, 16, h)
            Ob, Lb = oracle.attention_forward(q[b, h][None, None, None], Kb[None, None], Vb[None, None])
            np.testing.assert_allclose(o[b, h], Ob[0, 0, 0], atol=1e-14)
            np.testing.assert_allclose(lse[b, h], Lb[0, 0, 0], atol=1e-13)


def test_paged_gqa_group_shares_one_kv_head():
    # heads h and h' of the same group with identical queries give identical outputs;
    # changing KV head 1 leaves heads of group 0 untouched.
    P = _paged(Hq=8, Hkv=2)
    q = P.q.clone()
    q[:, 1] = q[:, 0]
    o1, _ = oracle.paged_decode(q, P.k_cache, P.v_cache, P.block_table, P.seq_lens, 16)
    assert np.array_equal(o1[:, 0], o1[:, 1])
    kc = P.k_cache.clone()
    kc[:, :, 1] += 1
    o2, _ = oracle.paged_decode(q, kc, P.v_cache, P.block_table, P.seq_lens, 16)
    assert np.array_equal(o1[:, :4], o2[:, :4])
    assert not np.array_equal(o1[:, 4:], o2[:, 4:])


def test_paged_streaming_and_split_equal_definition():
    P = _paged(seq_lens=[1, 16, 17, 70])
    o, lse = oracle.paged_decode(P.q, P.k_cache, P.v_cache, P.block_table, P.seq_lens, 16)
    o_s = oracle.paged_decode_streaming(P.q, P.k_cache, P.v_cache, P.block_table, P.seq_lens, 16)
    np.testing.assert_allclose(o_s, o, atol=1e-13)
    for S in (1, 2, 3, 4, 5, 16):
        o_k, lse_k = oracle.split_paged_decode(P.q, P.k_cache, P.v_cache, P.block_table, P.seq_lens, 16, S)
        np.testing.assert_allclose(o_k, o, atol=1e-13)
        np.testing.assert_allclose(lse_k, lse, atol=1e-13)


def test_paged_empty_sequence():
    P = _paged(seq_lens=[0, 5])
    o, lse = oracle.paged_decode(P.q, P.k_cache, P.v_cache, P.block_table, P.seq_lens, 16)
    assert np.all(o[0] == 0) and np.all(np.isneginf(lse[0]))
    o_k, lse_k = oracle.split_paged_decode(P.q, P.k_cache, P.v_cache, P.block_table, P.seq_lens, 16, 4)
    assert np.all(o_k[0] == 0) and np.all(np.isneginf(lse_k[0]))
    np.testing.assert_allclose(o_k[1], o[1], atol=1e-13)


# ---------------------------------------------------------------- IO model pins


def test_io_model_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "io_model.json")))
    std = oracle.standard_hbm_accesses(g["N"], g["d"])
    fl = oracle.flash_hbm_accesses(g["N"], g["d"], g["M_elements"])
    assert std == g["standard_accesses"]
    assert int(fl) == g["flash_accesses"]
    assert round(std / fl, 1) == g["ratio_approx"]


def test_materialised_memory_numbers():
    g = json.load(open(os.path.join(GOLDEN, "materialized_memory.json")))
    for c in g["cases"]:
        assert oracle.materialized_matrix_bytes(c["N"], c["bytes_per_elem"], c["n_matrices"], c["heads"]) == c["bytes"]


def test_varlen_oracle_is_per_sequence_attention_and_ignores_neighbours():
    # each packed sequence equals an isolated problem; changing another
    # sequence's tokens does not change it (independence of sequences)
    H, d = 3, 8
    lens = [5, 1, 17, 9]
    cu = np.concatenate([[0], np.cumsum(lens)])
    total = int(cu[-1])
    Q, K, V = (_rand((total, H, d), s) for s in (60, 61, 62))
    for causal in (False, True):
        O, L = oracle.attention_forward_varlen(Q, K, V, cu, causal=causal)
        for s, n in enumerate(lens):
            a = int(cu[s])
            # single-sequence closed checks: causal row 0 returns V[0]
            if causal:
                np.testing.assert_allclose(O[a], V[a], atol=1e-15)
            P = oracle.attention_probs(Q[a:a + n].transpose(1, 0, 2)[None], K[a:a + n].transpose(1, 0, 2)[None],
                                       causal=causal)
            np.testing.assert_allclose(O[a:a + n].transpose(1, 0, 2), (P[0] @ V[a:a + n].transpose(1, 0, 2)),
                                       atol=1e-13)
        K2 = K.copy()
        K2[int(cu[2]):int(cu[3])] += _rand((lens[2], H, d), 63)  # perturb sequence 2 only
        O2, _ = oracle.attention_forward_varlen(Q, K2, V, cu, causal=causal)
        keep = np.r_[0:int(cu[2]), int(cu[3]):total]
        np.testing.assert_array_equal(O2[keep], O[keep])
        assert not np.allclose(O2[int(cu[2]):int(cu[3])], O[int(cu[2]):int(cu[3])])


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_backward_matches_finite_differences_of_the_packed_loss(causal):
    # the packed gradients are the derivative of sum(dO * O_varlen): central
    # differences through attention_forward_varlen on every coordinate of a
    # tiny ragged batch (lengths 3, 1, 0, 4), independent of the per-sequence
    # unpacking inside the backward
    H, d = 2, 3
    lens = [3, 1, 0, 4]
    cu = np.concatenate([[0], np.cumsum(lens)])
    total = int(cu[-1])
    Q, K, V, dO = (_rand((total, H, d), s) for s in (70, 71, 72, 73))
    scale = 0.7
    dQ, dK, dV = oracle.attention_backward_varlen(Q, K, V, dO, cu, causal=causal, scale=scale)

    def loss(q, k, v):
        o, _ = oracle.attention_forward_varlen(q, k, v, cu, causal=causal, scale=scale)
        return float((o * dO).sum())

    h = 1e-6
    for name, X, G in (("Q", Q, dQ), ("K", K, dK), ("V", V, dV)):
        num = np.zeros_like(X)
        for idx in np.ndindex(X.shape):
            Xp, Xm = X.copy(), X.copy()
            Xp[idx] += h
            Xm[idx] -= h
            args_p = [Xp if n == name else Y for n, Y in (("Q", Q), ("K", K), ("V", V))]
            args_m = [Xm if n == name else Y for n, Y in (("Q", Q), ("K", K), ("V", V))]
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        np.testing.assert_allclose(G, num, atol=1e-7, rtol=1e-6, err_msg=name)


def test_varlen_backward_sequences_are_independent():
    H, d = 2, 4
    lens = [5, 9, 2]
    cu = np.concatenate([[0], np.cumsum(lens)])
    total = int(cu[-1])
    Q, K, V, dO = (_rand((total, H, d), s) for s in (80, 81, 82, 83))
    g1 = oracle.attention_backward_varlen(Q, K, V, dO, cu, causal=True)
    K2 = K.copy()
    K2[5:14] += _rand((9, H, d), 84)  # sequence 1 only
    g2 = oracle.attention_backward_varlen(Q, K2, V, dO, cu, causal=True)
    keep = np.r_[0:5, 14:16]
    for a, b in zip(g1, g2):
        np.testing.assert_array_equal(a[keep], b[keep])
