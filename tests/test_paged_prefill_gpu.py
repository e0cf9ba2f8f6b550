"""Paged (chunked) prefill parity: fa_paged_prefill through the C ABI against
the fp64 oracle on the same seeded bf16 inputs.  Tolerances are the forward
ones: O max-abs <= 2e-2 and mean-abs <= 2e-3, LSE abs <= 1e-3.  Block-table
indexing is checked bit for bit: a chunk covering its whole sequence gives
exactly the packed ragged-batch forward's results on the same tokens."""
import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_10_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_TOL = 2e-2, 2e-3, 1e-3

# the chunked-prefill mix the kernel is measured on: 16 sequences, each a
# 2048-token chunk after a cached prefix of U[0, 30720] tokens, Hq=32, Hkv=8,
# d=128, 16-token blocks, causal
CHUNK = dict(num_seqs=16, q_len=2048, prefix_lo=0, prefix_hi=30720, Hq=32, Hkv=8, d=128, block_size=16)


def _dev(P):
    dev = torch.device("cuda")
    return [t.to(dev) for t in (P.q, P.k_cache, P.v_cache, P.block_table, P.cu_seqlens_q, P.seq_lens_k)]


def _run(fa, P, causal=True, scale=None, max_seqlen_q=None, expect=None):
    q, kc, vc, bt, cu, sl = _dev(P)
    O, L = fa.fa_paged_prefill(q, kc, vc, bt, cu, sl, P.max_seqlen_q if max_seqlen_q is None else max_seqlen_q,
                               causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == (fa.FA_OK if expect is None else expect)
    return O.float().cpu().numpy(), L.cpu().numpy()


def _ref(P, causal=True, scale=None):
    return oracle.paged_prefill(P.q, P.k_cache, P.v_cache, P.block_table, P.cu_seqlens_q, P.seq_lens_k,
                                P.block_size, causal=causal, scale=scale)


def _check(O, L, Oref, Lref):
    err = np.abs(O - Oref)
    assert np.isfinite(O).all()
    assert err.max(initial=0) <= O_MAX, err.max()
    assert err.mean() <= O_MEAN, err.mean()
    fin = np.isfinite(Lref)
    assert np.array_equal(np.isfinite(L), fin)
    assert np.abs(L[fin] - Lref[fin]).max(initial=0) <= LSE_TOL


EDGE_Q = [1, 17, 128, 129, 300, 0, 5, 200, 256]
EDGE_K = [1, 300, 128, 1000, 300, 50, 0, 100, 700]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_edge_chunks(fa, d, causal):
    # single-token chunks, chunks equal to the context, ragged tails, empty
    # chunks, an empty context, and chunks longer than their context (rows
    # before the context start see no key)
    P = wl.paged_prefill_inputs(EDGE_Q, EDGE_K, 8, 2, d, block_size=16, seed=40 + d)
    O, L = _run(fa, P, causal)
    Oref, Lref = _ref(P, causal)
    _check(O, L, Oref, Lref)


@pytest.mark.parametrize("bs", [8, 16, 32, 64, 128, 256])
def test_block_sizes(fa, bs):
    P = wl.paged_prefill_inputs([77, 256, 3], [600, 256, 1025], 4, 4, 128, block_size=bs, seed=bs)
    O, L = _run(fa, P, True)
    Oref, Lref = _ref(P, True)
    _check(O, L, Oref, Lref)


def test_gqa_groups_and_scale(fa):
    for Hq, Hkv in ((8, 1), (8, 8), (6, 3)):
        P = wl.paged_prefill_inputs([100, 33], [400, 33], Hq, Hkv, 64, block_size=32, seed=Hq * 10 + Hkv)
        O, L = _run(fa, P, True, scale=0.2)
        Oref, Lref = _ref(P, True, scale=0.2)
        _check(O, L, Oref, Lref)


def test_whole_sequence_chunks_equal_ragged_forward_bitwise(fa):
    # q_len = kv_len puts each chunk's queries on the keys' own positions;
    # gathering the keys through the table must reproduce the contiguous
    # ragged-batch forward exactly (same tiles, same arithmetic)
    lens = [5, 128, 300, 1000, 129]
    H, d, bs = 4, 128, 16
    for causal in (False, True):
        P = wl.paged_prefill_inputs(lens, lens, H, H, d, block_size=bs, seed=77)
        O, L = _run(fa, P, causal)
        kc, vc = P.k_cache, P.v_cache
        K = torch.cat([kc[P.block_table[s, np.arange(n) // bs].long(), torch.arange(n) % bs] for s, n in
                       enumerate(lens)])
        V = torch.cat([vc[P.block_table[s, np.arange(n) // bs].long(), torch.arange(n) % bs] for s, n in
                       enumerate(lens)])
        dev = torch.device("cuda")
        Ov, Lv = fa.fa_fwd_varlen(P.q.to(dev), K.to(dev), V.to(dev), P.cu_seqlens_q.to(dev), max(lens),
                                  causal=causal)
        torch.cuda.synchronize()
        assert np.array_equal(O, Ov.float().cpu().numpy())
        assert np.array_equal(L, Lv.cpu().numpy())


def test_single_token_chunks_match_decode(fa):
    # q_len = 1 is the decode problem: the prefill kernel and the split-KV
    # decode kernel agree within the forward tolerance
    B, Hq, Hkv, d = 6, 16, 4, 128
    kv = [1, 15, 16, 17, 1000, 4097]
    P = wl.paged_prefill_inputs([1] * B, kv, Hq, Hkv, d, block_size=16, seed=9)
    O, L = _run(fa, P, True)
    q, kc, vc, bt, cu, sl = _dev(P)
    o, lse = fa.fa_paged_decode(q, kc, vc, bt, sl)
    torch.cuda.synchronize()
    _check(O, L, o.float().cpu().numpy(), lse.cpu().numpy().T)


def test_bad_block_table_entry_is_reported(fa):
    P = wl.paged_prefill_inputs([40, 60], [300, 200], 4, 2, 64, block_size=16, seed=12)
    Oref, Lref = _ref(P, True)
    P.block_table[1, 3] = P.k_cache.shape[0] + 5  # out of range, inside sequence 1's blocks
    O, L = _run(fa, P, True, expect=fa.FA_ERR_BAD_BLOCK_TABLE)
    _check(O[:40], L[:, :40], Oref[:40], Lref[:, :40])  # sequence 0 unaffected
    assert np.isfinite(O).all()
    # the context is usable again and the status word was cleared
    P.block_table[1, 3] = 0
    _run(fa, P, True)


def test_context_longer_than_its_table_row_is_reported(fa):
    P = wl.paged_prefill_inputs([10, 20], [100, 50], 2, 2, 64, block_size=16, seed=13)
    Oref, Lref = _ref(P, True)
    P.seq_lens_k[1] = P.block_table.shape[1] * 16 + 1
    q, kc, vc, bt, cu, sl = _dev(P)
    O = torch.full_like(q, 3.0)
    fa.fa_paged_prefill(q, kc, vc, bt, cu, sl, P.max_seqlen_q, causal=True, o=O)
    assert fa.fa_get_device_status() == fa.FA_ERR_INVALID_ARG
    On = O.float().cpu().numpy()
    assert (On[10:] == 3.0).all()
    _check(On[:10], np.zeros(0), Oref[:10], np.zeros(0))


def _chunk_mix(seed=0):
    c = CHUNK
    g = torch.Generator().manual_seed(wl.config_seed(seed, 7))
    prefix = torch.randint(c["prefix_lo"], c["prefix_hi"] + 1, (c["num_seqs"],), generator=g).tolist()
    q_lens = [c["q_len"]] * c["num_seqs"]
    kv = [p + c["q_len"] for p in prefix]
    return q_lens, kv


def test_chunked_prefill_mix_sampled_rows(fa):
    # the measured chunked-prefill mix at full size: sampled rows of three
    # chunks, three query heads each (two in one KV group)
    c = CHUNK
    q_lens, kv = _chunk_mix()
    P = wl.paged_prefill_inputs(q_lens, kv, c["Hq"], c["Hkv"], c["d"], block_size=c["block_size"],
                                seed=wl.config_seed(0, 7))
    O, L = _run(fa, P, True)
    cu = P.cu_seqlens_q.tolist()
    heads = [0, 1, c["Hq"] - 1]
    for s in (0, 7, c["num_seqs"] - 1):
        rows = np.unique(np.concatenate([np.arange(0, q_lens[s], 331), [q_lens[s] - 1, 127, 128]]))
        Or, Lr = oracle.paged_prefill_rows(P.q, P.k_cache, P.v_cache, P.block_table, P.cu_seqlens_q, P.seq_lens_k,
                                           P.block_size, s, rows, heads, causal=True)
        for t, h in enumerate(heads):
            _check(O[cu[s] + rows, h], L[h, cu[s] + rows], Or[t], Lr[t])


def test_deterministic(fa):
    P = wl.paged_prefill_inputs([300, 7], [900, 7], 8, 2, 128, block_size=16, seed=14)
    a = _run(fa, P, True)
    b = _run(fa, P, True)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_gather_retrieves_exact_rows(fa):
    # block-table indexing checked bit for bit: q = c e_0 for every token, all
    # keys zero but one target per (sequence, KV head) inside the cached prefix
    # (so every causal row sees it); each output row must be that key's V row
    q_lens, kv = [5, 130, 1, 64], [40, 700, 2000, 64 + 900]
    Hq, Hkv = 8, 2
    for bs in (16, 64):
        P = wl.paged_prefill_inputs(q_lens, kv, Hq, Hkv, 128, block_size=bs, seed=31)
        P.q.zero_()
        P.q[..., 0] = 8.0
        P.k_cache.zero_()
        g = torch.Generator().manual_seed(7)
        tg = {}
        for s in range(len(q_lens)):
            for h in range(Hkv):
                t = int(torch.randint(0, kv[s] - q_lens[s] + 1, (1,), generator=g))
                tg[s, h] = t
                P.k_cache[int(P.block_table[s, t // bs]), t % bs, h, 0] = 64.0
        O, L = _run(fa, P, True)
        cu = P.cu_seqlens_q.tolist()
        for s in range(len(q_lens)):
            for h in range(Hq):
                t = tg[s, h // (Hq // Hkv)]
                want = P.v_cache[int(P.block_table[s, t // bs]), t % bs, h // (Hq // Hkv)].float().numpy()
                rows = O[cu[s]:cu[s + 1], h]
                assert np.array_equal(rows, np.broadcast_to(want, rows.shape)), (bs, s, h)
