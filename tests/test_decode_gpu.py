"""Paged split-KV GQA decode parity: the CUDA path (through the C ABI) against
the fp64 oracle on the same seeded inputs; integer/indexing behaviour is
checked bit-exactly (output invariance under physical block placement)."""
import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_10_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_TOL = 2e-2, 2e-3, 1e-3


def _dev(P):
    d = torch.device("cuda")
    return (P.q.to(d), P.k_cache.to(d), P.v_cache.to(d), P.block_table.to(d), P.seq_lens.to(d))


def _run(fa, P, num_splits=0, expect_status=0):
    q, kc, vc, bt, sl = _dev(P)
    o, lse = fa.fa_paged_decode(q, kc, vc, bt, sl, num_splits=num_splits)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == expect_status
    return o.float().cpu().numpy(), lse.cpu().numpy()


def _compact(P, b):
    """Sequence b alone, with only its own cache blocks (same values, identity
    table), so the oracle does not widen the whole cache to fp64."""
    nb = (int(P.seq_lens[b]) + 15) // 16
    ids = P.block_table[b, :nb].long()
    bt = torch.arange(max(nb, 1), dtype=torch.int32)[None]
    return wl.PagedInputs(P.q[b:b + 1], P.k_cache[ids], P.v_cache[ids], bt, P.seq_lens[b:b + 1], 16)


def _check(o, lse, oref, lref):
    err = np.abs(o - oref)
    assert np.isfinite(o).all()
    assert err.max() <= O_MAX, err.max()
    assert err.mean() <= O_MEAN, err.mean()
    fin = np.isfinite(lref)
    assert np.array_equal(np.isfinite(lse), fin)
    assert np.abs(lse[fin] - lref[fin]).max(initial=0) <= LSE_TOL


@pytest.mark.parametrize("G", [1, 4, 8, 16])
@pytest.mark.parametrize("num_splits", [0, 1, 3, 16])
def test_small_against_oracle(fa, G, num_splits):
    Hkv = 2
    P = wl.paged_inputs(5, G * Hkv, Hkv, 128, 1, 1, seed=G * 31 + num_splits,
                        seq_lens=[1, 15, 16, 17, 700])
    o, lse = _run(fa, P, num_splits)
    oref, lref = oracle.paged_decode(P.q, P.k_cache, P.v_cache, P.block_table, P.seq_lens, 16)
    _check(o, lse, oref, lref)


def test_empty_and_long_sequences(fa):
    P = wl.paged_inputs(4, 32, 8, 128, 1, 1, seed=7, seq_lens=[0, 1, 4096, 9000], spare_blocks=3)
    o, lse = _run(fa, P)
    oref, lref = oracle.paged_decode(P.q, P.k_cache, P.v_cache, P.block_table, P.seq_lens, 16)
    _check(o, lse, oref, lref)
    assert np.all(o[0] == 0) and np.all(np.isneginf(lse[0]))


def test_split_count_changes_only_rounding(fa):
    P = wl.paged_inputs(3, 32, 8, 128, 1, 1, seed=9, seq_lens=[3000, 5000, 20000])
    outs = [_run(fa, P, s)[0] for s in (1, 2, 7, 16)]
    for o in outs[1:]:
        assert np.abs(o - outs[0]).max() <= 1e-2


def test_physical_placement_is_bit_exact(fa):
    P = wl.paged_inputs(6, 32, 8, 128, 100, 5000, seed=11)
    o1, l1 = _run(fa, P, 16)
    perm = torch.from_numpy(np.random.default_rng(5).permutation(P.num_blocks))
    inv = torch.argsort(perm)
    bt = P.block_table.clone()
    used = bt >= 0
    bt[used] = inv[bt[used].long()].to(torch.int32)
    P2 = wl.PagedInputs(P.q, P.k_cache[perm], P.v_cache[perm], bt, P.seq_lens, 16)
    o2, l2 = _run(fa, P2, 16)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_entries_past_the_sequence_are_never_read(fa):
    P = wl.paged_inputs(3, 32, 8, 128, 1, 1, seed=13, seq_lens=[40, 100, 17], max_blocks=32)
    o1, l1 = _run(fa, P)
    bt = P.block_table.clone()
    bt[bt < 0] = 2**30  # garbage past each row's last block
    o2, l2 = _run(fa, wl.PagedInputs(P.q, P.k_cache, P.v_cache, bt, P.seq_lens, 16))
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_out_of_range_block_is_skipped_and_reported(fa):
    P = wl.paged_inputs(2, 8, 2, 128, 1, 1, seed=17, seq_lens=[64, 64])
    bt = P.block_table.clone()
    bad = int(bt[1, 2])
    bt[1, 2] = P.num_blocks + 5
    o, lse = _run(fa, wl.PagedInputs(P.q, P.k_cache, P.v_cache, bt, P.seq_lens, 16), expect_status=fa.FA_ERR_BAD_BLOCK_TABLE)
    oref, lref = oracle.paged_decode(P.q, P.k_cache, P.v_cache, P.block_table, P.seq_lens, 16)
    _check(o[:1], lse[:1], oref[:1], lref[:1])
    # sequence 1 behaves as if the keys of logical block 2 were masked
    kc, vc, q = oracle.to_f64(P.k_cache), oracle.to_f64(P.v_cache), oracle.to_f64(P.q)
    keep = np.r_[0:32, 48:64]
    for h in range(8):
        g = h // 4
        K = oracle.gather_paged_keys(kc, P.block_table[1].numpy(), 64, 16, g)[keep]
        V = oracle.gather_paged_keys(vc, P.block_table[1].numpy(), 64, 16, g)[keep]
        Or, Lr = oracle.attention_forward(q[1, h][None, None, None], K[None, None], V[None, None])
        assert np.abs(o[1, h] - Or[0, 0, 0]).max() <= O_MAX
        assert abs(lse[1, h] - Lr[0, 0, 0]) <= LSE_TOL
    assert bad >= 0


def test_full_gqa_decode_config_sampled(fa):
    # batch 64, 32 query heads on 8 KV heads, d 128, L ~ U[512, 32768],
    # 16-token blocks, split into up to 16 chunks (the benchmarked launch)
    P = wl.paged_inputs(64, 32, 8, 128, 512, 32768, seed=wl.config_seed(0, 5), max_blocks=2048)
    o, lse = _run(fa, P, 16)
    rng = np.random.default_rng(0)
    bs = sorted(set([0, 63] + list(rng.choice(64, 4, replace=False))))
    for b in bs:
        sub = _compact(P, b)
        oref, lref = oracle.paged_decode(sub.q, sub.k_cache, sub.v_cache, sub.block_table, sub.seq_lens, 16)
        _check(o[b:b + 1], lse[b:b + 1], oref, lref)


def _plant_retrieval(P, seed, limits):
    """Integer mirror of the gather: q is c * e_0 for every head, every key is
    zero except one target key per (sequence, KV head) whose first coordinate
    is 64, so the target's logit exceeds every other by ~45 and softmax puts
    weight 1 on it to fp32 precision: o must equal that key's V row exactly.
    limits[b] bounds the target's logical position.  Returns the targets."""
    g = torch.Generator().manual_seed(seed)
    B, Hq, d = P.q.shape
    Hkv = P.k_cache.shape[2]
    P.q.zero_()
    P.q[..., 0] = 8.0
    P.k_cache.zero_()
    targets = torch.zeros(B, Hkv, dtype=torch.long)
    for b in range(B):
        for kv in range(Hkv):
            t = int(torch.randint(0, int(limits[b]), (1,), generator=g))
            targets[b, kv] = t
            phys = int(P.block_table[b, t // P.block_size])
            P.k_cache[phys, t % P.block_size, kv, 0] = 64.0
    return targets


def test_gather_retrieves_exact_rows(fa):
    # block-table indexing checked bit for bit: every (sequence, query head)
    # returns exactly the V row its target key maps to through the table
    for bs, num_splits in ((16, 0), (16, 1), (16, 5), (64, 0), (64, 1)):
        P = wl.paged_inputs(6, 16, 4, 128, 1, 1, block_size=bs, seed=21, seq_lens=[1, 16, 17, 333, 4096, 9999])
        tg = _plant_retrieval(P, 5, P.seq_lens.tolist())
        o, lse = _run(fa, P, num_splits)
        G = 16 // 4
        for b in range(6):
            for h in range(16):
                t = int(tg[b, h // G])
                phys = int(P.block_table[b, t // bs])
                want = P.v_cache[phys, t % bs, h // G].float().numpy()
                assert np.array_equal(o[b, h], want), (bs, num_splits, b, h)


@pytest.mark.parametrize("bs", [32, 64, 256])
def test_larger_cache_blocks(fa, bs):
    # blocks of 32..256 tokens are walked as 16-token chunks through the table
    P = wl.paged_inputs(4, 16, 4, 128, 1, 1, block_size=bs, seed=bs, seq_lens=[1, bs - 1, bs + 17, 3000])
    for num_splits in (0, 1, 7):
        o, lse = _run(fa, P, num_splits)
        oref, lref = oracle.paged_decode(P.q, P.k_cache, P.v_cache, P.block_table, P.seq_lens, bs)
        _check(o, lse, oref, lref)


@pytest.mark.parametrize("G", [1, 4, 8])
def test_head_dim_64(fa, G):
    Hkv = 4
    P = wl.paged_inputs(5, G * Hkv, Hkv, 64, 1, 1, seed=40 + G, seq_lens=[0, 1, 17, 700, 5000])
    for num_splits in (0, 1, 3):
        o, lse = _run(fa, P, num_splits)
        oref, lref = oracle.paged_decode(P.q, P.k_cache, P.v_cache, P.block_table, P.seq_lens, 16)
        _check(o, lse, oref, lref)


def test_head_dim_64_exact_retrieval_and_graph(fa):
    P = wl.paged_inputs(3, 8, 2, 64, 1, 1, block_size=32, seed=44, seq_lens=[5, 300, 2000])
    tg = _plant_retrieval(P, 9, P.seq_lens.tolist())
    o, _ = _run(fa, P)
    for b in range(3):
        for h in range(8):
            t = int(tg[b, h // 4])
            want = P.v_cache[int(P.block_table[b, t // 32]), t % 32, h // 4].float().numpy()
            assert np.array_equal(o[b, h], want)
    q, kc, vc, bt, sl = _dev(P)
    layer = (q, kc, vc, torch.empty_like(q), torch.empty(3, 8, dtype=torch.float32, device=q.device))
    g = fa.DecodeGraph([layer], bt, sl)
    g.launch()
    torch.cuda.synchronize()
    assert np.array_equal(layer[3].float().cpu().numpy(), o)
    g.close()
