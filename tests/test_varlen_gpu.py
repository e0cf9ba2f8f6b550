"""Packed ragged-batch (varlen) forward parity: fa_fwd_varlen through the C ABI
against the fp64 oracle's per-sequence attention on the same seeded bf16
inputs.  Tolerances are the forward ones: O max-abs <= 2e-2 and mean-abs
<= 2e-3, LSE abs <= 1e-3 (bf16 inputs, fp32 accumulation).  Properties that
hold at any size (packed == dense bit for bit, and packed == the key-padding
mask on the valid rows) cover the full-size workloads."""
import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_10_gb300 import workloads as wl
from gradcheck import check_grads, packed_slices

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_TOL = 2e-2, 2e-3, 1e-3

# the length mixes the varlen forward is measured on: the BERT-large-shaped
# padded configuration's lengths (H=16, d=64, non-causal) and a long-context
# prefill mix (H=16, d=128, causal)
BERT_LENGTHS = dict(B=16, lo=128, hi=512)
LONG_LENGTHS = dict(num_seqs=16, lo=512, hi=16384)


def _run(fa, x, causal, max_seqlen=None, scale=None):
    dev = torch.device("cuda")
    O, L = fa.fa_fwd_varlen(x.Q.to(dev), x.K.to(dev), x.V.to(dev), x.cu_seqlens.to(dev),
                            x.max_seqlen if max_seqlen is None else max_seqlen, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    return O.float().cpu().numpy(), L.cpu().numpy()


def _check(O, L, Oref, Lref):
    err = np.abs(O - Oref)
    assert np.isfinite(O).all()
    assert err.max(initial=0) <= O_MAX, err.max()
    assert err.mean() <= O_MEAN, err.mean()
    fin = np.isfinite(Lref)
    assert np.array_equal(np.isfinite(L), fin)
    assert np.abs(L[fin] - Lref[fin]).max(initial=0) <= LSE_TOL


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_edge_lengths(fa, d, causal):
    # empty sequences (first, middle, last), a single token, tile boundaries
    # (128, 256), ragged tails and a sequence spanning several tile pairs
    lens = [0, 1, 17, 128, 129, 0, 300, 1000, 256, 0]
    x = wl.varlen_inputs(lens, 3, d, seed=11 + d)
    O, L = _run(fa, x, causal)
    Oref, Lref = oracle.attention_forward_varlen(x.Q, x.K, x.V, x.cu_seqlens, causal=causal)
    _check(O, L, Oref, Lref)


def test_single_sequence_and_loose_max_seqlen(fa):
    # one sequence, and a max_seqlen larger than needed (extra grid rows exit)
    x = wl.varlen_inputs([777], 2, 128, seed=4)
    for causal in (False, True):
        O, L = _run(fa, x, causal, max_seqlen=2000)
        Oref, Lref = oracle.attention_forward_varlen(x.Q, x.K, x.V, x.cu_seqlens, causal=causal)
        _check(O, L, Oref, Lref)


def test_custom_scale(fa):
    x = wl.varlen_inputs([50, 200, 3], 2, 64, seed=8)
    O, L = _run(fa, x, True, scale=0.3)
    Oref, Lref = oracle.attention_forward_varlen(x.Q, x.K, x.V, x.cu_seqlens, causal=True, scale=0.3)
    _check(O, L, Oref, Lref)


def test_packed_equals_dense_bitwise(fa):
    # B equal-length sequences packed [B*N, H, d] give exactly the dense
    # [B, H, N, d] kernel's results: same tiles, same order, masked keys
    # contribute exact zeros whichever rows the tile holds
    B, H, N, d = 3, 4, 333, 128
    x = wl.varlen_inputs([N] * B, H, d, seed=21)
    dev = torch.device("cuda")
    for causal in (False, True):
        O, L = _run(fa, x, causal)
        dense = [t.reshape(B, N, H, d).permute(0, 2, 1, 3).contiguous().to(dev) for t in (x.Q, x.K, x.V)]
        Od, Ld = fa.fa_fwd(*dense, causal=causal)
        torch.cuda.synchronize()
        Od = Od.permute(0, 2, 1, 3).reshape(B * N, H, d).float().cpu().numpy()
        Ld = Ld.permute(1, 0, 2).reshape(H, B * N).cpu().numpy()
        assert np.array_equal(O, Od)
        assert np.array_equal(L, Ld)


def test_bert_lengths_match_key_padding(fa):
    # the BERT-large-shaped padded workload: packing the valid tokens gives the
    # key-padding kernel's values on every valid row, bit for bit
    H, d, Npad = 16, 64, 512
    lens = wl.padded_lengths(**BERT_LENGTHS, seed=wl.config_seed(0, 2)).tolist()
    x = wl.varlen_inputs(lens, H, d, seed=wl.config_seed(0, 2))
    O, L = _run(fa, x, False)
    cu = x.cu_seqlens.tolist()
    B = len(lens)
    dev = torch.device("cuda")
    dense = []
    for t in (x.Q, x.K, x.V):
        z = torch.zeros(B, H, Npad, d, dtype=torch.bfloat16)
        for s in range(B):
            z[s, :, :lens[s]] = t[cu[s]:cu[s + 1]].permute(1, 0, 2)
        dense.append(z.to(dev))
    Od, Ld = fa.fa_fwd(*dense, causal=False, kv_lens=torch.tensor(lens, dtype=torch.int32, device=dev))
    torch.cuda.synchronize()
    Od, Ld = Od.float().cpu().numpy(), Ld.cpu().numpy()
    for s in range(B):
        assert np.array_equal(O[cu[s]:cu[s + 1]], Od[s, :, :lens[s]].transpose(1, 0, 2))
        assert np.array_equal(L[:, cu[s]:cu[s + 1]], Ld[s, :, :lens[s]])
    # and two whole sequences against the oracle
    for s in (0, B - 1):
        a, b = cu[s], cu[s + 1]
        Oref, Lref = oracle.attention_forward_varlen(x.Q[a:b], x.K[a:b], x.V[a:b], [0, b - a])
        _check(O[a:b], L[:, a:b], Oref, Lref)


def test_long_mix_sampled_rows(fa):
    # the long-context mix at full size, in the launch bench.py times:
    # sampled rows of the first, a middle and the last sequence, two heads each
    H, d = 16, 128
    lens = wl.varlen_lengths(**LONG_LENGTHS, seed=wl.config_seed(0, 6))
    x = wl.varlen_inputs(lens, H, d, seed=wl.config_seed(0, 6))
    O, L = _run(fa, x, True)
    cu = x.cu_seqlens.tolist()
    for s in (0, len(lens) // 2, len(lens) - 1):
        a, n = cu[s], lens[s]
        rows = np.unique(np.concatenate([np.arange(0, n, 397), [0, 127, 128, n - 1]]))
        rows = rows[rows < n]
        q, k, v = (t[a:a + n].permute(1, 0, 2)[None] for t in (x.Q, x.K, x.V))
        heads = [(0, 0), (0, H - 1)]
        Oref, Lref = oracle.attention_forward_rows(q, k, v, rows, causal=True, heads=heads)
        for t, (_, h) in enumerate(heads):
            _check(O[a + rows, h], L[h, a + rows], Oref[t], Lref[t])


def test_device_side_bad_offsets_are_reported(fa):
    # a sequence longer than max_seqlen, and offsets running past total, are
    # found on the device: that sequence is left unwritten, the others are
    # computed, and the status word reports FA_ERR_INVALID_ARG
    x = wl.varlen_inputs([100, 300, 50], 2, 64, seed=31)
    dev = torch.device("cuda")
    Q, K, V = (t.to(dev) for t in (x.Q, x.K, x.V))
    Oref, Lref = oracle.attention_forward_varlen(x.Q, x.K, x.V, x.cu_seqlens, causal=True)
    O = torch.full_like(Q, 7.0)
    fa.fa_fwd_varlen(Q, K, V, x.cu_seqlens.to(dev), 256, causal=True, O=O)
    assert fa.fa_get_device_status() == fa.FA_ERR_INVALID_ARG
    On = O.float().cpu().numpy()
    assert (On[100:400] == 7.0).all()
    _check(On[:100], np.zeros(0), Oref[:100], np.zeros(0))
    _check(On[400:], np.zeros(0), Oref[400:], np.zeros(0))
    cu_bad = torch.tensor([0, 100, 400, 460], dtype=torch.int32, device=dev)  # ends past total = 450
    O2 = torch.full_like(Q, 7.0)
    fa.fa_fwd_varlen(Q, K, V, cu_bad, 300, causal=True, O=O2)
    assert fa.fa_get_device_status() == fa.FA_ERR_INVALID_ARG
    assert (O2[400:].float() == 7.0).all()
    # the context is still usable and the status word was cleared
    O3, L3 = _run(fa, x, True)
    _check(O3, L3, Oref, Lref)


def test_deterministic(fa):
    x = wl.varlen_inputs([5, 700, 129, 1], 2, 128, seed=3)
    a = _run(fa, x, True)
    b = _run(fa, x, True)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# ---------------------------------------------------------------- backward


def _bwd(fa, x, causal, max_seqlen=None):
    dev = torch.device("cuda")
    Q, K, V, dO, cu = (t.to(dev) for t in (x.Q, x.K, x.V, x.dO, x.cu_seqlens))
    ms = x.max_seqlen if max_seqlen is None else max_seqlen
    O, L = fa.fa_fwd_varlen(Q, K, V, cu, ms, causal=causal)
    grads = fa.fa_bwd_varlen(Q, K, V, O, dO, L, cu, ms, causal=causal)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    return [g.float().cpu().numpy() for g in grads]


def _check_grads(grads, refs, cu_seqlens):
    """Per (sequence, head): relative L2 <= 1e-2 and the largest element error
    <= 2e-2 of the slice's largest element (tests/gradcheck.py)."""
    H = np.asarray(refs[0]).shape[1]
    check_grads(grads, refs, packed_slices(cu_seqlens, H))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_backward_edge_lengths(fa, d, causal):
    lens = [1, 17, 0, 128, 129, 300, 1000, 256]
    x = wl.varlen_inputs(lens, 3, d, seed=50 + d)
    grads = _bwd(fa, x, causal)
    refs = oracle.attention_backward_varlen(x.Q, x.K, x.V, x.dO, x.cu_seqlens, causal=causal)
    _check_grads(grads, refs, x.cu_seqlens.tolist())


def test_backward_packed_equals_dense(fa):
    # equal-length sequences: dK and dV are bit-identical to the dense
    # backward (same tiles, rows of other sequences contribute exact zeros);
    # dQ is summed by reductions whose order varies, so it is compared in norm
    B, H, N, d = 3, 4, 333, 128
    x = wl.varlen_inputs([N] * B, H, d, seed=61)
    dev = torch.device("cuda")
    for causal in (False, True):
        gv = _bwd(fa, x, causal)
        dense = [t.reshape(B, N, H, d).permute(0, 2, 1, 3).contiguous().to(dev) for t in (x.Q, x.K, x.V, x.dO)]
        O, L = fa.fa_fwd(*dense[:3], causal=causal)
        gd = fa.fa_bwd(*dense[:3], O, dense[3], L, causal=causal)
        torch.cuda.synchronize()
        gd = [g.permute(0, 2, 1, 3).reshape(B * N, H, d).float().cpu().numpy() for g in gd]
        assert np.array_equal(gv[1], gd[1]) and np.array_equal(gv[2], gd[2])
        assert np.linalg.norm(gv[0] - gd[0]) <= 1e-3 * np.linalg.norm(gd[0])


def test_backward_long_mix_two_sequences(fa):
    # a mix of long sequences; the shortest and the longest are checked in full
    lens = [512, 4096, 1500, 2900, 700, 3333]
    H, d = 4, 128
    x = wl.varlen_inputs(lens, H, d, seed=62)
    grads = _bwd(fa, x, True)
    cu = x.cu_seqlens.tolist()
    for s in (0, 1):
        a, b = cu[s], cu[s + 1]
        refs = oracle.attention_backward_varlen(x.Q[a:b], x.K[a:b], x.V[a:b], x.dO[a:b], [0, b - a], causal=True)
        _check_grads([g[a:b] for g in grads], refs, [0, b - a])


@pytest.mark.parametrize("d", [64, 128])
def test_backward_short_sequences_inside_a_long_mix(fa, d):
    # one-token, one-tile and ragged short sequences between long ones, with
    # H = 6 so the last group of four (sequence, head) pairs is partly filled;
    # every sequence and head is judged on its own
    lens = [3000, 1, 128, 2048, 17, 700, 129]
    x = wl.varlen_inputs(lens, 6, d, seed=64 + d)
    for causal in (True, False):
        grads = _bwd(fa, x, causal)
        refs = oracle.attention_backward_varlen(x.Q, x.K, x.V, x.dO, x.cu_seqlens, causal=causal)
        _check_grads(grads, refs, x.cu_seqlens.tolist())


def test_backward_bad_offsets_are_reported(fa):
    x = wl.varlen_inputs([100, 50], 2, 64, seed=63)
    dev = torch.device("cuda")
    Q, K, V, dO = (t.to(dev) for t in (x.Q, x.K, x.V, x.dO))
    cu = x.cu_seqlens.to(dev)
    O, L = fa.fa_fwd_varlen(Q, K, V, cu, 100, causal=True)
    bad = torch.tensor([0, 100, 140], dtype=torch.int32, device=dev)  # ends before total = 150
    fa.fa_bwd_varlen(Q, K, V, O, dO, L, bad, 100, causal=True)
    assert fa.fa_get_device_status() == fa.FA_ERR_INVALID_ARG
    # the context is still usable
    grads = _bwd(fa, x, True)
    refs = oracle.attention_backward_varlen(x.Q, x.K, x.V, x.dO, x.cu_seqlens, causal=True)
    _check_grads(grads, refs, x.cu_seqlens.tolist())
