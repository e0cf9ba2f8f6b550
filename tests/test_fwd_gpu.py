"""Forward parity: the CUDA path (through the C ABI) against the fp64 oracle on
the same seeded bf16 inputs.  Tolerances: O max-abs <= 2e-2 and mean-abs
<= 2e-3, LSE abs <= 1e-3 (bf16 inputs, fp32 accumulation)."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_10_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_TOL = 2e-2, 2e-3, 1e-3


def _run(fa, x, causal, kv_lens=None, scale=None):
    dev = torch.device("cuda")
    kv = None if kv_lens is None else kv_lens.to(dev)
    O, L = fa.fa_fwd(x.Q.to(dev), x.K.to(dev), x.V.to(dev), causal=causal, kv_lens=kv, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    return O.float().cpu().numpy(), L.cpu().numpy()


def _check(O, L, Oref, Lref, v_std=1.0):
    # the O bounds are stated for unit-variance values; they scale with |V|
    err = np.abs(O - Oref)
    assert np.isfinite(O).all()
    assert err.max() <= O_MAX * v_std, err.max()
    assert err.mean() <= O_MEAN * v_std, err.mean()
    fin = np.isfinite(Lref)
    assert np.array_equal(np.isfinite(L), fin)
    assert np.abs(L[fin] - Lref[fin]).max(initial=0) <= LSE_TOL


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_tiny_config(fa, causal, d):
    x = wl.dense_inputs(1, 2, 256, d, seed=0)
    O, L = _run(fa, x, causal)
    Oref, Lref = oracle.attention_forward(x.Q, x.K, x.V, causal=causal)
    _check(O, L, Oref, Lref)


@pytest.mark.parametrize("N", [1, 2, 17, 127, 128, 129, 255, 300, 513])
@pytest.mark.parametrize("causal", [False, True])
def test_ragged_lengths(fa, N, causal):
    x = wl.dense_inputs(2, 3, N, 64, seed=N)
    O, L = _run(fa, x, causal)
    Oref, Lref = oracle.attention_forward(x.Q, x.K, x.V, causal=causal)
    _check(O, L, Oref, Lref)


@pytest.mark.parametrize("N", [1, 200, 384])
def test_ragged_lengths_d128(fa, N):
    x = wl.dense_inputs(1, 2, N, 128, seed=N + 7)
    for causal in (False, True):
        O, L = _run(fa, x, causal)
        Oref, Lref = oracle.attention_forward(x.Q, x.K, x.V, causal=causal)
        _check(O, L, Oref, Lref)


def test_key_padding_bert_shape(fa):
    B, H, N, d = 16, 16, 512, 64
    kv = wl.padded_lengths(B, 128, 512, seed=wl.config_seed(0, 2))
    x = wl.dense_inputs(B, H, N, d, seed=wl.config_seed(0, 2))
    O, L = _run(fa, x, False, kv_lens=kv)
    Oref, Lref = oracle.attention_forward(x.Q, x.K, x.V, causal=False, kv_lens=kv.numpy())
    _check(O, L, Oref, Lref)


def test_key_padding_edge_lengths(fa):
    # lengths 0 (every row empty), 1, a tile boundary and a ragged tail
    kv = torch.tensor([0, 1, 128, 129, 200, 256], dtype=torch.int32)
    x = wl.dense_inputs(6, 2, 256, 64, seed=5)
    for causal in (False, True):
        O, L = _run(fa, x, causal, kv_lens=kv)
        Oref, Lref = oracle.attention_forward(x.Q, x.K, x.V, causal=causal, kv_lens=kv.numpy())
        _check(O, L, Oref, Lref)
        assert np.all(O[0] == 0) and np.all(np.isneginf(L[0]))


def test_boosted_logits_exercise_rescaling(fa):
    x = wl.boosted_inputs(2, 4, 1024, 64, seed=wl.config_seed(0, 3))
    O, L = _run(fa, x, True)
    Oref, Lref = oracle.attention_forward(x.Q, x.K, x.V, causal=True)
    _check(O, L, Oref, Lref)


def test_large_logits_and_custom_scale(fa):
    # std 3 and scale 1 give logits of magnitude ~100: every tile moves the max
    x = wl.dense_inputs(1, 2, 640, 64, seed=11, std=3.0)
    for causal in (False, True):
        O, L = _run(fa, x, causal, scale=1.0)
        Oref, Lref = oracle.attention_forward(x.Q, x.K, x.V, causal=causal, scale=1.0)
        _check(O, L, Oref, Lref, v_std=3.0)


def test_deterministic(fa):
    x = wl.dense_inputs(2, 2, 700, 128, seed=3)
    a = _run(fa, x, True)
    b = _run(fa, x, True)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_gpt2_medium_4k_sampled_heads(fa):
    B, H, N, d = 8, 16, 4096, 64
    x = wl.boosted_inputs(B, H, N, d, seed=wl.config_seed(0, 3))
    O, L = _run(fa, x, True)
    heads = [(0, 0), (3, 7), (7, 15)]
    rows = np.arange(N)
    Oref, Lref = oracle.attention_forward_rows(x.Q, x.K, x.V, rows, causal=True, heads=heads)
    for t, (b, h) in enumerate(heads):
        _check(O[b, h], L[b, h], Oref[t], Lref[t])


@pytest.mark.parametrize("N", [16384, 65536])
def test_long_context_sampled_rows(fa, N):
    B, H, d = 1, 16, 128
    x = wl.dense_inputs(B, H, N, d, seed=wl.config_seed(0, 4))
    O, L = _run(fa, x, True)
    rows = np.unique(np.concatenate([np.arange(0, N, 509), [N - 1, 127, 128, N - 128]]))
    heads = [(0, 0), (0, H - 1)]
    Oref, Lref = oracle.attention_forward_rows(x.Q, x.K, x.V, rows, causal=True, heads=heads)
    for t, (b, h) in enumerate(heads):
        _check(O[b, h][rows], L[b, h][rows], Oref[t], Lref[t])


@pytest.mark.parametrize("causal", [True, False])
def test_longest_sequence_sampled_rows(fa, causal):
    """The largest single-sequence case the suite runs: N = 262144 (N^2 > 2^31,
    2048 query tiles per head), checked on rows sampled across the whole
    sequence, the first and last tiles and a tile boundary."""
    B, H, N, d = 1, 2, 262144, 128
    x = wl.dense_inputs(B, H, N, d, seed=wl.config_seed(0, 4) + 7)
    O, L = _run(fa, x, causal)
    rows = np.unique(np.concatenate([np.arange(0, N, 8191), [0, 127, 128, N - 129, N - 128, N - 1]]))
    heads = [(0, 0), (0, H - 1)]
    Oref, Lref = oracle.attention_forward_rows(x.Q, x.K, x.V, rows, causal=causal, heads=heads)
    for t, (b, h) in enumerate(heads):
        _check(O[b, h][rows], L[b, h][rows], Oref[t], Lref[t])
