"""Backward parity: forward + backward through the C ABI against the fp64
oracle's analytic gradients on the same seeded inputs.  Tolerance, per
(batch entry, head) of dQ, dK and dV: relative L2 error <= 1e-2 and the
largest element error <= 2e-2 of the slice's largest element (bf16 inputs,
fp32 accumulation; tests/gradcheck.py states the bounds and their floor)."""
import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_10_gb300 import workloads as wl
from gradcheck import check_grads, dense_slices

pytestmark = pytest.mark.gpu


def _rel(a, b):
    den = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (den if den > 0 else 1.0)


def _run(fa, x, causal, kv_lens=None, scale=None):
    dev = torch.device("cuda")
    Q, K, V, dO = (t.to(dev) for t in (x.Q, x.K, x.V, x.dO))
    kv = None if kv_lens is None else kv_lens.to(dev)
    O, L = fa.fa_fwd(Q, K, V, causal=causal, kv_lens=kv, scale=scale)
    dQ, dK, dV = fa.fa_bwd(Q, K, V, O, dO, L, causal=causal, kv_lens=kv, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    return tuple(t.float().cpu().numpy() for t in (dQ, dK, dV))


def _check(got, ref):
    B, H = np.asarray(ref[0]).shape[:2]
    check_grads(got, ref, dense_slices(B, H))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_tiny_config(fa, causal, d):
    x = wl.dense_inputs(1, 2, 256, d, seed=0)
    got = _run(fa, x, causal)
    ref = oracle.attention_backward(x.Q, x.K, x.V, x.dO, causal=causal)
    _check(got, ref)


@pytest.mark.parametrize("N", [1, 17, 128, 129, 300, 513])
@pytest.mark.parametrize("causal", [False, True])
def test_ragged_lengths(fa, N, causal):
    x = wl.dense_inputs(2, 2, N, 64, seed=100 + N)
    got = _run(fa, x, causal)
    ref = oracle.attention_backward(x.Q, x.K, x.V, x.dO, causal=causal)
    _check(got, ref)


@pytest.mark.parametrize("N", [200, 384])
def test_ragged_lengths_d128(fa, N):
    x = wl.dense_inputs(1, 2, N, 128, seed=200 + N)
    for causal in (False, True):
        got = _run(fa, x, causal)
        ref = oracle.attention_backward(x.Q, x.K, x.V, x.dO, causal=causal)
        _check(got, ref)


@pytest.mark.parametrize("B,H", [(1, 6), (2, 3), (1, 5)])
@pytest.mark.parametrize("d", [64, 128])
def test_head_group_tail(fa, B, H, d):
    # the backward grid runs over groups of four (batch, head) pairs: B*H = 6
    # and 5 leave a partly filled last group
    x = wl.dense_inputs(B, H, 300, d, seed=300 + 10 * B + H + d)
    for causal in (False, True):
        got = _run(fa, x, causal)
        ref = oracle.attention_backward(x.Q, x.K, x.V, x.dO, causal=causal)
        _check(got, ref)


def test_key_padding_bert_shape(fa):
    B, H, N, d = 16, 16, 512, 64
    kv = wl.padded_lengths(B, 128, 512, seed=wl.config_seed(0, 2))
    x = wl.dense_inputs(B, H, N, d, seed=wl.config_seed(0, 2))
    got = _run(fa, x, False, kv_lens=kv)
    ref = oracle.attention_backward(x.Q, x.K, x.V, x.dO, causal=False, kv_lens=kv.numpy())
    _check(got, ref)
    for b in range(B):
        L = int(kv[b])
        assert np.all(got[1][b, :, L:] == 0) and np.all(got[2][b, :, L:] == 0)


def test_key_padding_edge_lengths(fa):
    kv = torch.tensor([0, 1, 127, 128, 129, 256], dtype=torch.int32)
    x = wl.dense_inputs(6, 2, 256, 64, seed=6)
    for causal in (False, True):
        got = _run(fa, x, causal, kv_lens=kv)
        ref = oracle.attention_backward(x.Q, x.K, x.V, x.dO, causal=causal, kv_lens=kv.numpy())
        for b in range(6):
            sub = tuple(g[b:b + 1] for g in got)
            refb = tuple(r[b:b + 1] for r in ref)
            if int(kv[b]) == 0:
                assert all(np.all(s == 0) for s in sub)
            else:
                _check(sub, refb)


def test_gpt2_medium_1k_boosted(fa):
    x = wl.boosted_inputs(8, 16, 1024, 64, seed=wl.config_seed(0, 3))
    got = _run(fa, x, True)
    ref = oracle.attention_backward(x.Q, x.K, x.V, x.dO, causal=True)
    _check(got, ref)


def test_gpt2_medium_4k_sampled_heads(fa):
    x = wl.boosted_inputs(8, 16, 4096, 64, seed=wl.config_seed(0, 3) + 1)
    got = _run(fa, x, True)
    for b, h in [(0, 0), (7, 15)]:
        ref = oracle.attention_backward(x.Q[b:b + 1, h:h + 1], x.K[b:b + 1, h:h + 1], x.V[b:b + 1, h:h + 1],
                                        x.dO[b:b + 1, h:h + 1], causal=True)
        _check(tuple(g[b:b + 1, h:h + 1] for g in got), ref)


def test_long_context_16k_sampled_head(fa):
    x = wl.dense_inputs(1, 16, 16384, 128, seed=wl.config_seed(0, 4))
    got = _run(fa, x, True)
    h = 15
    ref = oracle.attention_backward(x.Q[:, h:h + 1], x.K[:, h:h + 1], x.V[:, h:h + 1], x.dO[:, h:h + 1], causal=True)
    _check(tuple(g[:, h:h + 1] for g in got), ref)


def test_deterministic_dk_dv(fa):
    # dK and dV are written once per key tile (no atomics): bit-identical reruns
    x = wl.dense_inputs(1, 2, 640, 128, seed=8)
    a = _run(fa, x, True)
    b = _run(fa, x, True)
    assert np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])
    assert _rel(a[0], b[0]) <= 1e-6
