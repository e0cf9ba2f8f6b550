"""Decode step as one CUDA graph: replaying the recorded paged decodes must
give exactly the eager calls' results (the same kernels on the same
buffers), follow the buffers' new contents between launches, and refuse
invalid calls at creation without leaving an error behind.  The fused
single-split path is checked against the oracle and against the split path."""
import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_10_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _layers(n, B=4, Hq=32, Hkv=8, seq_lens=(1, 100, 2048, 5000), seed=0):
    dev = torch.device("cuda")
    P = wl.paged_inputs(B, Hq, Hkv, 128, 1, 1, seed=seed, seq_lens=list(seq_lens))
    layers = []
    for i in range(n):
        Pi = wl.paged_inputs(B, Hq, Hkv, 128, 1, 1, seed=seed + 100 + i, seq_lens=list(seq_lens))
        q, kc, vc = (t.to(dev) for t in (Pi.q, Pi.k_cache, Pi.v_cache))
        layers.append((q, kc, vc, torch.empty_like(q), torch.empty(B, Hq, dtype=torch.float32, device=dev)))
    return layers, P.block_table.to(dev), P.seq_lens.to(dev)


@pytest.mark.parametrize("num_splits", [0, 1])
def test_graph_replay_equals_eager_calls(fa, num_splits):
    layers, bt, sl = _layers(3)
    g = fa.DecodeGraph(layers, bt, sl, num_splits=num_splits)
    assert g.kernel_count == 3 * (1 if num_splits == 1 else 2)
    g.launch()
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    for q, kc, vc, o, lse in layers:
        oe, le = fa.fa_paged_decode(q, kc, vc, bt, sl, num_splits=num_splits)
        torch.cuda.synchronize()
        assert torch.equal(o, oe) and torch.equal(lse, le)
    g.close()


def test_graph_follows_new_contents(fa):
    layers, bt, sl = _layers(2, seq_lens=(10, 300, 4000, 4095))
    g = fa.DecodeGraph(layers, bt, sl)
    for step in range(3):
        # a new query per layer and a different visible length per sequence
        # (shorter, so every length stays inside the sequence's blocks)
        for i, (q, *_rest) in enumerate(layers):
            q.copy_(wl.device_normal_bf16(q.shape, 1000 * step + i, q.device))
        sl.sub_(1)
        g.launch()
        torch.cuda.synchronize()
        assert fa.fa_get_device_status() == fa.FA_OK
        for q, kc, vc, o, lse in layers:
            oe, le = fa.fa_paged_decode(q, kc, vc, bt, sl)
            torch.cuda.synchronize()
            assert torch.equal(o, oe) and torch.equal(lse, le)
    g.close()


def test_single_split_matches_oracle_and_split_path(fa):
    P = wl.paged_inputs(6, 16, 4, 128, 1, 1, seed=3, seq_lens=[0, 1, 16, 17, 511, 3000])
    dev = torch.device("cuda")
    q, kc, vc, bt, sl = (t.to(dev) for t in (P.q, P.k_cache, P.v_cache, P.block_table, P.seq_lens))
    o1, l1 = fa.fa_paged_decode(q, kc, vc, bt, sl, num_splits=1)
    o16, l16 = fa.fa_paged_decode(q, kc, vc, bt, sl, num_splits=16)
    torch.cuda.synchronize()
    oref, lref = oracle.paged_decode(P.q, P.k_cache, P.v_cache, P.block_table, P.seq_lens, 16)
    o1n, l1n = o1.float().cpu().numpy(), l1.cpu().numpy()
    assert np.abs(o1n - oref).max() <= 2e-2 and np.abs(o1n - oref).mean() <= 2e-3
    fin = np.isfinite(lref)
    assert np.array_equal(np.isfinite(l1n), fin) and np.abs(l1n[fin] - lref[fin]).max() <= 1e-3
    assert np.abs(o1n - o16.float().cpu().numpy()).max() <= 2e-2


def test_invalid_call_is_refused_at_creation(fa):
    layers, bt, sl = _layers(2)
    bad = [layers[0], (layers[1][0], layers[1][1], layers[1][2], layers[1][3], layers[1][4])]
    with pytest.raises(fa.FAError) as e:
        fa.DecodeGraph(bad, bt, sl, num_splits=17)  # outside 0..16
    assert e.value.status == fa.FA_ERR_UNSUPPORTED
    # nothing was left behind: the context still runs eager and graph decodes
    g = fa.DecodeGraph(layers, bt, sl)
    g.launch()
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    g.close()
