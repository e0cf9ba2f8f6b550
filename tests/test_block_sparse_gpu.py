"""Block-sparse forward parity: fa_fwd_block_sparse through the C ABI against
the fp64 block-sparse oracle on the same seeded bf16 inputs and masks.
Tolerances are the forward ones: O max-abs <= 2e-2 and mean-abs <= 2e-3,
LSE abs <= 1e-3.  An all-kept mask must reproduce the dense kernel bit for
bit (same tiles, same arithmetic)."""
import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_10_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_TOL = 2e-2, 2e-3, 1e-3

# the masks the kernel is measured on: butterfly plus a local window of 15
# key blocks before the diagonal, at N = 16384 and 65536 (H=16, d=128, causal)
BENCH_WINDOW = 15


def _run(fa, x, mask, causal, kv_lens=None, scale=None):
    dev = torch.device("cuda")
    kv = None if kv_lens is None else kv_lens.to(dev)
    O, L = fa.fa_fwd_block_sparse(x.Q.to(dev), x.K.to(dev), x.V.to(dev), mask.to(dev), causal=causal,
                                  kv_lens=kv, scale=scale)
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
@pytest.mark.parametrize("N", [300, 1000])
def test_random_shared_masks(fa, N, d, causal):
    nb = (N + 127) // 128
    x = wl.dense_inputs(1, 3, N, d, seed=N + d)
    m = wl.block_mask(nb, "random", p=0.4, seed=N)
    O, L = _run(fa, x, m, causal)
    Oref, Lref = oracle.block_sparse_forward(x.Q, x.K, x.V, m.numpy(), causal=causal)
    _check(O, L, Oref, Lref)


def test_per_head_masks_with_key_padding(fa):
    B, H, N, d = 2, 3, 700, 128
    nb = (N + 127) // 128
    x = wl.dense_inputs(B, H, N, d, seed=5)
    m = wl.block_mask(nb, "random", p=0.3, seed=6, heads=(B, H))
    kv = torch.tensor([700, 333], dtype=torch.int32)
    for causal in (False, True):
        O, L = _run(fa, x, m, causal, kv_lens=kv)
        Oref, Lref = oracle.block_sparse_forward(x.Q, x.K, x.V, m.numpy(), causal=causal, kv_lens=kv.numpy())
        _check(O, L, Oref, Lref)


def test_query_tile_with_no_kept_block(fa):
    # query block 2 keeps nothing (its CTA partner, block 3, keeps blocks):
    # its rows are empty; block 0 keeps only key block 3 (past its causal range)
    N, nb = 512, 4
    x = wl.dense_inputs(1, 2, N, 64, seed=7)
    m = torch.ones(nb, nb, dtype=torch.uint8)
    m[2] = 0
    m[0] = torch.tensor([0, 0, 0, 1], dtype=torch.uint8)
    for causal in (False, True):
        O, L = _run(fa, x, m, causal)
        Oref, Lref = oracle.block_sparse_forward(x.Q, x.K, x.V, m.numpy(), causal=causal)
        _check(O, L, Oref, Lref)
        assert np.all(O[:, :, 256:384] == 0) and np.all(np.isneginf(L[:, :, 256:384]))


def test_all_kept_mask_equals_dense_bitwise(fa):
    N = 1000
    nb = (N + 127) // 128
    x = wl.dense_inputs(2, 2, N, 128, seed=8)
    dev = torch.device("cuda")
    for causal in (False, True):
        O, L = _run(fa, x, torch.ones(nb, nb, dtype=torch.uint8), causal)
        Od, Ld = fa.fa_fwd(x.Q.to(dev), x.K.to(dev), x.V.to(dev), causal=causal)
        torch.cuda.synchronize()
        assert np.array_equal(O, Od.float().cpu().numpy())
        assert np.array_equal(L, Ld.cpu().numpy())


def test_butterfly_mask_custom_scale(fa):
    N = 1536
    x = wl.dense_inputs(1, 2, N, 128, seed=9)
    m = wl.block_mask(N // 128, "butterfly", window=1)
    O, L = _run(fa, x, m, True, scale=0.05)
    Oref, Lref = oracle.block_sparse_forward(x.Q, x.K, x.V, m.numpy(), causal=True, scale=0.05)
    _check(O, L, Oref, Lref)


@pytest.mark.parametrize("N", [16384, 65536])
def test_bench_masks_sampled_rows(fa, N):
    # the measured masks at full size: sampled rows of the first and last head
    B, H, d = 1, 16, 128
    x = wl.dense_inputs(B, H, N, d, seed=wl.config_seed(0, 4))
    m = wl.block_mask(N // 128, "butterfly", window=BENCH_WINDOW)
    O, L = _run(fa, x, m, True)
    rows = np.unique(np.concatenate([np.arange(0, N, 1021), [127, 128, N - 1]]))
    for h in (0, H - 1):
        xs = [t[:, h:h + 1] for t in (x.Q, x.K, x.V)]
        Oref, Lref = oracle.block_sparse_forward(*xs, m.numpy(), causal=True, rows=rows)
        _check(O[0, h][rows], L[0, h][rows], Oref[0, 0], Lref[0, 0])


def test_deterministic(fa):
    N = 900
    x = wl.dense_inputs(1, 2, N, 128, seed=10)
    m = wl.block_mask(8, "random", p=0.5, seed=11)
    a = _run(fa, x, m, True)
    b = _run(fa, x, m, True)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
