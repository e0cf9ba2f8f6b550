"""fa_paged_decode_noalloc: the decode entry point for callers that cannot
allocate device memory (e.g. engine plugins whose memory is assigned ahead of
time, or serving loops that avoid cudaMalloc/cudaFree because those can
synchronise the device).  Its split partials live in a fixed array inside the
library instead of a caller workspace.  These tests call it through the C ABI
and compare it with fa_paged_decode (caller workspace) and with the fp64
oracle within the decode tolerances, on calls in a row with different inputs,
so that leftovers of one call in the shared array cannot leak into the next.
One case fills the array exactly (B * Hq * splits = 32768 partial states,
the decode benchmark's shape at a shorter context), one runs d = 64 with
32-token cache blocks.

The file is named to be collected last."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_10_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_TOL = 2e-2, 2e-3, 1e-3
MAX_STATES = 32768


def _dev(P):
    d = torch.device("cuda")
    return P.q.to(d), P.k_cache.to(d), P.v_cache.to(d), P.block_table.to(d), P.seq_lens.to(d)


def _raw_noalloc(so, q, kc, vc, bt, sl, o, lse, num_splits):
    B, Hq, d = q.shape
    NB, bs, Hkv, _ = kc.shape
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return so.fa_paged_decode_noalloc(p(q), p(kc), p(vc), p(bt), p(sl), p(o), p(lse), B, Hq, Hkv, d, bs,
                                      int(bt.shape[1]), NB, num_splits, 1.0 / np.sqrt(d), stream)


def _check(o, lse, oref, lref):
    err = np.abs(o - oref)
    assert np.isfinite(o).all()
    assert err.max() <= O_MAX, err.max()
    assert err.mean() <= O_MEAN, err.mean()
    fin = np.isfinite(lref)
    assert np.array_equal(np.isfinite(lse), fin)
    assert np.abs(lse[fin] - lref[fin]).max(initial=0) <= LSE_TOL


def _cases():
    return [
        # (inputs, num_splits)
        (wl.paged_inputs(8, 32, 8, 128, 1, 3000, seed=21), 16),
        (wl.paged_inputs(5, 16, 4, 128, 1, 1, seed=22, seq_lens=[0, 17, 900, 16, 2500]), 3),
        # exactly the array's capacity: 64 * 32 * 16 = 32768 states
        (wl.paged_inputs(64, 32, 8, 128, 1, 600, seed=24), 16),
        # head dimension 64, 32-token cache blocks
        (wl.paged_inputs(6, 8, 2, 64, 1, 2000, block_size=32, seed=25), 7),
    ]


def test_noalloc_matches_workspace_entry_point_and_oracle_on_calls_in_a_row(fa):
    so = fa.load()
    cases = _cases()
    B, Hq = cases[2][0].q.shape[:2]
    assert B * Hq * cases[2][1] == MAX_STATES
    for P, num_splits in cases:
        q, kc, vc, bt, sl = _dev(P)
        o_ref, l_ref = fa.fa_paged_decode(q, kc, vc, bt, sl, num_splits=num_splits)
        o = torch.full_like(q, float("nan"))
        lse = torch.full((q.shape[0], q.shape[1]), float("nan"), dtype=torch.float32, device=q.device)
        st = _raw_noalloc(so, q, kc, vc, bt, sl, o, lse, num_splits)
        assert st == fa.FA_OK, fa.status_string(st)
        torch.cuda.synchronize()
        assert fa.fa_get_device_status() == fa.FA_OK
        a, la = o.float().cpu().numpy(), lse.cpu().numpy()
        # against the workspace entry point ...
        _check(a, la, o_ref.float().cpu().numpy(), l_ref.cpu().numpy())
        # ... and against the oracle on the same inputs
        oo, lo = oracle.paged_decode(P.q, P.k_cache, P.v_cache, P.block_table, P.seq_lens, P.block_size)
        _check(a, la, oo, lo)


def test_noalloc_rejects_requests_beyond_its_scratch(fa):
    so = fa.load()
    P = wl.paged_inputs(65, 32, 8, 128, 1, 40, seed=23)
    q, kc, vc, bt, sl = _dev(P)
    o = torch.empty_like(q)
    lse = torch.empty((65, 32), dtype=torch.float32, device=q.device)
    # 65 * 32 * 16 = 33280 partial states > 32768: refused, nothing launched
    assert _raw_noalloc(so, q, kc, vc, bt, sl, o, lse, 16) == fa.FA_ERR_UNSUPPORTED
    # the same batch with 15 splits fits (31200 states)
    assert _raw_noalloc(so, q, kc, vc, bt, sl, o, lse, 15) == fa.FA_OK
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK


def test_noalloc_rejects_table_geometry_like_the_workspace_entry_point(fa):
    # a table row whose keys (max_blocks * block_size) overflow 32-bit indexing
    # is refused by both entry points before anything is launched
    so = fa.load()
    P = wl.paged_inputs(2, 8, 2, 128, 1, 40, seed=26)
    q, kc, vc, bt, sl = _dev(P)
    o = torch.empty_like(q)
    lse = torch.empty((2, 8), dtype=torch.float32, device=q.device)
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    huge = (1 << 31) // 16  # max_blocks * 16 = 2^31 > INT_MAX
    st = so.fa_paged_decode_noalloc(p(q), p(kc), p(vc), p(bt), p(sl), p(o), p(lse), 2, 8, 2, 128, 16, huge,
                                    int(kc.shape[0]), 4, 0.1, stream)
    assert st == fa.FA_ERR_UNSUPPORTED
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=q.device)
    st = so.fa_paged_decode(p(q), p(kc), p(vc), p(bt), p(sl), p(o), p(lse), 2, 8, 2, 128, 16, huge,
                            int(kc.shape[0]), 4, 0.1, p(ws), ctypes.c_size_t(ws.numel()), stream)
    assert st == fa.FA_ERR_UNSUPPORTED
