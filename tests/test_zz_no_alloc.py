"""fa_paged_decode_noalloc: the decode entry point for callers that cannot
allocate device memory (e.g. engine plugins whose memory is assigned ahead of
time, or serving loops that avoid cudaMalloc/cudaFree because those can
synchronise the device).  Its split partials live in a fixed array inside the
library instead of a caller workspace.  These tests call it through the C ABI
and compare it with fa_paged_decode (caller workspace) within the decode
tolerances, on two calls in a row with different inputs, so that leftovers of
the first call in the shared array cannot leak into the second.

The file is named to be collected last."""
import ctypes

import numpy as np
import pytest
import torch

from exact_io_aware_10_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_TOL = 2e-2, 2e-3, 1e-3


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


def _close(a, b):
    err = np.abs(a - b)
    return err.max() <= O_MAX and err.mean() <= O_MEAN


def test_noalloc_matches_workspace_entry_point_on_two_calls(fa):
    so = fa.load()
    cases = [wl.paged_inputs(8, 32, 8, 128, 1, 3000, seed=21),
             wl.paged_inputs(5, 16, 4, 128, 1, 1, seed=22, seq_lens=[0, 17, 900, 16, 2500])]
    for num_splits, P in zip((16, 3), cases):
        q, kc, vc, bt, sl = _dev(P)
        o_ref, l_ref = fa.fa_paged_decode(q, kc, vc, bt, sl, num_splits=num_splits)
        o = torch.full_like(q, float("nan"))
        lse = torch.full((q.shape[0], q.shape[1]), float("nan"), dtype=torch.float32, device=q.device)
        st = _raw_noalloc(so, q, kc, vc, bt, sl, o, lse, num_splits)
        assert st == fa.FA_OK, fa.status_string(st)
        torch.cuda.synchronize()
        assert fa.fa_get_device_status() == fa.FA_OK
        a, b = o.float().cpu().numpy(), o_ref.float().cpu().numpy()
        assert np.isfinite(a).all()
        assert _close(a, b)
        la, lb = lse.cpu().numpy(), l_ref.cpu().numpy()
        fin = np.isfinite(lb)
        assert np.array_equal(np.isfinite(la), fin)
        assert np.abs(la[fin] - lb[fin]).max(initial=0) <= LSE_TOL


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
