"""Failure detection without a GPU fault: a pipeline wait that can never
complete must give up after its limit, latch FA_ERR_TIMEOUT in the device
status word, and leave the CUDA context usable."""
import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_10_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives(fa):
    assert fa.fa_get_device_status() == fa.FA_OK  # start clean
    assert fa.fa_selftest_wait_timeout(20000) == fa.FA_OK  # launch accepted
    assert fa.fa_get_device_status() == fa.FA_ERR_TIMEOUT
    assert fa.fa_get_device_status() == fa.FA_OK  # reading clears the word
    # the context still runs real work correctly
    x = wl.dense_inputs(1, 2, 256, 64, seed=3)
    dev = torch.device("cuda")
    O, L = fa.fa_fwd(x.Q.to(dev), x.K.to(dev), x.V.to(dev), causal=True)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    Oref, _ = oracle.attention_forward(x.Q, x.K, x.V, causal=True)
    assert np.abs(O.float().cpu().numpy() - Oref).max() <= 2e-2
