"""Device bounds checks: the FA_DEBUG build of the library guards every global
load or store its kernels' threads issue (TMA copies clip by themselves) and
latches FA_ERR_OUT_OF_BOUNDS instead of touching memory outside a buffer.  It
stands in for a memory checker, which this pool does not offer.  The edge-case
workloads (ragged and one-row problems, key padding, empty and one-token
sequences, all block sizes, split counts, bad table entries and bad offsets
that the kernels are defined to detect) run against it in a process of their
own (tests/debug_bounds_cases.py), followed by the backward's, the forward's
and paged decode's failure paths: a warp the others wait on is stalled by
the debug build's injection hooks, the bounded waits give up, the call reports FA_ERR_TIMEOUT
without hanging, and the next call matches a clean run."""
import os
import subprocess
import sys

import pytest

from exact_io_aware_10_gb300 import build

pytestmark = pytest.mark.gpu

CASES = os.path.join(os.path.dirname(os.path.abspath(__file__)), "debug_bounds_cases.py")


def test_release_build_carries_no_checks(fa):
    so = fa.load()
    assert so.fa_debug_build() == 0
    assert so.fa_selftest_bounds(None) == fa.FA_OK
    assert fa.fa_get_device_status() == fa.FA_OK  # the guard is the constant true


def test_debug_build_keeps_every_edge_case_in_bounds():
    path = build.build(debug=True)
    env = dict(os.environ, FA_GB300_LIB=path)
    r = subprocess.run([sys.executable, CASES], env=env, capture_output=True, text=True, timeout=1200)
    out = r.stdout + r.stderr
    assert r.returncode == 0, out[-4000:]
    assert "all cases in bounds" in r.stdout, out[-4000:]
    assert "ok   bounds guard self-test: FA_ERR_OUT_OF_BOUNDS" in r.stdout
    assert "ok   packed d=128 backward with its MMA warp stalled: FA_ERR_TIMEOUT" in r.stdout
    assert "ok   packed d=128 forward with its MMA warp stalled: FA_ERR_TIMEOUT" in r.stdout
    assert "ok   decode d=128 splits=4 with its TMA warp stalled: FA_ERR_TIMEOUT" in r.stdout
