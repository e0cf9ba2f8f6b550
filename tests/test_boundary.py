"""The C-ABI library loads on the host, exports every entry point declared in
include/fa.h, and rejects invalid arguments before touching the GPU."""
import ctypes
import os
import re
import subprocess
import sys

import pytest

from exact_io_aware_10_gb300 import build as fab
from exact_io_aware_10_gb300 import lib as fl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def so():
    fab.build()
    return fl.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("fa_fwd", "fa_fwd_ex", "fa_fwd_varlen", "fa_fwd_block_sparse", "fa_paged_prefill", "fa_bwd",
              "fa_bwd_workspace_size", "fa_paged_decode", "fa_decode_graph_create", "fa_decode_graph_launch",
              "fa_paged_decode_workspace_size", "fa_get_device_status", "fa_status_string", "fa_version"):
        assert n in names


def test_library_exports_every_declared_symbol(so):
    for n in declared_functions():
        assert hasattr(so, n), n
    assert set(declared_functions()) <= set(fl.SIGNATURES)


def test_status_strings(so):
    for code, name in [(0, "FA_OK"), (1, "FA_ERR_INVALID_ARG"), (2, "FA_ERR_UNSUPPORTED"), (3, "FA_ERR_CUDA"),
                       (4, "FA_ERR_TIMEOUT"), (5, "FA_ERR_BAD_BLOCK_TABLE"), (6, "FA_ERR_OUT_OF_BOUNDS")]:
        assert so.fa_status_string(code).decode() == name
    assert so.fa_status_string(99).decode() == "FA_ERR_UNKNOWN"
    assert so.fa_version() == 109


def _fake(n=1):
    # 256-byte aligned fake device addresses; validation rejects before any use
    return [ctypes.c_void_p(0x10000000 + 0x1000 * i) for i in range(n)]


def test_forward_argument_validation(so):
    Q, K, V, O, L = _fake(5)
    s = ctypes.c_void_p(0)
    assert so.fa_fwd(Q, K, V, O, L, 1, 1, 16, 96, 0, 0.1, s) == fl.FA_ERR_UNSUPPORTED
    assert so.fa_fwd(Q, K, V, O, L, 0, 1, 16, 64, 0, 0.1, s) == fl.FA_ERR_INVALID_ARG
    assert so.fa_fwd(Q, K, V, O, L, 1, 1, -1, 64, 0, 0.1, s) == fl.FA_ERR_INVALID_ARG
    assert so.fa_fwd(None, K, V, O, L, 1, 1, 16, 64, 0, 0.1, s) == fl.FA_ERR_INVALID_ARG
    assert so.fa_fwd(Q, K, V, O, L, 1, 1, 16, 64, 0, 0.0, s) == fl.FA_ERR_INVALID_ARG
    assert so.fa_fwd(Q, K, V, O, L, 1, 1, 16, 64, 0, float("nan"), s) == fl.FA_ERR_INVALID_ARG
    assert so.fa_fwd(ctypes.c_void_p(0x10000008), K, V, O, L, 1, 1, 16, 64, 0, 0.1, s) == fl.FA_ERR_INVALID_ARG
    # more batch entries than the grid's z dimension holds
    assert so.fa_fwd(Q, K, V, O, L, 65536, 1, 16, 64, 0, 0.1, s) == fl.FA_ERR_UNSUPPORTED
    # N = 0 is a valid no-op and launches nothing
    assert so.fa_fwd(Q, K, V, O, L, 1, 1, 0, 64, 0, 0.1, s) == fl.FA_OK


def test_block_sparse_argument_validation(so):
    Q, K, V, O, L, M = _fake(6)
    s = ctypes.c_void_p(0)
    f = so.fa_fwd_block_sparse
    # (Q, K, V, O, LSE, B, H, N, d, causal, scale, kv_lens, block_mask, per_head, stream)
    assert f(Q, K, V, O, L, 1, 2, 1024, 96, 0, 0.1, None, M, 0, s) == fl.FA_ERR_UNSUPPORTED
    assert f(Q, K, V, O, L, 1, 2, 1024, 128, 0, 0.1, None, None, 0, s) == fl.FA_ERR_INVALID_ARG
    assert f(Q, K, V, O, L, 0, 2, 1024, 128, 0, 0.1, None, M, 0, s) == fl.FA_ERR_INVALID_ARG
    assert f(Q, K, V, O, L, 1, 2, 1024, 128, 0, 0.0, None, M, 0, s) == fl.FA_ERR_INVALID_ARG
    assert f(Q, K, V, O, L, 1, 2, 262144 + 1, 128, 0, 0.1, None, M, 0, s) == fl.FA_ERR_UNSUPPORTED
    assert f(Q, K, V, O, L, 65536, 1, 1024, 128, 0, 0.1, None, M, 0, s) == fl.FA_ERR_UNSUPPORTED
    assert f(Q, K, V, O, L, 1, 2, 0, 128, 0, 0.1, None, M, 0, s) == fl.FA_OK  # N = 0: no-op


def test_varlen_forward_argument_validation(so):
    Q, K, V, O, L, cu = _fake(6)
    s = ctypes.c_void_p(0)
    f = so.fa_fwd_varlen
    # (Q, K, V, O, LSE, cu_seqlens, num_seqs, total, max_seqlen, H, d, causal, scale, stream)
    assert f(Q, K, V, O, L, cu, 2, 100, 64, 4, 96, 0, 0.1, s) == fl.FA_ERR_UNSUPPORTED
    assert f(Q, K, V, O, L, cu, 0, 100, 64, 4, 64, 0, 0.1, s) == fl.FA_ERR_INVALID_ARG
    assert f(Q, K, V, O, L, cu, 2, -1, 64, 4, 64, 0, 0.1, s) == fl.FA_ERR_INVALID_ARG
    assert f(Q, K, V, O, L, cu, 2, 100, -1, 4, 64, 0, 0.1, s) == fl.FA_ERR_INVALID_ARG
    assert f(Q, K, V, O, L, cu, 2, 100, 64, 0, 64, 0, 0.1, s) == fl.FA_ERR_INVALID_ARG
    assert f(Q, K, V, O, L, None, 2, 100, 64, 4, 64, 0, 0.1, s) == fl.FA_ERR_INVALID_ARG
    assert f(Q, K, V, O, None, cu, 2, 100, 64, 4, 64, 0, 0.1, s) == fl.FA_ERR_INVALID_ARG
    assert f(Q, K, V, O, L, cu, 2, 100, 64, 4, 64, 0, float("inf"), s) == fl.FA_ERR_INVALID_ARG
    assert f(Q, ctypes.c_void_p(0x10000004), V, O, L, cu, 2, 100, 64, 4, 64, 0, 0.1, s) == fl.FA_ERR_INVALID_ARG
    # a max_seqlen needing more than 65535 grid rows is outside the kernel's grid
    assert f(Q, K, V, O, L, cu, 2, 100, 256 * 65536, 4, 64, 0, 0.1, s) == fl.FA_ERR_UNSUPPORTED
    # more sequences than the grid's z dimension holds
    assert f(Q, K, V, O, L, cu, 65536, 100, 64, 4, 64, 0, 0.1, s) == fl.FA_ERR_UNSUPPORTED
    # an empty batch is a valid no-op and launches nothing
    assert f(Q, K, V, O, L, cu, 2, 0, 0, 4, 64, 0, 0.1, s) == fl.FA_OK


def test_paged_prefill_argument_validation(so):
    q, kc, vc, bt, cu, sl, o, lse = _fake(8)
    s = ctypes.c_void_p(0)

    def call(**kw):
        a = dict(num_seqs=2, total_q=100, max_seqlen_q=64, Hq=8, Hkv=2, d=128, num_blocks=10, block_size=16,
                 max_blocks=4, causal=1, scale=0.1)
        a.update(kw)
        return so.fa_paged_prefill(a.get("q", q), kc, vc, a.get("bt", bt), cu, sl, o, lse, a["num_seqs"],
                                   a["total_q"], a["max_seqlen_q"], a["Hq"], a["Hkv"], a["d"], a["num_blocks"],
                                   a["block_size"], a["max_blocks"], a["causal"], a["scale"], s)

    assert call(d=96) == fl.FA_ERR_UNSUPPORTED
    assert call(Hkv=3) == fl.FA_ERR_INVALID_ARG          # Hq % Hkv != 0
    assert call(num_seqs=0) == fl.FA_ERR_INVALID_ARG
    assert call(total_q=-1) == fl.FA_ERR_INVALID_ARG
    assert call(num_blocks=0) == fl.FA_ERR_INVALID_ARG
    assert call(max_blocks=0) == fl.FA_ERR_INVALID_ARG
    assert call(scale=-1.0) == fl.FA_ERR_INVALID_ARG
    for bad_bs in (4, 12, 24, 48, 136, 200):            # not a multiple of 8 dividing 128 or of 128
        assert call(block_size=bad_bs) == fl.FA_ERR_UNSUPPORTED, bad_bs
    for good_bs in (8, 16, 32, 64, 128, 256, 384):
        assert call(block_size=good_bs, total_q=0) == fl.FA_OK, good_bs
    assert call(num_seqs=65536) == fl.FA_ERR_UNSUPPORTED
    assert call(num_blocks=1 << 27) == fl.FA_ERR_UNSUPPORTED  # cache rows past int32
    assert call(q=None) == fl.FA_ERR_INVALID_ARG
    assert call(bt=None) == fl.FA_ERR_INVALID_ARG
    assert call(q=ctypes.c_void_p(0x10000002)) == fl.FA_ERR_INVALID_ARG
    assert call(total_q=0) == fl.FA_OK                  # no-op


def test_decode_graph_argument_validation(so):
    ptrs = (ctypes.c_void_p * 2)(0x10000000, 0x10001000)
    h = ctypes.c_void_p()
    args = [ptrs, ptrs, ptrs, ptrs, None, ctypes.c_void_p(0x10002000), ctypes.c_void_p(0x10003000),
            1, 8, 2, 128, 16, 4, 10, 0, 0.1, ctypes.c_void_p(0x10004000), 1 << 20]
    assert so.fa_decode_graph_create(None, 2, *args) == fl.FA_ERR_INVALID_ARG  # no handle
    assert so.fa_decode_graph_create(ctypes.byref(h), 0, *args) == fl.FA_ERR_INVALID_ARG  # no calls
    assert not h.value
    assert so.fa_decode_graph_launch(None, None) == fl.FA_ERR_INVALID_ARG
    assert so.fa_decode_graph_kernel_count(None) == 0
    so.fa_decode_graph_destroy(None)  # a no-op


def test_varlen_backward_argument_validation(so):
    p = _fake(11)
    s = ctypes.c_void_p(0)
    need = so.fa_bwd_varlen_workspace_size(2, 100, 64, 4, 128)
    # -D and -LSE2 rows, the fp32 dQ accumulator, 256 bytes for the work counter
    assert need == 2 * (((2 * 4 * 128 * 4) + 255) // 256 * 256) + (100 * 4 * 128 * 4 + 255) // 256 * 256 + 256
    assert so.fa_bwd_varlen_workspace_size(0, 100, 64, 4, 128) == 0
    f = so.fa_bwd_varlen

    def call(num_seqs=2, total=100, max_seqlen=64, H=4, d=128, scale=0.1, ws=need, cu=p[9]):
        return f(*p[:9], cu, num_seqs, total, max_seqlen, H, d, 1, scale, p[10], ws, s)

    assert call(d=96) == fl.FA_ERR_UNSUPPORTED
    assert call(num_seqs=0) == fl.FA_ERR_INVALID_ARG
    assert call(H=0) == fl.FA_ERR_INVALID_ARG
    assert call(scale=0.0) == fl.FA_ERR_INVALID_ARG
    assert call(cu=None) == fl.FA_ERR_INVALID_ARG
    assert call(ws=need - 1) == fl.FA_ERR_INVALID_ARG
    assert call(num_seqs=65536) == fl.FA_ERR_UNSUPPORTED
    assert call(total=0) == fl.FA_OK  # no-op


def test_backward_argument_validation(so):
    ptrs = _fake(10)
    s = ctypes.c_void_p(0)
    need = so.fa_bwd_workspace_size(2, 3, 100, 64)
    bh, npad = 2 * 3, 128
    assert need == 2 * ((bh * npad * 4 + 255) // 256) * 256 + ((bh * 100 * 64 * 4 + 255) // 256) * 256 + 256
    assert so.fa_bwd_workspace_size(0, 1, 1, 64) == 0
    assert so.fa_bwd(*ptrs[:9], 2, 3, 100, 64, 0, 0.1, None, ptrs[9], need - 1, s) == fl.FA_ERR_INVALID_ARG
    assert so.fa_bwd(*ptrs[:9], 2, 3, 100, 64, 0, 0.1, None, None, need, s) == fl.FA_ERR_INVALID_ARG
    assert so.fa_bwd(*ptrs[:9], 2, 3, 100, 80, 0, 0.1, None, ptrs[9], need, s) == fl.FA_ERR_UNSUPPORTED


def test_decode_argument_validation(so):
    q, kc, vc, bt, sl, o, lse, ws = _fake(8)
    s = ctypes.c_void_p(0)
    need = so.fa_paged_decode_workspace_size(4, 32, 128, 0)
    n = 4 * 32 * 16
    assert need == ((n * 128 * 4 + 255) // 256) * 256 + ((n * 2 * 4 + 255) // 256) * 256
    assert so.fa_paged_decode_workspace_size(4, 32, 128, 17) == 0
    args = dict(B=4, Hq=32, Hkv=8, d=128, bs=16, mb=8, nb=32, S=0)

    def call(**kw):
        a = {**args, **kw}
        return so.fa_paged_decode(q, kc, vc, bt, sl, o, lse, a["B"], a["Hq"], a["Hkv"], a["d"], a["bs"], a["mb"],
                                  a["nb"], a["S"], 0.088, ws, need, s)

    assert call(Hkv=5) == fl.FA_ERR_INVALID_ARG          # Hq % Hkv != 0
    assert call(d=96) == fl.FA_ERR_UNSUPPORTED
    for bad_bs in (8, 24, 40):                             # not a multiple of 16
        assert call(bs=bad_bs) == fl.FA_ERR_UNSUPPORTED
    assert call(S=17) == fl.FA_ERR_UNSUPPORTED
    assert so.fa_paged_decode_workspace_size(4, 32, 128, 1) == 0  # one split: fused, no workspace
    assert call(nb=0) == fl.FA_ERR_INVALID_ARG


def test_selftest_argument_validation(so):
    s = ctypes.c_void_p(0)
    assert so.fa_selftest_wait_timeout(0, s) == fl.FA_ERR_INVALID_ARG
    assert so.fa_selftest_wait_timeout(2000000, s) == fl.FA_ERR_INVALID_ARG
    # the backward stall injection exists in debug builds only
    assert so.fa_debug_stall_backward(-1, 1000) == fl.FA_ERR_INVALID_ARG
    assert so.fa_debug_stall_backward(0, 0) == fl.FA_ERR_INVALID_ARG
    assert so.fa_debug_stall_backward(0, 2000000) == fl.FA_ERR_INVALID_ARG
    assert so.fa_debug_stall_backward(0, 1000) == fl.FA_ERR_UNSUPPORTED
    assert so.fa_debug_stall_forward(-1, 1000) == fl.FA_ERR_INVALID_ARG
    assert so.fa_debug_stall_forward(0, 0) == fl.FA_ERR_INVALID_ARG
    assert so.fa_debug_stall_forward(0, 1000) == fl.FA_ERR_UNSUPPORTED
    assert so.fa_debug_stall_decode(-1, 1000) == fl.FA_ERR_INVALID_ARG
    assert so.fa_debug_stall_decode(0, 1000) == fl.FA_ERR_UNSUPPORTED


def test_binding_has_every_name_the_bench_and_smoke_use():
    # bench.py and smoke() call the Python binding by attribute; a missing
    # wrapper would only show up on the GPU machine
    for path in ("bench.py", "__graft_entry__.py"):
        src = open(os.path.join(ROOT, path)).read()
        for name in set(re.findall(r"\blib\.([A-Za-z_][A-Za-z_0-9]*)", src)):
            assert hasattr(fl, name), (path, name)


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    # no fallback: without the built library the binding raises instead of computing
    monkeypatch.setattr(fl, "_LIB", None)
    monkeypatch.setattr(fl, "library_path", lambda: str(tmp_path / "libfa_gb300.so"))
    with pytest.raises(FileNotFoundError):
        fl.load()


def test_host_tensors_are_refused(so):
    # the binding takes device tensors only: host tensors raise before any call
    import torch

    x = torch.zeros(1, 1, 16, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        fl.fa_fwd(x, x, x)


def test_debug_build_compiles_and_reports_itself():
    # the FA_DEBUG variant (device bounds checks) builds from the same sources;
    # loading it needs no GPU
    path = fab.build(debug=True)
    code = (f"import ctypes; so = ctypes.CDLL({path!r}); "
            "print(so.fa_debug_build(), so.fa_debug_stall_backward(0, 1000), so.fa_debug_stall_backward(-1, 1000), "
            "so.fa_debug_stall_forward(0, 1000), so.fa_debug_stall_forward(0, 2000000), "
            "so.fa_debug_stall_decode(0, 1000), so.fa_debug_stall_decode(0, 0))")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=120)
    # debug build; the stall injections arm (host state only) and check their arguments
    ok, bad = str(fl.FA_OK), str(fl.FA_ERR_INVALID_ARG)
    assert r.returncode == 0 and r.stdout.split() == ["1", ok, bad, ok, bad, ok, bad], r.stdout + r.stderr
