"""Python binding of the C ABI in ``include/fa.h``.

Argument marshalling only: tensors are checked for dtype/shape/contiguity,
their device pointers and the current CUDA stream are handed to the shared
library, and outputs / workspaces the caller did not pass are allocated with
torch (device memory plumbing).  Every step of the attention path runs in the
library's CUDA kernels; there is no fallback: if the library is missing the
call raises.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

from . import build as _build

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_CUDA = 3
FA_ERR_TIMEOUT = 4
FA_ERR_BAD_BLOCK_TABLE = 5
FA_ERR_OUT_OF_BOUNDS = 6

# name -> (restype, argtypes); mirrors include/fa.h
_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "fa_status_string": (ctypes.c_char_p, [_i]),
    "fa_version": (_i, []),
    "fa_fwd": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp]),
    "fa_fwd_ex": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp, _vp]),
    "fa_fwd_varlen": (_i, [_vp] * 6 + [_i, _i, _i, _i, _i, _i, _f, _vp]),
    "fa_fwd_block_sparse": (_i, [_vp] * 5 + [_i] * 5 + [_f, _vp, _vp, _i, _vp]),
    "fa_bwd_varlen_workspace_size": (_sz, [_i] * 5),
    "fa_bwd_varlen": (_i, [_vp] * 10 + [_i] * 6 + [_f, _vp, _sz, _vp]),
    "fa_decode_graph_create": (_i, [_vp, _i] + [_vp] * 7 + [_i] * 8 + [_f, _vp, _sz]),
    "fa_decode_graph_launch": (_i, [_vp, _vp]),
    "fa_decode_graph_kernel_count": (_i, [_vp]),
    "fa_decode_graph_destroy": (None, [_vp]),
    "fa_paged_prefill": (_i, [_vp] * 8 + [_i] * 10 + [_f, _vp]),
    "fa_bwd_workspace_size": (_sz, [_i, _i, _i, _i]),
    "fa_bwd": (_i, [_vp] * 9 + [_i, _i, _i, _i, _i, _f, _vp, _vp, _sz, _vp]),
    "fa_paged_decode_workspace_size": (_sz, [_i, _i, _i, _i]),
    "fa_paged_decode": (_i, [_vp] * 7 + [_i] * 8 + [_f, _vp, _sz, _vp]),
    "fa_get_device_status": (_i, [_vp]),
    "fa_selftest_wait_timeout": (_i, [ctypes.c_uint, _vp]),
    "fa_debug_build": (_i, []),
    "fa_selftest_bounds": (_i, [_vp]),
    "fa_debug_stall_backward": (_i, [_i, ctypes.c_uint]),
    "fa_debug_stall_forward": (_i, [_i, ctypes.c_uint]),
    "fa_debug_stall_decode": (_i, [_i, ctypes.c_uint]),
    "fa_paged_decode_noalloc": (_i, [_vp] * 7 + [_i] * 8 + [_f, _vp]),
}

_LIB = None


class FAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {status_string(status)} ({status})")


def library_path() -> str:
    """The shared library this binding loads: the release build, or the build
    named by the FA_GB300_LIB environment variable (e.g. the debug build with
    device bounds checks, ``build.build(debug=True)``)."""
    return os.environ.get("FA_GB300_LIB") or _build.LIB_PATH


def load():
    """Load the shared library (built by ``__graft_entry__.build()``)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = library_path()
    if not os.path.exists(path):
        raise FileNotFoundError(f"{path} is missing: build it with __graft_entry__.build() "
                                f"(python -m exact_io_aware_10_gb300.build)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


def status_string(status: int) -> str:
    try:
        return load().fa_status_string(int(status)).decode()
    except (FileNotFoundError, OSError):
        return f"status {status}"


def _check(status: int, where: str):
    if status != FA_OK:
        raise FAError(status, where)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _need(t, dtype, shape, name):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def fa_fwd(Q, K, V, causal=False, scale=None, kv_lens=None, O=None, LSE=None, stream=None):
    """O, LSE = attention(Q, K, V) for [B, H, N, d] bf16 CUDA tensors."""
    lib = load()
    B, H, N, d = Q.shape
    for t, n in ((Q, "Q"), (K, "K"), (V, "V")):
        _need(t, torch.bfloat16, (B, H, N, d), n)
    if O is None:
        O = torch.empty_like(Q)
    if LSE is None:
        LSE = torch.empty((B, H, N), dtype=torch.float32, device=Q.device)
    _need(O, torch.bfloat16, (B, H, N, d), "O")
    _need(LSE, torch.float32, (B, H, N), "LSE")
    if kv_lens is not None:
        _need(kv_lens, torch.int32, (B,), "kv_lens")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    st = lib.fa_fwd_ex(_p(Q), _p(K), _p(V), _p(O), _p(LSE), B, H, N, d, int(bool(causal)), scale, _p(kv_lens),
                       _stream(stream))
    _check(st, "fa_fwd")
    return O, LSE


def fa_fwd_block_sparse(Q, K, V, block_mask, causal=False, scale=None, kv_lens=None, O=None, LSE=None,
                        stream=None):
    """Block-sparse forward: block_mask is a CUDA uint8 tensor [nb, nb] (shared)
    or [B, H, nb, nb], nb = ceil(N / 128); non-zero keeps a 128 x 128 block."""
    lib = load()
    B, H, N, d = Q.shape
    for t, n in ((Q, "Q"), (K, "K"), (V, "V")):
        _need(t, torch.bfloat16, (B, H, N, d), n)
    nb = (N + 127) // 128
    _need(block_mask, torch.uint8, None, "block_mask")
    if tuple(block_mask.shape) == (nb, nb):
        per_head = 0
    elif tuple(block_mask.shape) == (B, H, nb, nb):
        per_head = 1
    else:
        raise ValueError(f"block_mask must be [{nb}, {nb}] or [{B}, {H}, {nb}, {nb}]")
    if O is None:
        O = torch.empty_like(Q)
    if LSE is None:
        LSE = torch.empty((B, H, N), dtype=torch.float32, device=Q.device)
    _need(O, torch.bfloat16, (B, H, N, d), "O")
    _need(LSE, torch.float32, (B, H, N), "LSE")
    if kv_lens is not None:
        _need(kv_lens, torch.int32, (B,), "kv_lens")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    st = lib.fa_fwd_block_sparse(_p(Q), _p(K), _p(V), _p(O), _p(LSE), B, H, N, d, int(bool(causal)), scale,
                                 _p(kv_lens), _p(block_mask), per_head, _stream(stream))
    _check(st, "fa_fwd_block_sparse")
    return O, LSE


def fa_fwd_varlen(Q, K, V, cu_seqlens, max_seqlen, causal=False, scale=None, O=None, LSE=None, stream=None):
    """O [total, H, d], LSE [H, total] for a packed ragged batch.

    cu_seqlens is a CUDA int32 tensor [num_seqs + 1] of sequence offsets;
    max_seqlen (a Python int) bounds the longest sequence.
    """
    lib = load()
    total, H, d = Q.shape
    for t, n in ((Q, "Q"), (K, "K"), (V, "V")):
        _need(t, torch.bfloat16, (total, H, d), n)
    _need(cu_seqlens, torch.int32, None, "cu_seqlens")
    if cu_seqlens.dim() != 1 or cu_seqlens.numel() < 2:
        raise ValueError("cu_seqlens must be 1-D with num_seqs + 1 >= 2 entries")
    num_seqs = cu_seqlens.numel() - 1
    if O is None:
        O = torch.empty_like(Q)
    if LSE is None:
        LSE = torch.empty((H, total), dtype=torch.float32, device=Q.device)
    _need(O, torch.bfloat16, (total, H, d), "O")
    _need(LSE, torch.float32, (H, total), "LSE")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    st = lib.fa_fwd_varlen(_p(Q), _p(K), _p(V), _p(O), _p(LSE), _p(cu_seqlens), num_seqs, total, int(max_seqlen),
                           H, d, int(bool(causal)), scale, _stream(stream))
    _check(st, "fa_fwd_varlen")
    return O, LSE


def fa_bwd_varlen_workspace_size(num_seqs, total, max_seqlen, H, d) -> int:
    return int(load().fa_bwd_varlen_workspace_size(int(num_seqs), int(total), int(max_seqlen), int(H), int(d)))


def fa_bwd_varlen(Q, K, V, O, dO, LSE, cu_seqlens, max_seqlen, causal=False, scale=None, dQ=None, dK=None,
                  dV=None, workspace=None, stream=None):
    """dQ, dK, dV [total, H, d] for the packed ragged batch of fa_fwd_varlen."""
    lib = load()
    total, H, d = Q.shape
    for t, n in ((Q, "Q"), (K, "K"), (V, "V"), (O, "O"), (dO, "dO")):
        _need(t, torch.bfloat16, (total, H, d), n)
    _need(LSE, torch.float32, (H, total), "LSE")
    _need(cu_seqlens, torch.int32, None, "cu_seqlens")
    if cu_seqlens.dim() != 1 or cu_seqlens.numel() < 2:
        raise ValueError("cu_seqlens must be 1-D with num_seqs + 1 >= 2 entries")
    num_seqs = cu_seqlens.numel() - 1
    dQ = torch.empty_like(Q) if dQ is None else dQ
    dK = torch.empty_like(K) if dK is None else dK
    dV = torch.empty_like(V) if dV is None else dV
    for t, n in ((dQ, "dQ"), (dK, "dK"), (dV, "dV")):
        _need(t, torch.bfloat16, (total, H, d), n)
    ws_bytes = fa_bwd_varlen_workspace_size(num_seqs, total, max_seqlen, H, d)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=Q.device)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    st = lib.fa_bwd_varlen(_p(Q), _p(K), _p(V), _p(O), _p(dO), _p(LSE), _p(dQ), _p(dK), _p(dV), _p(cu_seqlens),
                           num_seqs, total, int(max_seqlen), H, d, int(bool(causal)), scale, _p(workspace),
                           workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "fa_bwd_varlen")
    return dQ, dK, dV


def fa_bwd_workspace_size(B, H, N, d) -> int:
    return int(load().fa_bwd_workspace_size(B, H, N, d))


def fa_bwd(Q, K, V, O, dO, LSE, causal=False, scale=None, kv_lens=None, dQ=None, dK=None, dV=None,
           workspace=None, stream=None):
    """dQ, dK, dV of sum(dO * O) by recomputation from O and LSE."""
    lib = load()
    B, H, N, d = Q.shape
    for t, n in ((Q, "Q"), (K, "K"), (V, "V"), (O, "O"), (dO, "dO")):
        _need(t, torch.bfloat16, (B, H, N, d), n)
    _need(LSE, torch.float32, (B, H, N), "LSE")
    dQ = torch.empty_like(Q) if dQ is None else dQ
    dK = torch.empty_like(K) if dK is None else dK
    dV = torch.empty_like(V) if dV is None else dV
    for t, n in ((dQ, "dQ"), (dK, "dK"), (dV, "dV")):
        _need(t, torch.bfloat16, (B, H, N, d), n)
    if kv_lens is not None:
        _need(kv_lens, torch.int32, (B,), "kv_lens")
    ws_bytes = fa_bwd_workspace_size(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=Q.device)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    st = lib.fa_bwd(_p(Q), _p(K), _p(V), _p(O), _p(dO), _p(LSE), _p(dQ), _p(dK), _p(dV), B, H, N, d,
                    int(bool(causal)), scale, _p(kv_lens), _p(workspace), workspace.numel() * workspace.element_size(),
                    _stream(stream))
    _check(st, "fa_bwd")
    return dQ, dK, dV


def fa_paged_decode_workspace_size(B, Hq, d, num_splits=0) -> int:
    return int(load().fa_paged_decode_workspace_size(B, Hq, d, num_splits))


def fa_paged_decode(q, k_cache, v_cache, block_table, seq_lens, scale=None, num_splits=0, o=None, lse=None,
                    workspace=None, stream=None, want_lse=True):
    """Paged split-KV GQA decode: o [B, Hq, d] bf16 (and lse [B, Hq] fp32)."""
    lib = load()
    B, Hq, d = q.shape
    NB, bs, Hkv, d2 = k_cache.shape
    _need(q, torch.bfloat16, None, "q")
    _need(k_cache, torch.bfloat16, None, "k_cache")
    _need(v_cache, torch.bfloat16, (NB, bs, Hkv, d2), "v_cache")
    _need(block_table, torch.int32, None, "block_table")
    _need(seq_lens, torch.int32, (B,), "seq_lens")
    if d2 != d:
        raise ValueError("k_cache head dimension must match q")
    if block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("block_table must be [B, max_blocks]")
    max_blocks = int(block_table.shape[1])
    o = torch.empty_like(q) if o is None else o
    _need(o, torch.bfloat16, (B, Hq, d), "o")
    if want_lse and lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    if lse is not None:
        _need(lse, torch.float32, (B, Hq), "lse")
    ws_bytes = fa_paged_decode_workspace_size(B, Hq, d, num_splits)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=q.device)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    st = lib.fa_paged_decode(_p(q), _p(k_cache), _p(v_cache), _p(block_table), _p(seq_lens), _p(o), _p(lse),
                             B, Hq, Hkv, d, bs, max_blocks, NB, int(num_splits), scale, _p(workspace),
                             workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "fa_paged_decode")
    return o, lse


def fa_paged_prefill(q, k_cache, v_cache, block_table, cu_seqlens_q, seq_lens_k, max_seqlen_q, causal=True,
                     scale=None, o=None, lse=None, stream=None):
    """Chunked prefill over a paged KV cache: o [total_q, Hq, d] bf16 and
    lse [Hq, total_q] fp32 for query chunks packed by cu_seqlens_q (CUDA int32
    [num_seqs + 1]); chunk s is the last tokens of a context of
    seq_lens_k[s] keys (bottom-right causal alignment)."""
    lib = load()
    total_q, Hq, d = q.shape
    NB, bs, Hkv, d2 = k_cache.shape
    _need(q, torch.bfloat16, None, "q")
    _need(k_cache, torch.bfloat16, None, "k_cache")
    _need(v_cache, torch.bfloat16, (NB, bs, Hkv, d2), "v_cache")
    _need(block_table, torch.int32, None, "block_table")
    _need(cu_seqlens_q, torch.int32, None, "cu_seqlens_q")
    if d2 != d:
        raise ValueError("k_cache head dimension must match q")
    if cu_seqlens_q.dim() != 1 or cu_seqlens_q.numel() < 2:
        raise ValueError("cu_seqlens_q must be 1-D with num_seqs + 1 >= 2 entries")
    num_seqs = cu_seqlens_q.numel() - 1
    _need(seq_lens_k, torch.int32, (num_seqs,), "seq_lens_k")
    if block_table.dim() != 2 or block_table.shape[0] != num_seqs:
        raise ValueError("block_table must be [num_seqs, max_blocks]")
    max_blocks = int(block_table.shape[1])
    o = torch.empty_like(q) if o is None else o
    _need(o, torch.bfloat16, (total_q, Hq, d), "o")
    if lse is None:
        lse = torch.empty((Hq, total_q), dtype=torch.float32, device=q.device)
    _need(lse, torch.float32, (Hq, total_q), "lse")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    st = lib.fa_paged_prefill(_p(q), _p(k_cache), _p(v_cache), _p(block_table), _p(cu_seqlens_q), _p(seq_lens_k),
                              _p(o), _p(lse), num_seqs, total_q, int(max_seqlen_q), Hq, Hkv, d, NB, bs, max_blocks,
                              int(bool(causal)), scale, _stream(stream))
    _check(st, "fa_paged_prefill")
    return o, lse


class DecodeGraph:
    """A decode step (one paged decode per layer) recorded as a CUDA graph.

    ``layers`` is a list of (q, k_cache, v_cache, o, lse) tensors, one per
    call; lse may be None.  block_table, seq_lens, num_splits, scale and the
    workspace are shared by every call.  The graph keeps the tensors' device
    addresses: update their contents between launches, and keep them alive.
    """

    def __init__(self, layers, block_table, seq_lens, scale=None, num_splits=0, workspace=None):
        lib = load()
        q0, k0 = layers[0][0], layers[0][1]
        B, Hq, d = q0.shape
        NB, bs, Hkv, _ = k0.shape
        for q, kc, vc, o, lse in layers:
            _need(q, torch.bfloat16, (B, Hq, d), "q")
            _need(kc, torch.bfloat16, (NB, bs, Hkv, d), "k_cache")
            _need(vc, torch.bfloat16, (NB, bs, Hkv, d), "v_cache")
            _need(o, torch.bfloat16, (B, Hq, d), "o")
            if lse is not None:
                _need(lse, torch.float32, (B, Hq), "lse")
        _need(block_table, torch.int32, None, "block_table")
        _need(seq_lens, torch.int32, (B,), "seq_lens")
        if block_table.dim() != 2 or block_table.shape[0] != B:
            raise ValueError("block_table must be [B, max_blocks]")
        ws_bytes = fa_paged_decode_workspace_size(B, Hq, d, num_splits)
        if workspace is None:
            workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=q0.device)
        n = len(layers)
        arr = ctypes.c_void_p * n
        ptrs = [arr(*[t.data_ptr() for t in col]) for col in zip(*[(l[0], l[1], l[2], l[3]) for l in layers])]
        have_lse = all(l[4] is not None for l in layers)
        lse_arr = arr(*[l[4].data_ptr() for l in layers]) if have_lse else None
        scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
        h = ctypes.c_void_p()
        st = lib.fa_decode_graph_create(ctypes.byref(h), n, ptrs[0], ptrs[1], ptrs[2], ptrs[3], lse_arr,
                                        _p(block_table), _p(seq_lens), B, Hq, Hkv, d, bs, int(block_table.shape[1]),
                                        NB, int(num_splits), scale, _p(workspace),
                                        workspace.numel() * workspace.element_size())
        _check(st, "fa_decode_graph_create")
        self._lib, self._h = lib, h
        self._keep = (layers, block_table, seq_lens, workspace)  # the graph holds their addresses

    @property
    def kernel_count(self) -> int:
        return int(self._lib.fa_decode_graph_kernel_count(self._h))

    def launch(self, stream=None):
        _check(self._lib.fa_decode_graph_launch(self._h, _stream(stream)), "fa_decode_graph_launch")

    def close(self):
        if self._h:
            self._lib.fa_decode_graph_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def fa_paged_decode_noalloc(q, k_cache, v_cache, block_table, seq_lens, scale=None, num_splits=0, o=None, lse=None,
                            stream=None, want_lse=True):
    """fa_paged_decode for callers that cannot allocate device memory: the
    split partials live in the library's fixed device array (at most
    B * Hq * num_splits = 32768 states; calls that overlap on the GPU race).
    Outputs are still passed in by the caller (``o``/``lse``); the ones left
    as None are allocated here only as a convenience of this binding."""
    lib = load()
    B, Hq, d = q.shape
    NB, bs, Hkv, d2 = k_cache.shape
    _need(q, torch.bfloat16, None, "q")
    _need(k_cache, torch.bfloat16, None, "k_cache")
    _need(v_cache, torch.bfloat16, (NB, bs, Hkv, d2), "v_cache")
    _need(block_table, torch.int32, None, "block_table")
    _need(seq_lens, torch.int32, (B,), "seq_lens")
    if block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("block_table must be [B, max_blocks]")
    o = torch.empty_like(q) if o is None else o
    _need(o, torch.bfloat16, (B, Hq, d), "o")
    if want_lse and lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    if lse is not None:
        _need(lse, torch.float32, (B, Hq), "lse")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    st = lib.fa_paged_decode_noalloc(_p(q), _p(k_cache), _p(v_cache), _p(block_table), _p(seq_lens), _p(o), _p(lse),
                                     B, Hq, Hkv, d, bs, int(block_table.shape[1]), NB, int(num_splits), scale,
                                     _stream(stream))
    _check(st, "fa_paged_decode_noalloc")
    return o, lse


def fa_selftest_wait_timeout(timeout_us=20000, stream=None) -> int:
    """Launch the bounded-wait self-test; returns the launch status (the
    device result is read with fa_get_device_status)."""
    return int(load().fa_selftest_wait_timeout(int(timeout_us), _stream(stream)))


def fa_get_device_status(stream=None) -> int:
    """Synchronise the stream and return (then clear) the device status code."""
    return int(load().fa_get_device_status(_stream(stream)))
