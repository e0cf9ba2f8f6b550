"""Edge-case workloads run against the FA_DEBUG build of the library (device
bounds checks on every global access the kernels' threads issue), in a
process of its own: the library path comes from FA_GB300_LIB.

Every case must leave the status word at FA_OK -- or, for the cases that feed
a bad block-table entry or bad packed offsets on purpose, at the error those
inputs are defined to report -- and never at FA_ERR_OUT_OF_BOUNDS.  The bad
inputs are ones the kernels already detect and skip without touching memory
outside the buffers; the debug build confirms that they do.  The last cases
stall the backward's and the forward's MMA warp and the decode split kernel's
TMA warp through the debug build's injection hooks: the call must end with
FA_ERR_TIMEOUT and the next one must match a clean run.
Prints one line per case and exits non-zero on the first failure."""
from __future__ import annotations

import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from exact_io_aware_10_gb300 import lib as fa  # noqa: E402
from exact_io_aware_10_gb300 import workloads as wl  # noqa: E402

DEV = torch.device("cuda")


def check(name, expect=(0,)):
    torch.cuda.synchronize()
    st = fa.fa_get_device_status()
    ok = st in expect and st != fa.FA_ERR_OUT_OF_BOUNDS
    print(f"{'ok  ' if ok else 'FAIL'} {name}: {fa.status_string(st)}", flush=True)
    if not ok:
        sys.exit(1)


def dense_cases():
    for d in (64, 128):
        for N in (1, 17, 129, 300):
            for causal in (False, True):
                x = wl.dense_inputs(2, 3, N, d, seed=N + d)
                Q, K, V, dO = (t.to(DEV) for t in (x.Q, x.K, x.V, x.dO))
                O, L = fa.fa_fwd(Q, K, V, causal=causal)
                fa.fa_bwd(Q, K, V, O, dO, L, causal=causal)
                check(f"dense d={d} N={N} causal={causal}")
    kv = torch.tensor([0, 1, 127, 128, 129, 256], dtype=torch.int32, device=DEV)
    x = wl.dense_inputs(6, 2, 256, 64, seed=6)
    Q, K, V, dO = (t.to(DEV) for t in (x.Q, x.K, x.V, x.dO))
    for causal in (False, True):
        O, L = fa.fa_fwd(Q, K, V, causal=causal, kv_lens=kv)
        fa.fa_bwd(Q, K, V, O, dO, L, causal=causal, kv_lens=kv)
        check(f"key padding edge lengths causal={causal}")
    # head groups smaller than H (long N) and a partly filled backward head group
    x = wl.dense_inputs(1, 5, 20000, 128, seed=7)
    Q, K, V, dO = (t.to(DEV) for t in (x.Q, x.K, x.V, x.dO))
    O, L = fa.fa_fwd(Q, K, V, causal=True)
    fa.fa_bwd(Q, K, V, O, dO, L, causal=True)
    check("B1 H5 N20000 d128 causal")


def block_sparse_cases():
    N = 300
    x = wl.dense_inputs(2, 2, N, 128, seed=9)
    Q, K, V = (t.to(DEV) for t in (x.Q, x.K, x.V))
    nb = (N + 127) // 128
    g = torch.Generator().manual_seed(1)
    shared = (torch.rand(nb, nb, generator=g) < 0.5).to(torch.uint8).to(DEV)
    per_head = (torch.rand(2, 2, nb, nb, generator=g) < 0.5).to(torch.uint8).to(DEV)
    for m in (shared, per_head):
        fa.fa_fwd_block_sparse(Q, K, V, m, causal=True)
        check(f"block-sparse mask {tuple(m.shape)}")


def varlen_cases():
    lens = [0, 1, 17, 128, 129, 0, 300, 1000, 256, 0]
    for d in (64, 128):
        x = wl.varlen_inputs(lens, 3, d, seed=11 + d)
        Q, K, V, dO, cu = (t.to(DEV) for t in (x.Q, x.K, x.V, x.dO, x.cu_seqlens))
        for causal in (False, True):
            O, L = fa.fa_fwd_varlen(Q, K, V, cu, x.max_seqlen, causal=causal)
            fa.fa_bwd_varlen(Q, K, V, O, dO, L, cu, x.max_seqlen, causal=causal)
            check(f"varlen d={d} causal={causal}")
    # offsets past total and a sequence longer than max_seqlen: reported, skipped
    x = wl.varlen_inputs([100, 300, 50], 2, 64, seed=31)
    Q, K, V, dO = (t.to(DEV) for t in (x.Q, x.K, x.V, x.dO))
    O, L = fa.fa_fwd_varlen(Q, K, V, x.cu_seqlens.to(DEV), 256, causal=True)
    check("varlen sequence longer than max_seqlen", expect=(fa.FA_ERR_INVALID_ARG,))
    bad = torch.tensor([0, 100, 400, 460], dtype=torch.int32, device=DEV)
    fa.fa_fwd_varlen(Q, K, V, bad, 300, causal=True, O=O, LSE=L)
    fa.fa_bwd_varlen(Q, K, V, O, dO, L, bad, 300, causal=True)
    check("varlen offsets past total", expect=(fa.FA_ERR_INVALID_ARG,))


def paged_prefill_cases():
    for bs in (16, 32, 64, 128, 256):
        P = wl.paged_prefill_inputs([40, 1, 300, 0, 129], [300, 1, 900, 77, 129], 4, 2, 64, block_size=bs, seed=bs)
        q, kc, vc, bt, cu, sl = (t.to(DEV) for t in (P.q, P.k_cache, P.v_cache, P.block_table, P.cu_seqlens_q,
                                                      P.seq_lens_k))
        fa.fa_paged_prefill(q, kc, vc, bt, cu, sl, P.max_seqlen_q, causal=True)
        check(f"paged prefill block_size={bs}")
    P = wl.paged_prefill_inputs([40, 60], [300, 200], 4, 2, 64, block_size=16, seed=12)
    P.block_table[1, 3] = P.k_cache.shape[0] + 5
    q, kc, vc, bt, cu, sl = (t.to(DEV) for t in (P.q, P.k_cache, P.v_cache, P.block_table, P.cu_seqlens_q,
                                                  P.seq_lens_k))
    fa.fa_paged_prefill(q, kc, vc, bt, cu, sl, P.max_seqlen_q, causal=True)
    check("paged prefill bad table entry", expect=(fa.FA_ERR_BAD_BLOCK_TABLE,))


def decode_cases():
    for d in (64, 128):
        for bs in (16, 32):
            P = wl.paged_inputs(5, 16, 4, d, 1, 1, block_size=bs, seed=bs + d, seq_lens=[0, 17, 900, 16, 2500])
            q, kc, vc, bt, sl = (t.to(DEV) for t in (P.q, P.k_cache, P.v_cache, P.block_table, P.seq_lens))
            for splits in (0, 1, 3, 16):
                fa.fa_paged_decode(q, kc, vc, bt, sl, num_splits=splits)
                fa.fa_paged_decode_noalloc(q, kc, vc, bt, sl, num_splits=splits)
                check(f"decode d={d} block_size={bs} splits={splits}")
    P = wl.paged_inputs(2, 8, 2, 128, 1, 1, seed=17, seq_lens=[64, 64])
    bt = P.block_table.clone()
    bt[1, 2] = P.num_blocks + 5
    q, kc, vc, sl = (t.to(DEV) for t in (P.q, P.k_cache, P.v_cache, P.seq_lens))
    fa.fa_paged_decode(q, kc, vc, bt.to(DEV), sl, num_splits=4)
    check("decode bad table entry", expect=(fa.FA_ERR_BAD_BLOCK_TABLE,))


def stall_cases(so):
    # the backward's MMA warp stops at work item 0 (debug hook) with 20 ms wait
    # limits: the call reports FA_ERR_TIMEOUT, every CTA ends, and the next
    # call gives the gradients of a clean run
    def dense(d):
        x = wl.dense_inputs(2, 4, 1000, d, seed=40 + d)
        Q, K, V, dO = (t.to(DEV) for t in (x.Q, x.K, x.V, x.dO))
        O, L = fa.fa_fwd(Q, K, V, causal=True)
        return lambda: fa.fa_bwd(Q, K, V, O, dO, L, causal=True)

    def packed(d):
        x = wl.varlen_inputs([700, 1, 300, 129], 4, d, seed=50 + d)
        Q, K, V, dO, cu = (t.to(DEV) for t in (x.Q, x.K, x.V, x.dO, x.cu_seqlens))
        O, L = fa.fa_fwd_varlen(Q, K, V, cu, x.max_seqlen, causal=True)
        return lambda: fa.fa_bwd_varlen(Q, K, V, O, dO, L, cu, x.max_seqlen, causal=True)

    for kind, make in (("dense", dense), ("packed", packed)):
        for d in (64, 128):
            run = make(d)
            ref = [t.float() for t in run()]
            check(f"{kind} d={d} backward before the stall")
            if so.fa_debug_stall_backward(0, 20000) != fa.FA_OK:
                print("FAIL the stall injection did not arm")
                sys.exit(1)
            run()
            check(f"{kind} d={d} backward with its MMA warp stalled", expect=(fa.FA_ERR_TIMEOUT,))
            got = [t.float() for t in run()]
            check(f"{kind} d={d} backward after the stall")
            for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
                err = (g - r).abs().max().item()
                tol = 1e-2 * r.abs().max().item() + 1e-6
                if not err <= tol:
                    print(f"FAIL {kind} d={d} {name} after the stall: max error {err:.3g} > {tol:.3g}")
                    sys.exit(1)


def forward_stall_cases(so):
    # the forward's MMA warp in CTA 0 issues nothing (debug hook) with 20 ms wait
    # limits: the call reports FA_ERR_TIMEOUT, every CTA ends, the next call is clean
    def dense(d):
        x = wl.dense_inputs(2, 4, 1000, d, seed=60 + d)
        Q, K, V = (t.to(DEV) for t in (x.Q, x.K, x.V))
        return lambda: fa.fa_fwd(Q, K, V, causal=True)

    def packed(d):
        x = wl.varlen_inputs([700, 1, 300, 129], 4, d, seed=70 + d)  # sequence 0 is the longest
        Q, K, V, cu = (t.to(DEV) for t in (x.Q, x.K, x.V, x.cu_seqlens))
        return lambda: fa.fa_fwd_varlen(Q, K, V, cu, x.max_seqlen, causal=True)

    for kind, make in (("dense", dense), ("packed", packed)):
        for d in (64, 128):
            run = make(d)
            ref = [t.float() for t in run()]
            check(f"{kind} d={d} forward before the stall")
            if so.fa_debug_stall_forward(0, 20000) != fa.FA_OK:
                print("FAIL the forward stall injection did not arm")
                sys.exit(1)
            run()
            check(f"{kind} d={d} forward with its MMA warp stalled", expect=(fa.FA_ERR_TIMEOUT,))
            got = [t.float() for t in run()]
            check(f"{kind} d={d} forward after the stall")
            for name, g, r in zip(("O", "LSE"), got, ref):
                if not torch.equal(g, r):
                    print(f"FAIL {kind} d={d} {name} after the stall differs from the clean run")
                    sys.exit(1)


def decode_stall_cases(so):
    # the decode split kernel's TMA warp in CTA 0 (first sequence, first split)
    # loads nothing: FA_ERR_TIMEOUT, every CTA ends, the next call is clean
    for d in (64, 128):
        for splits in (1, 4):
            P = wl.paged_inputs(2, 16, 4, d, 1, 1, block_size=16, seed=80 + d, seq_lens=[900, 2500])
            q, kc, vc, bt, sl = (t.to(DEV) for t in (P.q, P.k_cache, P.v_cache, P.block_table, P.seq_lens))
            ref = [t.float() for t in fa.fa_paged_decode(q, kc, vc, bt, sl, num_splits=splits)]
            check(f"decode d={d} splits={splits} before the stall")
            if so.fa_debug_stall_decode(0, 20000) != fa.FA_OK:
                print("FAIL the decode stall injection did not arm")
                sys.exit(1)
            fa.fa_paged_decode(q, kc, vc, bt, sl, num_splits=splits)
            check(f"decode d={d} splits={splits} with its TMA warp stalled", expect=(fa.FA_ERR_TIMEOUT,))
            got = [t.float() for t in fa.fa_paged_decode(q, kc, vc, bt, sl, num_splits=splits)]
            check(f"decode d={d} splits={splits} after the stall")
            for name, g, r in zip(("o", "lse"), got, ref):
                if not torch.equal(g, r):
                    print(f"FAIL decode d={d} splits={splits} {name} after the stall differs from the clean run")
                    sys.exit(1)


if __name__ == "__main__":
    so = fa.load()
    if so.fa_debug_build() != 1:
        print("FAIL FA_GB300_LIB does not name a debug build")
        sys.exit(1)
    so.fa_selftest_bounds(None)
    torch.cuda.synchronize()
    st = fa.fa_get_device_status()
    print(f"{'ok  ' if st == fa.FA_ERR_OUT_OF_BOUNDS else 'FAIL'} bounds guard self-test: {fa.status_string(st)}",
          flush=True)
    if st != fa.FA_ERR_OUT_OF_BOUNDS:
        sys.exit(1)
    check("status word cleared")
    dense_cases()
    block_sparse_cases()
    varlen_cases()
    paged_prefill_cases()
    decode_cases()
    stall_cases(so)
    forward_stall_cases(so)
    decode_stall_cases(so)
    print("all cases in bounds")
