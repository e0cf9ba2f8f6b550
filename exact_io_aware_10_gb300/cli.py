"""Run one attention entry point on seeded synthetic inputs, e.g. for a
profiler:  python -m exact_io_aware_10_gb300.cli fwd --N 16384 --iters 2

Subcommands: fwd (block-sparse with --sparse-window W: butterfly mask plus W
local key blocks), bwd (runs fwd once to produce O/LSE, then bwd), decode,
varlen / varlen_bwd (packed ragged batch of --num-seqs sequences, lengths U[--seq-lo, --seq-hi]),
prefill (paged chunked prefill: --num-seqs chunks of --chunk tokens after cached
prefixes of U[0, --prefix-hi] tokens, --Hq/--Hkv heads, --block-size-token blocks).
Prints the CUDA-event times of the last iteration and the median and minimum
over all --iters iterations.
"""
from __future__ import annotations

import argparse
import os
import sys

import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

from exact_io_aware_10_gb300 import lib  # noqa: E402
from exact_io_aware_10_gb300 import workloads as wl  # noqa: E402


class _Marks:
    """CUDA events recorded on the current stream, one per record() call."""

    def __init__(self):
        self.events = []

    def record(self):
        e = torch.cuda.Event(enable_timing=True)
        e.record()
        self.events.append(e)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("op", choices=["fwd", "bwd", "decode", "varlen", "varlen_bwd", "prefill"])
    ap.add_argument("--B", type=int, default=1)
    ap.add_argument("--H", type=int, default=16)
    ap.add_argument("--N", type=int, default=16384)
    ap.add_argument("--d", type=int, default=128)
    ap.add_argument("--noncausal", action="store_true")
    ap.add_argument("--iters", type=int, default=2)
    ap.add_argument("--Hq", type=int, default=32)
    ap.add_argument("--Hkv", type=int, default=8)
    ap.add_argument("--L-lo", type=int, default=512)
    ap.add_argument("--L-hi", type=int, default=32768)
    ap.add_argument("--splits", type=int, default=16)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--num-seqs", type=int, default=16)
    ap.add_argument("--seq-lo", type=int, default=512)
    ap.add_argument("--seq-hi", type=int, default=16384)
    ap.add_argument("--chunk", type=int, default=2048)
    ap.add_argument("--prefix-hi", type=int, default=30720)
    ap.add_argument("--block-size", type=int, default=16)
    ap.add_argument("--sparse-window", type=int, default=None)
    a = ap.parse_args(argv)
    dev = torch.device("cuda")
    lib.load()
    causal = not a.noncausal
    start, end = _Marks(), _Marks()
    if a.op in ("fwd", "bwd"):
        shp = (a.B, a.H, a.N, a.d)
        Q, K, V, dO = (wl.device_normal_bf16(shp, a.seed + i, dev) for i in range(4))
        O, L = lib.fa_fwd(Q, K, V, causal=causal)
        mask = None
        if a.sparse_window is not None:
            mask = wl.block_mask((a.N + 127) // 128, "butterfly", window=a.sparse_window).to(dev)
        for _ in range(a.iters):
            start.record()
            if a.op == "fwd" and mask is not None:
                lib.fa_fwd_block_sparse(Q, K, V, mask, causal=causal, O=O, LSE=L)
            elif a.op == "fwd":
                lib.fa_fwd(Q, K, V, causal=causal, O=O, LSE=L)
            else:
                lib.fa_bwd(Q, K, V, O, dO, L, causal=causal)
            end.record()
    elif a.op == "varlen_bwd":
        lens = wl.varlen_lengths(a.num_seqs, a.seq_lo, a.seq_hi, seed=a.seed)
        cu = [0]
        for n in lens:
            cu.append(cu[-1] + n)
        shp = (cu[-1], a.H, a.d)
        Q, K, V, dO = (wl.device_normal_bf16(shp, a.seed + i, dev) for i in range(4))
        cu = torch.tensor(cu, dtype=torch.int32, device=dev)
        O, L = lib.fa_fwd_varlen(Q, K, V, cu, max(lens), causal=causal)
        ws = torch.empty(lib.fa_bwd_varlen_workspace_size(len(lens), shp[0], max(lens), a.H, a.d), dtype=torch.uint8,
                         device=dev)
        grads = lib.fa_bwd_varlen(Q, K, V, O, dO, L, cu, max(lens), causal=causal, workspace=ws)
        for _ in range(a.iters):
            start.record()
            lib.fa_bwd_varlen(Q, K, V, O, dO, L, cu, max(lens), causal=causal, dQ=grads[0], dK=grads[1], dV=grads[2],
                              workspace=ws)
            end.record()
    elif a.op == "varlen":
        lens = wl.varlen_lengths(a.num_seqs, a.seq_lo, a.seq_hi, seed=a.seed)
        cu = [0]
        for n in lens:
            cu.append(cu[-1] + n)
        shp = (cu[-1], a.H, a.d)
        Q, K, V = (wl.device_normal_bf16(shp, a.seed + i, dev) for i in range(3))
        cu = torch.tensor(cu, dtype=torch.int32, device=dev)
        O, L = lib.fa_fwd_varlen(Q, K, V, cu, max(lens), causal=causal)
        for _ in range(a.iters):
            start.record()
            lib.fa_fwd_varlen(Q, K, V, cu, max(lens), causal=causal, O=O, LSE=L)
            end.record()
    elif a.op == "prefill":
        g = torch.Generator().manual_seed(a.seed)
        prefix = torch.randint(0, a.prefix_hi + 1, (a.num_seqs,), generator=g).tolist()
        kv = [p + a.chunk for p in prefix]
        bs = a.block_size
        sl, table, NB, _ = wl.paged_layout(a.num_seqs, 0, 0, bs, a.seed, None, kv)
        cu = torch.arange(0, (a.num_seqs + 1) * a.chunk, a.chunk, dtype=torch.int32, device=dev)
        q = wl.device_normal_bf16((a.num_seqs * a.chunk, a.Hq, a.d), a.seed + 1, dev)
        kc = wl.device_normal_bf16((NB, bs, a.Hkv, a.d), a.seed + 2, dev)
        vc = wl.device_normal_bf16((NB, bs, a.Hkv, a.d), a.seed + 3, dev)
        sl, table = sl.to(dev), table.to(dev)
        o, lse = lib.fa_paged_prefill(q, kc, vc, table, cu, sl, a.chunk, causal=causal)
        for _ in range(a.iters):
            start.record()
            lib.fa_paged_prefill(q, kc, vc, table, cu, sl, a.chunk, causal=causal, o=o, lse=lse)
            end.record()
    else:
        sl, table, NB, _ = wl.paged_layout(a.B, a.L_lo, a.L_hi, 16, a.seed, None)
        q = wl.device_normal_bf16((a.B, a.Hq, a.d), a.seed + 1, dev)
        kc = wl.device_normal_bf16((NB, 16, a.Hkv, a.d), a.seed + 2, dev)
        vc = wl.device_normal_bf16((NB, 16, a.Hkv, a.d), a.seed + 3, dev)
        sl, table = sl.to(dev), table.to(dev)
        for _ in range(a.iters):
            start.record()
            lib.fa_paged_decode(q, kc, vc, table, sl, num_splits=a.splits)
            end.record()
    torch.cuda.synchronize()
    st = lib.fa_get_device_status()
    times = sorted(s.elapsed_time(e) for s, e in zip(start.events, end.events))
    last = start.events[-1].elapsed_time(end.events[-1])
    print(f"{a.op}: {last:.3f} ms (last iteration), median {times[len(times) // 2]:.3f} ms, min {times[0]:.3f} ms "
          f"over {len(times)}, status {lib.status_string(st)}")
    return 0 if st == lib.FA_OK else 1


if __name__ == "__main__":
    sys.exit(main())
