#!/usr/bin/env python
"""Benchmark of the exact IO-aware attention hot path on GB300.

One step = one pass of the whole path over one batch of synthetic input:
  1. forward   B=1, H=16, N=16384, d=128, causal          (fa_fwd)
  2. backward  same tensors, by recomputation              (fa_bwd)
  3. forward   B=1, H=16, N=65536, d=128, causal          (fa_fwd)
  4. paged GQA decode: B=64, Hq=32, Hkv=8, d=128, L ~ U[512, 32768],
     16-token blocks, random physical placement, 16 splits (fa_paged_decode)
Metric: attention fwd/bwd TFLOP/s (steps 1-3, algorithmic FLOPs: 4 B H N^2 d
halved for causal, backward 2.5x) and paged-decode HBM GB/s (step 4), each
also as a fraction of the measured peaks.  `value` is the fwd/bwd TFLOP/s;
the decode figure is in `decode`.  Inputs are seeded synthetic tensors drawn
on the device; every per-kernel input is larger than the 129 MB L2.

After the step (outside `value`), the same run times the encoder- and
decoder-shaped configurations at d = 64 (BERT-large-shaped B16 H16 N512 with
key padding, GPT-2-medium-shaped B8 H16 N1024 / N4096 causal with boosted
logits), forward and backward, with L2 flushed before every timed call, and
the built extensions (ragged batch, paged prefill, block-sparse, decode-step
graph).  `roofline` carries one block of flat keys per kernel: the forward
(the dominant kernel), the backward call, the decode pair and the small
configurations.

`--impl reference` times the fp64 CPU oracle on a bounded sample of the same
workload instead (rank 0 only).  Under torchrun every rank runs an
independent replica (the path has no exchange step); rank 0 prints one JSON
line with the max-over-ranks timing.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

NCORES = len(os.sched_getaffinity(0))
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, str(NCORES))

import numpy as np  # noqa: E402
import torch  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from exact_io_aware_10_gb300 import accounting as acc  # noqa: E402
from exact_io_aware_10_gb300 import workloads as wl  # noqa: E402

METRIC = "attention fwd/bwd TFLOP/s (% of BF16 peak); paged-decode HBM GB/s (% of peak)"
PREFILL = dict(B=1, H=16, d=128, N_fb=16384, N_f=65536)
DECODE = dict(B=64, Hq=32, Hkv=8, d=128, L_lo=512, L_hi=32768, block=16, max_blocks=2048, splits=16)
# packed ragged-batch forward workloads, timed after the step: the BERT-large-
# shaped padded configuration's lengths packed without padding, and a long-
# context causal prefill mix; lengths are uniform integers in [lo, hi]
VARLEN = {
    "bert": dict(num_seqs=16, lo=128, hi=512, H=16, d=64, causal=False, config_id=2, padded_N=512),
    "long": dict(num_seqs=16, lo=512, hi=16384, H=16, d=128, causal=True, config_id=6, padded_N=None),
}
# chunked prefill over a paged cache, timed after the step: every sequence
# appends a q_len-token chunk to a cached prefix of U[prefix_lo, prefix_hi]
# tokens (GQA heads, 16-token blocks, seeded random block placement)
PAGED_PREFILL = dict(num_seqs=16, q_len=2048, prefix_lo=0, prefix_hi=30720, Hq=32, Hkv=8, d=128, block_size=16,
                     config_id=7)
# block-sparse forward, timed after the step on the long-context shapes: a
# butterfly mask plus a local window of BLOCK_SPARSE_WINDOW key blocks
BLOCK_SPARSE_WINDOW = 15
# decode launch overhead, timed after the step: one decode step of
# DECODE_STEP["layers"] paged decodes (B sequences of `context` tokens, Hq/Hkv
# heads, 16-token blocks), issued eagerly call by call or replayed as one graph
DECODE_STEP = dict(layers=32, B=1, Hq=32, Hkv=8, d=128, context=2048, config_id=8)
WORKLOAD = ("long-context causal prefill B1 H16 d128 (fwd+bwd N=16384, fwd N=65536) + paged GQA decode "
            "B64 Hq32 Hkv8 d128 L~U[512,32768] block16 splits16")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# GB300 nominal dense figures, the denominators the targets are stated in.
# bf16: NVIDIA's HGX B300 specification gives 36 PFLOPS FP16/BF16 tensor
# throughput for eight GPUs with 2:4 sparsity, i.e. 2.25 PFLOPS dense per GPU
# (the primary figure).  NVIDIA's GB300 NVL72 rack specification gives 360
# PFLOPS FP16/BF16 with sparsity for 72 GPUs, i.e. 2.5 PFLOPS dense per GPU;
# every fraction is also reported against that stricter figure.  HBM3e: 8 TB/s.
NOMINAL = {"bf16_tflops": 2250.0, "bf16_tflops_nvl72": 2500.0, "hbm_gbs": 8000.0}
# ncu dram bytes (dram__bytes_read.sum + dram__bytes_write.sum) per launch of
# each kernel, one launch captured per shape, with the hash of the source file
# they were taken on: a figure turns null once its source changes.
TRAFFIC_RECORD = {
    "fwd": {"kernel": "fwd_kernel<128>", "source": "exact_io_aware_10_gb300/csrc/fa_fwd.cu",
            "sha256": "3630e69b48727d7ff1bb1c895d15cacd699d08e2946a893bf3bd288a84579226",
            "bytes": {"N16384": 290745600 + 47855104, "N65536": 1167099136 + 250001664}},
    "bwd": {"kernel": "bwd_pre_kernel<128> + bwd_main_kernel<128> + bwd_dq_kernel",
            "source": "exact_io_aware_10_gb300/csrc/fa_bwd.cu",
            "sha256": "b80c3f350e35ffe702e01ce477881e52f37febbf87a07351068eeb8b05309b10",
            "bytes": {"N16384_main": 407478016 + 222058752, "N16384_pre": 135283968 + 87193600,
                      "N16384_dq": 134224384 + 35507712}},
    "decode": {"kernel": "decode_split_kernel<128> + decode_combine_kernel<128>",
               "source": "exact_io_aware_10_gb300/csrc/fa_decode.cu",
               "sha256": "96643620437889a50b50449cfba8585c7840c835eb6f35ec53c73832317d557e",
               "bytes": {"B64": 4425079040 + 17810688 + 15574272 + 0}},
}
# the pages' encoder and decoder training shapes (BERT-large- and GPT-2-medium-
# shaped attention, d = 64), timed after the step, forward and backward.  Their
# inputs are close to or below the 129 MB L2, so L2 is flushed (a 256 MiB
# write) before every timed call.  The BERT shape's key-padding lengths are
# uniform in [128, 512]; its throughput counts the effective FLOPs (every query
# row against its sequence's valid keys), the formula count is reported beside.
SMALL = {
    "bert": dict(B=16, H=16, N=512, d=64, causal=False, kv=(128, 512), boost=False, config_id=2, seed_off=0),
    "gpt2_N1024": dict(B=8, H=16, N=1024, d=64, causal=True, kv=None, boost=True, config_id=3, seed_off=0),
    "gpt2_N4096": dict(B=8, H=16, N=4096, d=64, causal=True, kv=None, boost=True, config_id=3, seed_off=1),
}
L2_FLUSH_BYTES = 256 << 20


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def reduce_max(x, dist=None, device="cpu"):
    """Max of a per-rank float over all ranks (identity without a process group)."""
    if dist is None:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank, world, seconds):
    """Replicas: every rank does the same units; the job's rate is all ranks'
    units over the slowest rank's time."""
    return world * units_per_rank / seconds


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples (200 ms) of SM clock and throttle reasons."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        self.device_index = device_index

    def start(self):
        try:
            uuid = str(torch.cuda.get_device_properties(self.device_index).uuid)
            sel = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            sel = []
        try:
            self.proc = subprocess.Popen(["nvidia-smi", *sel, f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons, n = [], [], set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            n += 1
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": n}


# --------------------------------------------------------------------------- our arm
class Workload:
    """Device-resident inputs, outputs and workspaces of one step."""

    def __init__(self, dev, seed=0):
        from exact_io_aware_10_gb300 import lib

        self.lib = lib
        lib.load()
        P = PREFILL
        s4 = wl.config_seed(seed, 4)
        shp = (P["B"], P["H"], P["N_fb"], P["d"])
        self.Q, self.K, self.V, self.dO = (wl.device_normal_bf16(shp, s4 + i, dev) for i in range(4))
        self.O = torch.empty_like(self.Q)
        self.L = torch.empty(shp[:3], dtype=torch.float32, device=dev)
        self.dQ, self.dK, self.dV = (torch.empty_like(self.Q) for _ in range(3))
        self.ws_b = torch.empty(lib.fa_bwd_workspace_size(*shp), dtype=torch.uint8, device=dev)
        shp64 = (P["B"], P["H"], P["N_f"], P["d"])
        self.Q64, self.K64, self.V64 = (wl.device_normal_bf16(shp64, s4 + 10 + i, dev) for i in range(3))
        self.O64 = torch.empty_like(self.Q64)
        self.L64 = torch.empty(shp64[:3], dtype=torch.float32, device=dev)
        D = DECODE
        sl, table, NB, _ = wl.paged_layout(D["B"], D["L_lo"], D["L_hi"], D["block"], wl.config_seed(seed, 5),
                                           D["max_blocks"])
        self.seq_lens_host = sl
        self.seq_lens = sl.to(dev)
        self.table = table.to(dev)
        cshape = (NB, D["block"], D["Hkv"], D["d"])
        s5 = wl.config_seed(seed, 5)
        self.q = wl.device_normal_bf16((D["B"], D["Hq"], D["d"]), s5 + 1, dev)
        self.kc = wl.device_normal_bf16(cshape, s5 + 2, dev)
        self.vc = wl.device_normal_bf16(cshape, s5 + 3, dev)
        self.o = torch.empty_like(self.q)
        self.lse = torch.empty((D["B"], D["Hq"]), dtype=torch.float32, device=dev)
        self.ws_d = torch.empty(lib.fa_paged_decode_workspace_size(D["B"], D["Hq"], D["d"], D["splits"]),
                                dtype=torch.uint8, device=dev)

    # the four parts of a step, each a single C-ABI call on the current stream
    def fwd16(self):
        self.lib.fa_fwd(self.Q, self.K, self.V, causal=True, O=self.O, LSE=self.L)

    def bwd16(self):
        self.lib.fa_bwd(self.Q, self.K, self.V, self.O, self.dO, self.L, causal=True, dQ=self.dQ, dK=self.dK,
                        dV=self.dV, workspace=self.ws_b)

    def fwd64(self):
        self.lib.fa_fwd(self.Q64, self.K64, self.V64, causal=True, O=self.O64, LSE=self.L64)

    def decode(self):
        self.lib.fa_paged_decode(self.q, self.kc, self.vc, self.table, self.seq_lens, num_splits=DECODE["splits"],
                                 o=self.o, lse=self.lse, workspace=self.ws_d)

    PARTS = ("fwd16", "bwd16", "fwd64", "decode")
    LAUNCHES = {"fwd16": 1, "bwd16": 3, "fwd64": 1, "decode": 2}

    def flops(self):
        P = PREFILL
        f16 = acc.fwd_flops(P["B"], P["H"], P["N_fb"], P["d"], True)
        return {"fwd16": f16, "bwd16": acc.bwd_flops(P["B"], P["H"], P["N_fb"], P["d"], True),
                "fwd64": acc.fwd_flops(P["B"], P["H"], P["N_f"], P["d"], True)}

    def decode_bytes(self):
        D = DECODE
        return acc.decode_bytes(self.seq_lens_host.tolist(), D["Hq"], D["Hkv"], D["d"], D["block"])


class VarlenWorkload:
    """Device-resident packed inputs of one ragged-batch forward (and, where
    the mix has a padded form, the same tokens padded for fa_fwd_ex)."""

    def __init__(self, dev, name, seed=0):
        from exact_io_aware_10_gb300 import lib

        self.lib = lib
        c = VARLEN[name]
        self.c = c
        sd = wl.config_seed(seed, c["config_id"])
        if c["padded_N"] is not None:
            lens = wl.padded_lengths(c["num_seqs"], c["lo"], c["hi"], seed=sd).tolist()
        else:
            lens = wl.varlen_lengths(c["num_seqs"], c["lo"], c["hi"], seed=sd)
        self.lengths = lens
        total = sum(lens)
        cu = [0]
        for n in lens:
            cu.append(cu[-1] + n)
        self.cu = torch.tensor(cu, dtype=torch.int32, device=dev)
        shp = (total, c["H"], c["d"])
        self.Q, self.K, self.V = (wl.device_normal_bf16(shp, sd + 20 + i, dev) for i in range(3))
        self.O = torch.empty_like(self.Q)
        self.L = torch.empty((c["H"], total), dtype=torch.float32, device=dev)
        self.flops = acc.varlen_fwd_flops(lens, c["H"], c["d"], c["causal"])
        self.dO = wl.device_normal_bf16(shp, sd + 24, dev)
        self.dQ, self.dK, self.dV = (torch.empty_like(self.Q) for _ in range(3))
        self.ws = torch.empty(lib.fa_bwd_varlen_workspace_size(len(lens), total, max(lens), c["H"], c["d"]),
                              dtype=torch.uint8, device=dev)
        self.padded = None
        if c["padded_N"] is not None:
            B, N = len(lens), c["padded_N"]
            pshp = (B, c["H"], N, c["d"])
            self.padded = [wl.device_normal_bf16(pshp, sd + 30 + i, dev) for i in range(3)]
            self.Op = torch.empty_like(self.padded[0])
            self.Lp = torch.empty(pshp[:3], dtype=torch.float32, device=dev)
            self.kv = torch.tensor(lens, dtype=torch.int32, device=dev)

    def packed(self):
        self.lib.fa_fwd_varlen(self.Q, self.K, self.V, self.cu, max(self.lengths), causal=self.c["causal"],
                               O=self.O, LSE=self.L)

    def packed_bwd(self):
        self.lib.fa_bwd_varlen(self.Q, self.K, self.V, self.O, self.dO, self.L, self.cu, max(self.lengths),
                               causal=self.c["causal"], dQ=self.dQ, dK=self.dK, dV=self.dV, workspace=self.ws)

    def padded_fwd(self):
        self.lib.fa_fwd(*self.padded, causal=self.c["causal"], kv_lens=self.kv, O=self.Op, LSE=self.Lp)


def time_varlen(dev, seed, steps, warmup, barrier, max_over_ranks, world, peak_tf):
    """TFLOP/s of the packed ragged-batch forward on each VARLEN mix (useful
    FLOPs of the sequences), and of the padded equivalent where there is one."""
    out = {}
    for name in VARLEN:
        v = VarlenWorkload(dev, name, seed)
        parts = ("packed", "packed_bwd") if v.padded is None else ("packed", "padded_fwd")
        _, ms = time_parts(lambda p: getattr(v, p)(), parts, steps, warmup, barrier)
        assert v.lib.fa_get_device_status() == v.lib.FA_OK, "device status word reported an error"
        c = v.c
        r = {"H": c["H"], "d": c["d"], "causal": c["causal"], "num_seqs": c["num_seqs"],
             "lengths": f"U[{c['lo']},{c['hi']}]", "total_tokens": sum(v.lengths), "flops": v.flops}
        for p in parts:
            t = max_over_ranks(ms[p])
            fl = v.flops * (2.5 if p == "packed_bwd" else 1.0)
            tf = world * steps * fl / (t * 1e-3) / 1e12
            key = {"packed": "packed", "packed_bwd": "packed_backward"}.get(p, f"padded_to_{c['padded_N']}")
            r[key] = {"TFLOP/s": tf, "frac": tf / world / peak_tf, "frac_of_nominal": tf / world / NOMINAL["bf16_tflops"],
                      "ms": t / steps}
        out[f"varlen_{name}"] = r
        del v
        torch.cuda.empty_cache()
    return out


class PagedPrefillWorkload:
    """Device-resident chunks, paged cache and block table of PAGED_PREFILL."""

    def __init__(self, dev, seed=0):
        from exact_io_aware_10_gb300 import lib

        self.lib = lib
        c = PAGED_PREFILL
        sd = wl.config_seed(seed, c["config_id"])
        g = torch.Generator().manual_seed(sd)
        prefix = torch.randint(c["prefix_lo"], c["prefix_hi"] + 1, (c["num_seqs"],), generator=g).tolist()
        self.q_lens = [c["q_len"]] * c["num_seqs"]
        self.kv_lens = [p + c["q_len"] for p in prefix]
        sl, table, NB, _ = wl.paged_layout(c["num_seqs"], 0, 0, c["block_size"], sd, None, self.kv_lens)
        cu = [0]
        for n in self.q_lens:
            cu.append(cu[-1] + n)
        self.cu = torch.tensor(cu, dtype=torch.int32, device=dev)
        self.sl, self.table = sl.to(dev), table.to(dev)
        self.q = wl.device_normal_bf16((cu[-1], c["Hq"], c["d"]), sd + 1, dev)
        cshape = (NB, c["block_size"], c["Hkv"], c["d"])
        self.kc = wl.device_normal_bf16(cshape, sd + 2, dev)
        self.vc = wl.device_normal_bf16(cshape, sd + 3, dev)
        self.o = torch.empty_like(self.q)
        self.lse = torch.empty((c["Hq"], cu[-1]), dtype=torch.float32, device=dev)
        self.flops = acc.paged_prefill_flops(self.q_lens, self.kv_lens, c["Hq"], c["d"], True)

    def run(self):
        self.lib.fa_paged_prefill(self.q, self.kc, self.vc, self.table, self.cu, self.sl, max(self.q_lens),
                                  causal=True, o=self.o, lse=self.lse)


def time_paged_prefill(dev, seed, steps, warmup, barrier, max_over_ranks, world, peak_tf):
    w = PagedPrefillWorkload(dev, seed)
    _, ms = time_parts(lambda p: w.run(), ("run",), steps, warmup, barrier)
    assert w.lib.fa_get_device_status() == w.lib.FA_OK, "device status word reported an error"
    t = max_over_ranks(ms["run"])
    tf = world * steps * w.flops / (t * 1e-3) / 1e12
    c = PAGED_PREFILL
    out = {"num_seqs": c["num_seqs"], "q_len": c["q_len"], "prefix": f"U[{c['prefix_lo']},{c['prefix_hi']}]",
           "Hq": c["Hq"], "Hkv": c["Hkv"], "d": c["d"], "block_size": c["block_size"], "causal": "bottom-right",
           "flops": w.flops, "TFLOP/s": tf, "frac": tf / world / peak_tf,
           "frac_of_nominal": tf / world / NOMINAL["bf16_tflops"], "ms": t / steps}
    del w
    torch.cuda.empty_cache()
    return out


def time_block_sparse(w, steps, warmup, barrier, max_over_ranks, world, peak_tf, part_ms):
    """TFLOP/s (useful FLOPs: visible pairs of kept blocks) of the block-sparse
    forward at N = 16384 and 65536 on the step's own inputs, with its speed-up
    over the dense forward of the same step."""
    P = PREFILL
    out = {"mask": f"butterfly + local window of {BLOCK_SPARSE_WINDOW} key blocks, 128 x 128 blocks, causal"}
    for tag, (Q, K, V, O, L, dense_part) in {"N16384": (w.Q, w.K, w.V, w.O, w.L, "fwd16"),
                                             "N65536": (w.Q64, w.K64, w.V64, w.O64, w.L64, "fwd64")}.items():
        N = Q.shape[2]
        m = wl.block_mask(N // 128, "butterfly", window=BLOCK_SPARSE_WINDOW)
        flops = acc.block_sparse_flops(m.numpy(), P["B"], P["H"], N, P["d"], True)
        md = m.to(Q.device)
        _, ms = time_parts(lambda p: w.lib.fa_fwd_block_sparse(Q, K, V, md, causal=True, O=O, LSE=L), ("bs",),
                           steps, warmup, barrier)
        assert w.lib.fa_get_device_status() == w.lib.FA_OK, "device status word reported an error"
        t = max_over_ranks(ms["bs"])
        tf = world * steps * flops / (t * 1e-3) / 1e12
        out[tag] = {"kept_fraction_of_causal_pairs": flops / acc.fwd_flops(P["B"], P["H"], N, P["d"], True),
                    "flops": flops, "TFLOP/s": tf, "frac": tf / world / peak_tf,
                    "frac_of_nominal": tf / world / NOMINAL["bf16_tflops"], "ms": t / steps,
                    "speedup_vs_dense_forward": (part_ms[dense_part] / steps) / (t / steps)}
    return out


def time_decode_step(dev, seed, steps, warmup, barrier, max_over_ranks):
    """Per-step time of a small-batch decode step (one paged decode per layer):
    eager calls with 16 splits (split + combine) or 1 split (one fused launch),
    and the same step replayed as a CUDA graph.  Event time spans the whole
    step, so host launch gaps count."""
    from exact_io_aware_10_gb300 import lib

    c = DECODE_STEP
    sd = wl.config_seed(seed, c["config_id"])
    sl, table, NB, _ = wl.paged_layout(c["B"], 0, 0, 16, sd, None, [c["context"]] * c["B"])
    sl, table = sl.to(dev), table.to(dev)
    layers = []
    for i in range(c["layers"]):
        q = wl.device_normal_bf16((c["B"], c["Hq"], c["d"]), sd + 10 * i + 1, dev)
        kc = wl.device_normal_bf16((NB, 16, c["Hkv"], c["d"]), sd + 10 * i + 2, dev)
        vc = wl.device_normal_bf16((NB, 16, c["Hkv"], c["d"]), sd + 10 * i + 3, dev)
        layers.append((q, kc, vc, torch.empty_like(q), torch.empty(c["B"], c["Hq"], dtype=torch.float32,
                                                                   device=dev)))
    ws = torch.empty(lib.fa_paged_decode_workspace_size(c["B"], c["Hq"], c["d"], 16), dtype=torch.uint8, device=dev)

    def eager(splits):
        def run(_):
            for q, kc, vc, o, lse in layers:
                lib.fa_paged_decode(q, kc, vc, table, sl, num_splits=splits, o=o, lse=lse, workspace=ws)
        return run

    graphs = {s_: lib.DecodeGraph(layers, table, sl, num_splits=s_, workspace=ws) for s_ in (16, 1)}
    out = {"layers": c["layers"], "B": c["B"], "Hq": c["Hq"], "Hkv": c["Hkv"], "context": c["context"]}
    for name, fn, launches in (("eager_splits16", eager(16), 2 * c["layers"]),
                               ("eager_splits1", eager(1), c["layers"]),
                               ("graph_splits16", lambda _: graphs[16].launch(), graphs[16].kernel_count),
                               ("graph_splits1", lambda _: graphs[1].launch(), graphs[1].kernel_count)):
        _, ms = time_parts(fn, ("step",), steps, warmup, barrier)
        out[name] = {"ms_per_step": max_over_ranks(ms["step"]) / steps, "kernel_launches_per_step": launches}
    assert lib.fa_get_device_status() == lib.FA_OK, "device status word reported an error"
    for g in graphs.values():
        g.close()
    out["speedup_graph_vs_eager_splits16"] = out["eager_splits16"]["ms_per_step"] / out["graph_splits16"][
        "ms_per_step"]
    return out


def time_small_configs(dev, seed, steps, warmup, barrier, max_over_ranks, world, peak_tf):
    """Forward and backward TFLOP/s of the SMALL configurations, L2 flushed
    before every timed call.  Returns {name: {...}}."""
    from exact_io_aware_10_gb300 import lib

    flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    out = {}
    for name, c in SMALL.items():
        sd = wl.config_seed(seed, c["config_id"]) + c["seed_off"]
        shp = (c["B"], c["H"], c["N"], c["d"])
        if c["boost"]:
            x = wl.boosted_inputs(*shp, seed=sd)
            Q, K, V, dO = (t.to(dev) for t in (x.Q, x.K, x.V, x.dO))
        else:
            Q, K, V, dO = (wl.device_normal_bf16(shp, sd + i, dev) for i in range(4))
        kv_host = wl.padded_lengths(c["B"], c["kv"][0], c["kv"][1], seed=sd) if c["kv"] else None
        kv = None if kv_host is None else kv_host.to(dev)
        O = torch.empty_like(Q)
        L = torch.empty(shp[:3], dtype=torch.float32, device=dev)
        dQ, dK, dV = (torch.empty_like(Q) for _ in range(3))
        ws = torch.empty(lib.fa_bwd_workspace_size(*shp), dtype=torch.uint8, device=dev)
        causal = c["causal"]

        def run(p):
            if p == "fwd":
                lib.fa_fwd(Q, K, V, causal=causal, kv_lens=kv, O=O, LSE=L)
            else:
                lib.fa_bwd(Q, K, V, O, dO, L, causal=causal, kv_lens=kv, dQ=dQ, dK=dK, dV=dV, workspace=ws)

        _, ms = time_parts(run, ("fwd", "bwd"), steps, warmup, barrier, flush=flush_buf.zero_)
        assert lib.fa_get_device_status() == lib.FA_OK, "device status word reported an error"
        formula = acc.fwd_flops(*shp, causal)
        eff = acc.fwd_flops_padded(c["H"], c["N"], c["d"], kv_host.tolist()) if kv_host is not None else formula
        r = {"shape": f"B{c['B']} H{c['H']} N{c['N']} d{c['d']}", "causal": causal,
             "key_padding": None if kv_host is None else f"U[{c['kv'][0]},{c['kv'][1]}]",
             "boosted_logits": c["boost"], "flops_fwd": eff, "flops_fwd_formula": formula}
        for p, mult in (("fwd", 1.0), ("bwd", 2.5)):
            t = max_over_ranks(ms[p])
            tf = world * steps * mult * eff / (t * 1e-3) / 1e12
            r[p] = {"TFLOP/s": tf, "frac": tf / world / peak_tf, "frac_of_nominal": tf / world / NOMINAL["bf16_tflops"],
                    "ms": t / steps}
            if kv_host is not None:
                r[p]["formula_TFLOP/s"] = world * steps * mult * formula / (t * 1e-3) / 1e12
        out[name] = r
        del Q, K, V, dO, O, L, dQ, dK, dV, ws
        torch.cuda.empty_cache()
    del flush_buf
    torch.cuda.empty_cache()
    return out


class HostBuffers:
    """Pinned host copies of a step's inputs and outputs for the end-to-end run.
    A decode step's inputs are its queries, block table and sequence lengths:
    the paged K/V cache is state that stays on the device between decode
    steps (as a serving engine keeps it), so it is not re-uploaded every step;
    its one-time upload is timed separately (`cache_upload`)."""

    def __init__(self, w: Workload):
        self.w = w
        self.inputs = {"fwd16": [w.Q, w.K, w.V], "bwd16": [w.dO], "fwd64": [w.Q64, w.K64, w.V64],
                       "decode": [w.q, w.table, w.seq_lens]}
        self.outputs = {"fwd16": [w.O, w.L], "bwd16": [w.dQ, w.dK, w.dV], "fwd64": [w.O64, w.L64],
                        "decode": [w.o, w.lse]}
        self.h_in = {k: [t.cpu().pin_memory() for t in v] for k, v in self.inputs.items()}
        self.h_out = {k: [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in v]
                      for k, v in self.outputs.items()}

    def bytes(self, part):
        h2d = sum(t.numel() * t.element_size() for t in self.h_in[part])
        d2h = sum(t.numel() * t.element_size() for t in self.h_out[part])
        return h2d, d2h

    def cache_upload(self):
        """Bytes and seconds of one host-to-device upload of the paged K/V
        cache from pinned memory (one copy per cache tensor)."""
        hk, hv = (t.cpu().pin_memory() for t in (self.w.kc, self.w.vc))
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        self.w.kc.copy_(hk, non_blocking=True)
        self.w.vc.copy_(hv, non_blocking=True)
        b.record()
        torch.cuda.synchronize()
        nbytes = sum(t.numel() * t.element_size() for t in (hk, hv))
        del hk, hv
        return nbytes, a.elapsed_time(b) * 1e-3

    def run(self, part):
        for d, h in zip(self.inputs[part], self.h_in[part]):
            d.copy_(h, non_blocking=True)
        getattr(self.w, part)()
        for h, d in zip(self.h_out[part], self.outputs[part]):
            h.copy_(d, non_blocking=True)

    # parts whose kernels read each part's input buffers (bwd16 reads the
    # forward's Q, K, V as well as its own dO)
    READERS = {"fwd16": ("fwd16", "bwd16"), "bwd16": ("bwd16",), "fwd64": ("fwd64",), "decode": ("decode",)}

    def time_pipelined(self, parts, steps, warmup):
        """Milliseconds per step of `parts` with every step's inputs copied in
        and outputs copied out, the copies on their own streams: step s's
        inputs load while earlier kernels run, and its outputs drain while
        later ones run.  A copy into a buffer waits for the previous step's
        kernels that read it; a kernel waits for its inputs and for the
        previous step's read-out of its outputs."""
        comp = torch.cuda.current_stream()
        h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
        ev = {k: {p: torch.cuda.Event() for p in parts} for k in ("h2d", "comp", "d2h")}
        started = set()

        def one_step():
            for p in parts:
                for r in self.READERS[p]:
                    if r in started and r in parts:
                        h2d.wait_event(ev["comp"][r])
                with torch.cuda.stream(h2d):
                    for d, h in zip(self.inputs[p], self.h_in[p]):
                        d.copy_(h, non_blocking=True)
                ev["h2d"][p].record(h2d)
            for p in parts:
                comp.wait_event(ev["h2d"][p])
                if p in started:
                    comp.wait_event(ev["d2h"][p])
                getattr(self.w, p)()
                ev["comp"][p].record(comp)
                d2h.wait_event(ev["comp"][p])
                with torch.cuda.stream(d2h):
                    for h, d in zip(self.h_out[p], self.outputs[p]):
                        h.copy_(d, non_blocking=True)
                ev["d2h"][p].record(d2h)
                started.add(p)

        for _ in range(warmup):
            one_step()
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(h2d)
        for _ in range(steps):
            one_step()
        t1.record(d2h)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1) / steps


def source_sha(rel):
    with open(os.path.join(ROOT, rel), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def time_parts(fn_for_part, parts, steps, warmup, barrier, flush=None):
    """CUDA-event time of every call of every part over `steps` steps (after
    `warmup` untimed ones), on the current stream.  `flush`, if given, runs
    before each timed call, outside its events (an L2 flush)."""
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        for p in parts:
            fn_for_part(p)
    torch.cuda.synchronize()
    barrier()
    ev = {p: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
          for p in parts}
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for k in range(steps):
        for p in parts:
            if flush is not None:
                flush()
            ev[p][k][0].record(stream)
            fn_for_part(p)
            ev[p][k][1].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    barrier()
    per_part = {p: sum(a.elapsed_time(b) for a, b in ev[p]) for p in parts}  # ms over all steps
    return t0.elapsed_time(t1), per_part


def recorded_traffic(which):
    """ncu DRAM bytes per launch recorded for kernel family `which`, keyed by
    shape, or None when none were taken on the current source."""
    rec = TRAFFIC_RECORD[which]
    if not rec["sha256"] or rec["sha256"] != source_sha(rec["source"]) or not rec["bytes"]:
        return None
    return rec["bytes"]


def build_roofline(part_ms, flops, dbytes, K, peaks, peak_src):
    """The roofline record: the dominant kernel (the forward) in the standard
    keys, then flat bwd_* and decode_* blocks for the backward call and the
    decode pair.  achieved = algorithmic FLOPs (bytes) per call / CUDA-event
    time per call; traffic = ncu DRAM bytes per launch (null when not taken on
    the current source)."""
    P, D = PREFILL, DECODE
    peak_tf, peak_hbm = peaks["bf16_tflops"], peaks["hbm_gbs"]
    # forward: one launch of fwd_kernel<128> per fa_fwd call, two calls per step
    fwd_ms = part_ms["fwd16"] + part_ms["fwd64"]
    fwd_flops_step = flops["fwd16"] + flops["fwd64"]
    achieved = K * fwd_flops_step / (fwd_ms * 1e-3) / 1e12
    comp = {"N16384": acc.fwd_bytes(P["B"], P["H"], P["N_fb"], P["d"]),
            "N65536": acc.fwd_bytes(P["B"], P["H"], P["N_f"], P["d"])}
    t_fwd = recorded_traffic("fwd")
    traffic = sum(t_fwd[k] for k in comp) / 2.0 if t_fwd and all(k in t_fwd for k in comp) else None
    r = {"kernel": "fwd_kernel<128> (fa_fwd)", "bound": "tensor", "achieved": achieved, "peak": peak_tf,
         "unit": "TFLOP/s", "frac": achieved / peak_tf, "traffic": traffic,
         "compulsory_bytes": sum(comp.values()) / 2.0,
         "traffic_N16384": t_fwd.get("N16384") if t_fwd else None,
         "traffic_N65536": t_fwd.get("N65536") if t_fwd else None,
         "compulsory_N16384": comp["N16384"], "compulsory_N65536": comp["N65536"],
         "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum, one launch per shape",
         "peak_source": f"{peak_src} bf16_tflops (burst)",
         "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"],
         "frac_of_nominal": achieved / NOMINAL["bf16_tflops"],
         "frac_of_nominal_nvl72": achieved / NOMINAL["bf16_tflops_nvl72"],
         "nominal_peak": NOMINAL["bf16_tflops"],
         "launches_per_step": 2, "flops_per_step": fwd_flops_step,
         "fwd_N16384_TFLOP/s": K * flops["fwd16"] / (part_ms["fwd16"] * 1e-3) / 1e12,
         "fwd_N65536_TFLOP/s": K * flops["fwd64"] / (part_ms["fwd64"] * 1e-3) / 1e12}
    # backward: one fa_bwd call = bwd_pre, bwd_main, bwd_dq launches
    bwd = K * flops["bwd16"] / (part_ms["bwd16"] * 1e-3) / 1e12
    t_bwd = recorded_traffic("bwd")
    r.update({"bwd_kernel": "bwd_pre + bwd_main_kernel<128> + bwd_dq (fa_bwd, N=16384)", "bwd_bound": "tensor",
              "bwd_achieved": bwd, "bwd_frac": bwd / peak_tf,
              "bwd_frac_of_sustained": bwd / peaks["bf16_tflops_sustained"],
              "bwd_frac_of_nominal": bwd / NOMINAL["bf16_tflops"],
              "bwd_frac_of_nominal_nvl72": bwd / NOMINAL["bf16_tflops_nvl72"],
              "bwd_traffic": (sum(t_bwd[k] for k in ("N16384_pre", "N16384_main", "N16384_dq"))
                              if t_bwd and all(k in t_bwd for k in ("N16384_pre", "N16384_main", "N16384_dq"))
                              else None),
              "bwd_main_traffic": t_bwd.get("N16384_main") if t_bwd else None,
              "bwd_compulsory_bytes": acc.bwd_bytes(P["B"], P["H"], P["N_fb"], P["d"]),
              "bwd_flops_per_call": flops["bwd16"]})
    # decode: one fa_paged_decode call = split + combine launches
    dec = K * dbytes / (part_ms["decode"] * 1e-3) / 1e9
    t_dec = recorded_traffic("decode")
    r.update({"decode_kernel": "decode_split_kernel<128> + decode_combine_kernel<128> (fa_paged_decode)",
              "decode_bound": "hbm", "decode_achieved": dec, "decode_peak": peak_hbm, "decode_unit": "GB/s",
              "decode_frac": dec / peak_hbm, "decode_frac_of_nominal": dec / NOMINAL["hbm_gbs"],
              "decode_traffic": t_dec.get("B64") if t_dec else None,
              "decode_algorithmic_bytes": dbytes, "decode_peak_source": f"{peak_src} hbm_gbs"})
    return r


def small_roofline_keys(small):
    """Flat roofline keys of the small configurations (TFLOP/s and fraction of
    the measured peak per call)."""
    r = {}
    for name, v in small.items():
        for p in ("fwd", "bwd"):
            r[f"{name}_{p}_TFLOP/s"] = v[p]["TFLOP/s"]
            r[f"{name}_{p}_frac"] = v[p]["frac"]
            r[f"{name}_{p}_ms"] = v[p]["ms"]
            if "formula_TFLOP/s" in v[p]:
                r[f"{name}_{p}_formula_TFLOP/s"] = v[p]["formula_TFLOP/s"]
    return r


def run_ours(args):
    rank, world, local = dist_env()
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    def barrier():
        if dist is not None:
            dist.barrier()

    def max_over_ranks(x):
        return reduce_max(x, dist, dev)

    w = Workload(dev, seed=args.seed)
    peaks, peak_src = load_peaks()
    flops = w.flops()
    dbytes = w.decode_bytes()

    sampler = ClockSampler(local)
    sampler.start()
    total_ms, part_ms = time_parts(lambda p: getattr(w, p)(), Workload.PARTS, args.steps, args.warmup, barrier)
    clocks = sampler.stop()
    assert w.lib.fa_get_device_status() == w.lib.FA_OK, "device status word reported an error"
    total_ms = max_over_ranks(total_ms)
    part_ms = {p: max_over_ranks(v) for p, v in part_ms.items()}

    K = args.steps
    prefill_parts = ("fwd16", "bwd16", "fwd64")
    prefill_ms = sum(part_ms[p] for p in prefill_parts)
    prefill_flops = sum(flops.values())
    value = whole_job_rate(K * prefill_flops, world, prefill_ms * 1e-3) / 1e12
    dec_gbs = whole_job_rate(K * dbytes, world, part_ms["decode"] * 1e-3) / 1e9
    peak_tf, peak_hbm = peaks["bf16_tflops"], peaks["hbm_gbs"]

    def tf(p):
        return K * flops[p] / (part_ms[p] * 1e-3) / 1e12

    def tf_part(p):
        v = tf(p)
        return {"TFLOP/s": v, "frac": v / peak_tf, "frac_of_nominal": v / NOMINAL["bf16_tflops"],
                "ms": part_ms[p] / K}

    parts = {
        "fwd_N16384": tf_part("fwd16"),
        "bwd_N16384": tf_part("bwd16"),
        "fwd_N65536": tf_part("fwd64"),
        "decode": {"GB/s": dec_gbs / world, "frac": dec_gbs / world / peak_hbm,
                   "frac_of_nominal": dec_gbs / world / NOMINAL["hbm_gbs"], "ms": part_ms["decode"] / K},
        "denominators": {"measured_bf16_tflops": peak_tf, "measured_hbm_gbs": peak_hbm,
                         "nominal_bf16_tflops": NOMINAL["bf16_tflops"], "nominal_hbm_gbs": NOMINAL["hbm_gbs"],
                         "source": peak_src},
    }

    roofline = build_roofline(part_ms, flops, dbytes, K, peaks, peak_src)

    # end to end: the same parts through the C ABI with pinned host buffers,
    # host->device inputs and device->host outputs inside the timed region
    hb = HostBuffers(w)
    e2e_steps = max(3, min(args.steps, 10))
    e2e_total, e2e_part = time_parts(hb.run, Workload.PARTS, e2e_steps, 1, barrier)
    e2e_part = {p: max_over_ranks(v) for p, v in e2e_part.items()}
    e2e_prefill_ms = sum(e2e_part[p] for p in prefill_parts)
    e2e_value = world * e2e_steps * prefill_flops / (e2e_prefill_ms * 1e-3) / 1e12
    h2d = sum(hb.bytes(p)[0] for p in Workload.PARTS)
    d2h = sum(hb.bytes(p)[1] for p in Workload.PARTS)
    # the same step with the copies overlapped with the kernels (copy engines
    # on their own streams), prefill parts and decode pipelined separately
    pre_ms = max_over_ranks(hb.time_pipelined(prefill_parts, e2e_steps, 1))
    dec_ms = max_over_ranks(hb.time_pipelined(("decode",), e2e_steps, 1))
    pipe_value = world * prefill_flops / (pre_ms * 1e-3) / 1e12
    cache_bytes, cache_s = hb.cache_upload()
    e2e = {"value": pipe_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "decode_GB/s": world * dbytes / (dec_ms * 1e-3) / 1e9,
           "ms_per_step": pre_ms + dec_ms,
           "overlap": "inputs copied in and outputs copied out every step on separate copy streams, "
                      "overlapped with the kernels of neighbouring parts and steps",
           "decode_note": "decode inputs per step are q, block table and lengths; the paged K/V cache stays "
                          "resident (uploaded once, timed in decode_cache_upload_GB/s)",
           "decode_cache_bytes": cache_bytes, "decode_cache_upload_GB/s": cache_bytes / cache_s / 1e9,
           "serial": {"value": e2e_value, "unit": "TFLOP/s",
                      "decode_GB/s": world * e2e_steps * dbytes / (e2e_part["decode"] * 1e-3) / 1e9,
                      "ms_per_step": max_over_ranks(e2e_total) / e2e_steps,
                      "note": "copies and kernels in one stream, nothing overlapped"}}

    # the encoder- and decoder-shaped configurations (d = 64), after the step
    small = None
    if not args.skip_small_configs:
        small = time_small_configs(dev, args.seed, args.steps, args.warmup, barrier, max_over_ranks, world, peak_tf)
        roofline.update(small_roofline_keys(small))

    next_rows = None
    if not args.skip_next_rows:
        next_rows = time_varlen(dev, args.seed, args.steps, args.warmup, barrier, max_over_ranks, world, peak_tf)
        next_rows["paged_prefill"] = time_paged_prefill(dev, args.seed, args.steps, args.warmup, barrier,
                                                        max_over_ranks, world, peak_tf)
        next_rows["block_sparse"] = time_block_sparse(w, args.steps, args.warmup, barrier, max_over_ranks, world,
                                                      peak_tf, part_ms)
        next_rows["decode_step"] = time_decode_step(dev, args.seed, args.steps, args.warmup, barrier, max_over_ranks)
        next_rows["note"] = "timed after the step, outside value and ms_per_step; TFLOP/s count useful FLOPs only"

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_sample(args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": total_ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD, "parallelism": f"replicas{world}",
                       "l2": "step: every kernel's inputs exceed the 129 MB L2 (no flush); small configs: "
                             "L2 flushed before each call",
                       "value_is": "fwd+bwd TFLOP/s over parts 1-3; decode GB/s in 'decode'"},
            "decode": {"value": dec_gbs, "unit": "GB/s", "frac": dec_gbs / world / peak_hbm,
                       "peak": peak_hbm, "peak_source": f"{peak_src} hbm_gbs", "bytes_per_step": dbytes},
            "parts": parts, "roofline": roofline, "e2e": e2e, "cpu_baseline": cpu,
            "gpu_launches": K * sum(Workload.LAUNCHES.values()), "clocks": clocks, "configs": small,
            "next_rows": next_rows,
        }
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()


# --------------------------------------------------------------------------- oracle (CPU)
def _oracle_prefill_sample(seed, head, n_prefix):
    """Oracle forward + backward of one head of the long-prefill workload,
    restricted to its first ``n_prefix`` positions (a causal prefix is itself a
    causal attention problem).  Returns (seconds, algorithmic FLOPs)."""
    import oracle

    P = PREFILL
    g = torch.Generator().manual_seed(wl.config_seed(seed, 4) * 31 + head)
    shp = (1, 1, n_prefix, P["d"])
    Q, K, V, dO = (torch.randn(*shp, generator=g).to(torch.bfloat16) for _ in range(4))
    t0 = time.perf_counter()
    oracle.attention_forward(Q, K, V, causal=True)
    oracle.attention_backward(Q, K, V, dO, causal=True)
    dt = time.perf_counter() - t0
    return dt, acc.fwd_flops(1, 1, n_prefix, P["d"], True) + acc.bwd_flops(1, 1, n_prefix, P["d"], True)


def _oracle_decode_sample(seed, n_seq):
    import oracle

    D = DECODE
    sl, _, _, g = wl.paged_layout(D["B"], D["L_lo"], D["L_hi"], D["block"], wl.config_seed(seed, 5), D["max_blocks"])
    lens = sl[:n_seq].tolist()
    P = wl.paged_inputs(n_seq, D["Hq"], D["Hkv"], D["d"], 0, 0, D["block"], seed=seed + 77, seq_lens=lens)
    t0 = time.perf_counter()
    oracle.paged_decode(P.q, P.k_cache, P.v_cache, P.block_table, P.seq_lens, D["block"])
    dt = time.perf_counter() - t0
    return dt, acc.decode_bytes(lens, D["Hq"], D["Hkv"], D["d"], D["block"])


def _row_subset(N, every=64):
    """Every `every`-th query row plus the first and the last."""
    return np.unique(np.concatenate([np.arange(0, N, every), [0, N - 1]]))


def _causal_row_flops(rows, d):
    """Algorithmic forward FLOPs of the given causal rows: 4 d per visible key."""
    return 4.0 * d * float(np.sum(np.asarray(rows) + 1))


def cpu_baseline_sample(budget_s=30.0, seed=0):
    """The oracle as it stands, timed on this host's cores.  Following the
    measurement plan: the tiny, BERT-shaped and GPT-2 N=1024 configurations in
    full (forward + backward), the GPT-2 N=4096 one on whole heads; the
    long-context rows (16K forward, 16K backward, 64K forward) on a row subset
    (every 64th row plus the first and the last) of as many heads as the budget
    allows.  Sampled items report rows/s (or heads/s) and the full-size time
    extrapolated from it, labelled as extrapolated.  `value` is the algorithmic
    FLOPs of everything timed over the seconds it took."""
    import oracle

    out = {"unit": "TFLOP/s", "cores": NCORES, "kind": "oracle"}
    tot_fl, tot_s = 0.0, 0.0
    share = budget_s / 30.0  # the item budgets below are sized for 30 s

    def tick():
        return time.perf_counter()

    # config 1, in full: B1 H2 N256 d64, non-causal and causal
    x = wl.dense_inputs(1, 2, 256, 64, seed=wl.config_seed(seed, 1))
    t0 = tick()
    for causal in (False, True):
        oracle.attention_forward(x.Q, x.K, x.V, causal=causal)
        oracle.attention_backward(x.Q, x.K, x.V, x.dO, causal=causal)
    dt = tick() - t0
    fl = 3.5 * (acc.fwd_flops(1, 2, 256, 64, False) + acc.fwd_flops(1, 2, 256, 64, True))
    out["cfg1_s"] = dt
    tot_fl, tot_s = tot_fl + fl, tot_s + dt
    # config 2, in full: B16 H16 N512 d64, key padding U[128, 512]
    c = SMALL["bert"]
    sd = wl.config_seed(seed, c["config_id"])
    kv = wl.padded_lengths(c["B"], c["kv"][0], c["kv"][1], seed=sd)
    x = wl.dense_inputs(c["B"], c["H"], c["N"], c["d"], seed=sd)
    t0 = tick()
    oracle.attention_forward(x.Q, x.K, x.V, kv_lens=kv.numpy())
    oracle.attention_backward(x.Q, x.K, x.V, x.dO, kv_lens=kv.numpy())
    dt = tick() - t0
    out["cfg2_bert_s"] = dt
    tot_fl, tot_s = tot_fl + 3.5 * acc.fwd_flops_padded(c["H"], c["N"], c["d"], kv.tolist()), tot_s + dt
    # config 3, N = 1024 in full; N = 4096 on whole heads, extrapolated to all
    for name, heads_cap in (("gpt2_N1024", None), ("gpt2_N4096", max(1, int(2 * share)))):
        c = SMALL[name]
        sd = wl.config_seed(seed, c["config_id"]) + c["seed_off"]
        B, H = (c["B"], c["H"]) if heads_cap is None else (1, heads_cap)
        x = wl.boosted_inputs(B, H, c["N"], c["d"], seed=sd)
        t0 = tick()
        oracle.attention_forward(x.Q, x.K, x.V, causal=True)
        oracle.attention_backward(x.Q, x.K, x.V, x.dO, causal=True)
        dt = tick() - t0
        tot_fl, tot_s = tot_fl + 3.5 * acc.fwd_flops(B, H, c["N"], c["d"], True), tot_s + dt
        if heads_cap is None:
            out[f"cfg3_{name}_s"] = dt
        else:
            out[f"cfg3_{name}_heads_timed"] = B * H
            out[f"cfg3_{name}_s_extrapolated"] = dt * c["B"] * c["H"] / (B * H)
    # config 4 on a row subset of each head (long-context prefill, d = 128)
    P = PREFILL
    for item, N, bwd, cap_s in (("fwd_N16384", P["N_fb"], False, 2.0), ("bwd_N16384", P["N_fb"], True, 5.0),
                                ("fwd_N65536", P["N_f"], False, 6.0)):
        rows = _row_subset(N)
        n_rows, secs, fl, heads = 0, 0.0, 0.0, 0
        while heads < P["H"] and (heads == 0 or secs < cap_s * share):
            g = torch.Generator().manual_seed(wl.config_seed(seed, 4) * 31 + 1000 * heads + N)
            shp = (1, 1, N, P["d"])
            Q, K, V, dO = (torch.randn(*shp, generator=g).to(torch.bfloat16) for _ in range(4))
            t0 = tick()
            if bwd:
                oracle.attention_backward_rows(Q, K, V, dO, rows, causal=True)
            else:
                oracle.attention_forward_rows(Q, K, V, rows, causal=True)
            secs += tick() - t0
            fl += _causal_row_flops(rows, P["d"]) * (2.5 if bwd else 1.0)
            n_rows += len(rows)
            heads += 1
        rate = n_rows / secs
        out[f"{item}_rows_per_s"] = rate
        out[f"{item}_heads_timed"] = heads
        out[f"{item}_s_extrapolated"] = P["B"] * P["H"] * N / rate
        tot_fl, tot_s = tot_fl + fl, tot_s + secs
    # paged decode on two sequences
    d_dt, d_bytes = _oracle_decode_sample(seed, 2)
    out["decode_GB/s"] = d_bytes / d_dt / 1e9
    out["value"] = tot_fl / tot_s / 1e12
    out["seconds"] = tot_s + d_dt
    out["sample"] = ("fp64 numpy oracle: cfg 1-2 and GPT-2 N1024 in full, N4096 on whole heads, 16K/64K on every "
                     "64th row; *_extrapolated = full size")
    return out


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    fl_tot, t_tot = 0.0, 0.0
    for k in range(args.warmup + args.steps):
        dt, f = _oracle_prefill_sample(args.seed, k % PREFILL["H"], args.ref_prefix)
        if k >= args.warmup:
            fl_tot += f
            t_tot += dt
    value = fl_tot / t_tot / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * t_tot / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
        "config": {"workload": WORKLOAD, "sample": f"one head per step, causal prefix N={args.ref_prefix}",
                   "parallelism": "cpu"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": NCORES, "kind": "oracle",
                         "sample": f"fp64 numpy oracle fwd+bwd, one head of the long-prefill workload per step, "
                                   f"causal prefix N={args.ref_prefix}, d=128"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=30.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--skip-small-configs", action="store_true",
                    help="skip the BERT- and GPT-2-shaped d = 64 forward/backward timings")
    ap.add_argument("--skip-next-rows", action="store_true",
                    help="skip the ragged-batch, paged-prefill, block-sparse and decode-step timings")
    ap.add_argument("--ref-prefix", type=int, default=2048)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
