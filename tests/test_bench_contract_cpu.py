"""The bench's JSON-line contract, checked on the host.

The reference arm times the oracle on the host's cores, so it runs here without
a GPU: one JSON line from rank 0 with the contract's keys, nothing from other
ranks.  The product arm has no CPU path: without a GPU it must exit non-zero
and print no result line.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BENCH = os.path.join(ROOT, "bench.py")
SMALL = ["--steps", "2", "--warmup", "3", "--ref-prefix", "128"]


def _json_lines(text):
    out = []
    for line in text.splitlines():
        line = line.strip()
        if line.startswith("{"):
            out.append(json.loads(line))
    return out


def _run(cmd, env=None, timeout=240):
    return subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=timeout, env=env)


def test_reference_arm_prints_one_contract_line():
    r = _run([sys.executable, BENCH, "--impl", "reference"] + SMALL)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    j = lines[0]
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in j, key
    assert j["impl"] == "reference"
    assert j["unit"] == "TFLOP/s" and j["higher_is_better"] is True
    assert j["n_gpus"] == 1 and j["steps"] == 2 and j["warmup"] == 3
    assert j["value"] > 0 and j["ms_per_step"] > 0
    assert "workload" in j["config"]
    cb = j["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == j["value"] and cb["sample"]
    e2e = j["e2e"]
    assert e2e["value"] == j["value"] and e2e["unit"] == j["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_warmup_below_three_is_refused():
    r = _run([sys.executable, BENCH, "--impl", "reference", "--steps", "2", "--warmup", "2"])
    assert r.returncode != 0
    assert not _json_lines(r.stdout)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_reference_arm_under_two_ranks_prints_once():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), BENCH, "--impl", "reference",
           "--gpus", "2"] + SMALL
    r = _run(cmd)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    assert lines[0]["impl"] == "reference" and lines[0]["n_gpus"] == 2


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the behaviour on a host without a GPU")
def test_product_arm_fails_loudly_without_a_gpu():
    r = _run([sys.executable, BENCH, "--steps", "3", "--warmup", "3", "--no-cpu-baseline", "--skip-next-rows"])
    assert r.returncode != 0
    assert not _json_lines(r.stdout)


def test_roofline_record_is_flat_and_consistent():
    # every kernel's figures sit in flat scalar keys (a reader that keeps only
    # scalars keeps them all); fractions are achieved over the stated peaks
    sys.path.insert(0, ROOT)
    import bench

    peaks = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
    K = 10
    part_ms = {"fwd16": 8.0, "bwd16": 26.0, "fwd64": 115.0, "decode": 7.0}
    flops = {"fwd16": 1.0995e12, "bwd16": 2.7488e12, "fwd64": 1.7592e13}
    r = bench.build_roofline(part_ms, flops, 4.4e9, K, peaks, "measured")
    small = {"bert": {"fwd": {"TFLOP/s": 400.0, "frac": 0.2, "ms": 0.04, "formula_TFLOP/s": 600.0},
                      "bwd": {"TFLOP/s": 300.0, "frac": 0.15, "ms": 0.1}}}
    r.update(bench.small_roofline_keys(small))
    for k, v in r.items():
        assert v is None or isinstance(v, (int, float, str)), (k, type(v))
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["peak"] == 1900.0
    want = K * (flops["fwd16"] + flops["fwd64"]) / ((part_ms["fwd16"] + part_ms["fwd64"]) * 1e-3) / 1e12
    assert abs(r["achieved"] - want) < 1e-9 * want and abs(r["frac"] - want / 1900.0) < 1e-12
    bwd = K * flops["bwd16"] / (part_ms["bwd16"] * 1e-3) / 1e12
    assert abs(r["bwd_achieved"] - bwd) < 1e-9 * bwd and abs(r["bwd_frac"] - bwd / 1900.0) < 1e-12
    dec = K * 4.4e9 / (part_ms["decode"] * 1e-3) / 1e9
    assert r["decode_bound"] == "hbm" and abs(r["decode_frac"] - dec / 6800.0) < 1e-12
    assert r["bert_fwd_formula_TFLOP/s"] == 600.0 and r["bert_bwd_frac"] == 0.15
