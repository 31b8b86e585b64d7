"""CPU tests of the benchmark's bookkeeping: the algorithmic work per launch (flops and bytes
counted as the hot path defines them) and the traffic records."""
import hashlib
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from mlstm_matrix_memory_02_b300 import workloads as W  # noqa: E402


def test_forward_flops_by_hand():
    # per head and chunk: causal Q K^T and (S o D) V over the lower triangle including the
    # diagonal, L (L + 1) (dqk + dv); Q C^T and the state update, 2 * 2 L dqk dv
    L, d, heads, chunks = 64, 512, 16, 2048 // 64
    per_chunk = 2 * (L * (L + 1) // 2) * (d + d) + 2 * (2 * L * d * d)
    assert bench.fwd_flops(W.LAYER_1P3B) == per_chunk * chunks * heads
    assert abs(bench.fwd_flops(W.LAYER_1P3B) / 1e9 - 36.54) < 0.01
    assert abs(bench.fwd_flops(W.LAYER_350M) / 1e9 - 9.68) < 0.01


def test_forward_bytes_by_hand():
    # q, k, v in bf16, two fp32 gates per token, h once, the final (C, n, m) once
    w = W.LAYER_1P3B
    tokens = w.B * w.NH * w.S
    expect = tokens * (512 + 512 + 512) * 2 + tokens * 8 + tokens * 512 * 2 + 16 * (512 * 512 + 512 + 1) * 4
    assert bench.fwd_bytes(w, h_bytes=2) == expect
    assert abs(bench.fwd_bytes(w, h_bytes=2) / 1e6 - 151.3) < 0.1
    assert bench.fwd_bytes(w, h_bytes=4) - bench.fwd_bytes(w, h_bytes=2) == tokens * 512 * 2


def test_decode_bytes_by_hand():
    # per head: C and n read and written (fp32), m read and written, bf16 q k v, fp32 gates, h
    w = W.DECODE
    per_head = 2 * 256 * 256 * 4 + 2 * 256 * 4 + 2 * 4 + 3 * 256 * 2 + 2 * 4 + 256 * 4
    assert bench.dec_bytes(w) == 256 * 8 * per_head
    assert abs(bench.dec_bytes(w) / 1e9 - 1.083) < 0.001


def test_traffic_records_name_existing_sources():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        records = json.load(f)
    for kernel, rec in records.items():
        sources = rec.get("sources", [rec.get("source")])
        h = hashlib.sha256()
        for src in sources:
            path = os.path.join(ROOT, src)
            assert os.path.exists(path), (kernel, src)
            h.update(open(path, "rb").read())
        assert os.path.exists(os.path.join(ROOT, rec["profile"])), kernel
        got = bench.captured_traffic(kernel)
        # a record counts only while every source it lists is the one that was captured
        assert got == (float(rec["dram_bytes"]) if h.hexdigest()[:16] == rec["sha"] else None)
    assert bench.captured_traffic("no_such_kernel") is None


@pytest.mark.parametrize("name", ["1p3b", "350m", "stress"])
def test_bench_workloads_exist(name):
    w = W.WORKLOADS[name]
    assert w.S % w.chunk == 0 and w.DQK % 32 == 0 and w.DV % 32 == 0
