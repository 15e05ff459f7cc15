"""Host-side arithmetic of bench.py that the reported figures rest on: the
algorithmic bytes and flops of a layer call and of the accept step."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_layer_bytes_flops_draft():
    M, K, N = 64, 4096, 14336
    b, f = bench.layer_bytes_flops(M, K, N, [16, 16], verify=False)
    assert b == 2 * (N * K + M * K + M * N)   # W, x and y once, bf16
    assert f == 2 * M * N * K


def test_layer_bytes_flops_verify_adds_adapters_per_slice():
    M, K, N = 128, 4096, 6144
    ranks = [16, 8, 32]
    b1, _ = bench.layer_bytes_flops(M, K, N, ranks, verify=True, n_proj=1)
    b3, _ = bench.layer_bytes_flops(M, K, N, ranks, verify=True, n_proj=3)
    base = 2 * (N * K + M * K + M * N)
    assert b1 == base + sum(2 * r * K + 2 * N * r for r in ranks)
    assert b3 - b1 == sum(2 * r * K * 2 for r in ranks)  # one A stack per slice, B once


def test_accept_bytes():
    V, B, k = 128256, 4, 2
    accepted = [2, 0, 1, 2]  # requests 1 and 2 rejected: they read p_n and q_n
    assert bench.accept_bytes(B, V, accepted, k) == 4 * V * (1 + 2 + 2 + 1) + 8 * B * k


def test_job_throughput_units():
    # 128 verified tokens per step at 0.25 ms per step is 512 K tokens/s per rank
    assert bench.job_throughput(128, 1, 0.25) == pytest.approx(512000.0)
    assert bench.job_throughput(128, 4, 0.25) == pytest.approx(4 * 512000.0)
