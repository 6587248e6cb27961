"""The algorithmic work the benchmark divides by, counted independently of its closed forms.

Prefill TFLOP/s uses the number of causally visible (query, key) pairs; decode GB/s uses the K/V
bytes of every visible key.  Both closed forms are checked here against a direct count through the
oracle's own visibility rule (query position and visible range per token), on seeded batches."""

import numpy as np
import pytest

import bench
import workloads as W
from oracle import attention as A


def _pairs_by_count(kv_len, q_len, window=-1):
    total = 0
    for L, n in zip(kv_len.tolist(), q_len.tolist()):
        for t in range(n):
            lo, hi = A.visible_range(A.query_position(L, n, t), window)
            total += max(0, hi - lo + 1)
    return total


@pytest.mark.parametrize("seed", range(5))
def test_visible_pairs_closed_form_matches_a_direct_count(seed):
    rng = np.random.default_rng(seed)
    n = rng.integers(0, 60, 12)
    L = n + rng.integers(0, 90, 12)
    assert bench._visible_pairs(L, n) == _pairs_by_count(L, n)


def test_prefill_workload_flops_match_a_direct_count():
    b = W.workload(3)
    pairs = _pairs_by_count(b.kv_len, b.q_len)
    assert bench._visible_pairs(b.kv_len, b.q_len) == pairs
    # 4 D flops per pair and query head (QK^T and PV, a multiply and an add each)
    assert 4.0 * b.head_dim * b.num_qo_heads * pairs == pytest.approx(471745363968.0, rel=0, abs=0.5)


@pytest.mark.parametrize("dtype, window", [("bf16", -1), ("bf16", 100), ("e4m3", -1), ("e4m3", 4096)])
def test_decode_kv_bytes_match_a_direct_count(dtype, window):
    # the byte formula needs only the lengths: a stand-in batch with seeded lengths (no pools)
    from types import SimpleNamespace

    rng = np.random.default_rng(21)
    kv_len = rng.integers(1, 9000, 40)
    b = SimpleNamespace(kv_len=kv_len, window_left=window, kv_dtype=dtype, num_kv_heads=8, head_dim=128)
    keys = _pairs_by_count(kv_len, np.ones_like(kv_len), window)  # one query per request
    elem = 1 if dtype == "e4m3" else 2
    assert W.Batch.kv_bytes_read(b) == keys * 8 * 128 * elem * 2
