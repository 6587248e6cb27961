"""The seeded generator lays out valid batches: its CSR arrays and write slots agree with the oracle's
restatement of the pages' metadata rules, and every request's pages are distinct."""

import numpy as np

import workloads as W
from oracle import metadata as M


def _check(b):
    indptr, indices, last = M.csr_from_block_table(b.block_rows, b.kv_len, b.page_size)
    assert np.array_equal(indptr, b.kv_indptr)
    assert np.array_equal(indices, b.kv_indices)
    assert np.array_equal(last, b.last_page_len)
    sm = M.slot_mapping(b.block_rows, b.qo_indptr, b.kv_len, b.page_size)
    assert np.array_equal(sm, b.slot_mapping)
    assert len(set(b.kv_indices.tolist())) == len(b.kv_indices)
    assert b.kv_indices.max(initial=-1) < b.num_pages


def test_tiny_workload_recipe():
    b = W.workload(1)
    assert b.kv_len.tolist() == [7, 16, 33, 64]
    assert b.num_pages == 32 and b.page_size == 16 and b.head_dim == 64
    assert b.kv_indptr.tolist() == [0, 1, 2, 5, 9]
    assert b.last_page_len.tolist() == [7, 16, 1, 16]
    assert b.qo_indptr.tolist() == [0, 1, 2, 3, 4]
    _check(b)


def test_generator_is_seeded_and_consistent():
    a = W.make_batch([5, 40, 17], [1, 3, 17], 8, 4, 2, 16, seed=3)
    b = W.make_batch([5, 40, 17], [1, 3, 17], 8, 4, 2, 16, seed=3)
    assert np.array_equal(a.kv_indices, b.kv_indices)
    assert (a.q.view(-1).float() == b.q.view(-1).float()).all()
    _check(a)


def test_scaled_down_named_workloads():
    for n in (2, 3, 4):
        b = W.workload(n, scale_batch=0.05)
        _check(b)
    b3 = W.workload(3, scale_batch=0.25)
    assert b3.page_size == 1 and np.all(b3.last_page_len == 1)
    assert np.all(b3.q_len >= 128) and np.all(b3.kv_len - b3.q_len <= 4096)


def test_fp8_scale_is_amax_over_448():
    b = W.make_batch([300, 129], [1, 1], 128, 4, 2, 32, seed=5, kv_dtype="e4m3")
    amax = max(float(b.k_pool.float().abs().max()), float(b.k_new.float().abs().max()))
    assert b.k_scale == float(np.float32(amax) / np.float32(448.0))
