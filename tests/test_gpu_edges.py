"""GPU edge cases of the runs: an empty batch (B = 0), a batch whose requests all have no new token,
and a zero-token KV write -- each a no-op that launches nothing and leaves the device error word
clear."""

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pk():
    import paged_kv_attention_slot_gb300 as pk

    pk._lib.lib()
    assert pk.device_error() == 0
    yield pk
    assert pk.device_error() == 0


@pytest.mark.parametrize("mode", ["decode", "prefill", "mixed"])
def test_empty_batch_runs_are_no_ops(pk, mode):
    b = W.make_batch([100], [1], 16, 8, 2, 128, seed=1)
    cache = pk.KVCache(b.k_pool.cuda(), b.v_pool.cuda())
    p = pk.Plan().plan([0], [0], [], [], num_qo_heads=8, num_kv_heads=2, head_dim=128, page_size=16, mode=mode)
    assert p.info()["num_work"] == 0 and p.info()["total_tokens"] == 0
    q = torch.empty((0, 8, 128), dtype=torch.bfloat16, device="cuda")
    out, lse = p.run(q, cache, return_lse=True)
    torch.cuda.synchronize()
    assert out.shape == (0, 8, 128) and lse.shape == (0, 8)


def test_empty_ragged_batch_and_idle_requests(pk):
    q = torch.empty((0, 8, 128), dtype=torch.bfloat16, device="cuda")
    k = torch.empty((0, 2, 128), dtype=torch.bfloat16, device="cuda")
    p = pk.Plan().plan([0], [0], None, None, num_qo_heads=8, num_kv_heads=2, head_dim=128, mode="ragged")
    p.run_ragged(q, k, k)
    # requests with keys but no new token: nothing to compute, no row of output
    b = W.make_batch([100, 300], [0, 0], 16, 8, 2, 128, seed=2)
    cache = pk.KVCache(b.k_pool.cuda(), b.v_pool.cuda())
    p2 = pk.Plan().plan(b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, num_qo_heads=8, num_kv_heads=2,
                        head_dim=128, page_size=16, mode="prefill")
    assert p2.info()["num_work"] == 0
    p2.run(q, cache)
    torch.cuda.synchronize()


def test_zero_token_kv_store(pk):
    b = W.make_batch([100], [1], 16, 8, 2, 128, seed=3)
    pool = b.k_pool.cuda()
    before = pool.clone()
    cache = pk.KVCache(pool, b.v_pool.cuda())
    e = torch.empty((0, 2, 128), dtype=torch.bfloat16, device="cuda")
    pk.kv_store(e, e, torch.empty(0, dtype=torch.int64, device="cuda"), cache)
    torch.cuda.synchronize()
    assert torch.equal(pool, before)
