"""GPU parity of causal prefill / prefix-cached extend (tcgen05 kernel) against the CPU oracle."""

import numpy as np
import pytest
import torch

import workloads as W
from tests import gpu_common as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import paged_kv_attention_slot_gb300 as pk

    pk._lib.lib()
    assert pk.device_error() == 0
    yield
    assert pk.device_error() == 0


def _case(b, rows=None, **plan_kw):
    g = G.GpuBatch(b)
    g.store()
    plan = g.plan(**plan_kw)
    out, lse = g.run(plan)
    kp, vp, fmt = G.oracle_pools(b)
    ro, rl = G.oracle_attention(b, kp, vp, fmt, rows=rows)
    return G.compare(out, lse, ro, rl, rows=rows), plan


def test_prefill_single_tile_no_prefix():
    # one request, 32 new tokens, no cached prefix, G = 4: exactly one 128-row tile and one K tile
    b = W.make_batch([32], [32], 1, 8, 2, 128, seed=1)
    _case(b)


def test_prefill_multi_tile_with_prefix():
    b = W.make_batch([300], [70], 1, 8, 2, 128, seed=2)
    _case(b)


@pytest.mark.parametrize("hq, hkv", [(4, 4), (8, 4), (8, 2), (16, 2), (32, 2), (64, 1), (128, 1)])
def test_prefill_gqa_groups(hq, hkv):  # up to MQA with 128 query heads: one token per 128-row tile
    b = W.make_batch([129, 50, 400], [129, 17, 260], 1, hq, hkv, 128, seed=hq + hkv)
    _case(b)


@pytest.mark.parametrize("ps", [1, 4, 16, 64])
def test_prefill_page_sizes(ps):
    b = W.make_batch([1, 40, 257, 700], [1, 33, 200, 129], ps, 8, 2, 128, seed=10 + ps)
    _case(b)


def test_prefill_ragged_with_idle_requests():
    b = W.make_batch([90, 0, 13, 1000, 5], [0, 0, 13, 3, 5], 1, 16, 4, 128, seed=5)
    _case(b)


@pytest.mark.parametrize("window", [0, 7, 128, 300])
def test_prefill_sliding_window(window):
    b = W.make_batch([600, 140, 33], [200, 140, 1], 1, 8, 2, 128, seed=20 + window, window_left=window)
    _case(b)


def test_prefill_custom_scale_large_scores():
    # a large softmax scale stresses the lazy rescaling of the running maximum
    b = W.make_batch([512, 700], [256, 700], 1, 8, 2, 128, seed=7, sm_scale=1.5)
    _case(b)


def test_prefill_full_size_prefix_extend_sampled():
    # the benchmark's launch (all 1448 CTAs of the prefix-extend workload): every token row and head
    # of its longest and its shortest request, plus sampled rows of every other request
    b = W.workload(3)
    rng = np.random.default_rng(3)
    rows = []
    n = np.diff(b.qo_indptr)
    whole = {int(np.argmax(n)), int(np.argmin(n))}
    for i in range(b.batch_size):
        q0, q1 = int(b.qo_indptr[i]), int(b.qo_indptr[i + 1])
        if i in whole:
            rows += list(range(q0, q1))
        else:
            rows += [q0, q1 - 1] + rng.integers(q0, q1, size=3).tolist()
    stats, plan = _case(b, rows=sorted(set(rows)))
    assert plan.info()["num_work"] > 1000
    assert len(rows) > int(n.max()) + int(n.min())


# ---- split-KV prefill: few query items over long key ranges --------------------------------------
def test_prefill_split_long_prefix_few_tokens():
    # one request, 64 new tokens after a 20k-token prefix: 8 items on 152 SMs, so the planner cuts
    # each key range into chunks and a merge kernel combines them
    b = W.make_batch([20000], [64], 16, 32, 8, 128, seed=80)
    stats, plan = _case(b)
    info = plan.info()
    assert info["num_prefill_partials"] > 8 and info["num_merge"] == 8


@pytest.mark.parametrize("window", [-1, 700])
def test_prefill_split_forced_on_many_items(window):
    # a large planning SM count forces splits on a batch with ragged tiles, GQA 4 and page size 1
    b = W.make_batch([3000, 200, 2500], [300, 200, 1], 1, 16, 4, 128, seed=81, window_left=window)
    stats, plan = _case(b, num_sms=4096)
    assert plan.info()["num_prefill_partials"] > 0


def test_prefill_split_respects_max_splits():
    b = W.make_batch([5000, 1500], [100, 64], 16, 8, 2, 128, seed=82)
    stats, plan = _case(b, num_sms=4096, max_splits=3)
    items = plan.work_items()
    assert items[:, 6].max() >= 0 and plan.info()["num_prefill_partials"] <= 3 * plan.info()["num_merge"]


def test_prefill_long_request_sampled():
    # maximum-size case: one request, 8192 new tokens after a 32768-token prefix (up to 320 key tiles
    # per CTA), checked on sampled rows including the first and the last
    b = W.make_batch([32768 + 8192], [8192], 16, 32, 8, 128, seed=83)
    rows = sorted(set([0, 1, 63, 64, 4095, 8191] + np.random.default_rng(83).integers(0, 8192, size=6).tolist()))
    stats, plan = _case(b, rows=rows)
    assert plan.info()["num_work"] == 8192 // 64 * 8
