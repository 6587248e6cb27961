"""GPU parity of the KV write and paged decode (with split-KV merge) against the CPU oracle.

Small cases compare every output element; the full-size workloads (the launch configuration the
benchmark times) compare sampled requests the oracle computes one by one.  KV writes are bit-exact.
"""

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


# ---------------------------------------------------------------------------------------------
# KV write
# ---------------------------------------------------------------------------------------------
def test_kv_store_bf16_bit_exact_tiny_workload():
    b = W.workload(1)
    g = G.GpuBatch(b)
    g.store()
    torch.cuda.synchronize()
    kp, vp, _ = G.oracle_pools(b)
    assert np.array_equal(G.bf16_bits(g.k_pool), kp)
    assert np.array_equal(G.bf16_bits(g.v_pool), vp)


@pytest.mark.parametrize("D", [64, 128])
def test_kv_store_bf16_padding_and_strided_pool(D):
    import paged_kv_attention_slot_gb300 as pk

    torch.manual_seed(0)
    P, ps, H = 9, 4, 3
    # a pool whose pages are strided (one spare page-sized gap between pages)
    big_k = torch.zeros((P, 2, ps, H, D), dtype=torch.bfloat16, device="cuda")
    big_v = torch.zeros_like(big_k)
    kp, vp = big_k[:, 0], big_v[:, 0]
    cache = pk.KVCache(kp, vp)
    T = 11
    k = torch.randn((T, H, D), device="cuda").bfloat16()
    v = torch.randn((T, H, D), device="cuda").bfloat16()
    slots = torch.tensor([0, 5, -1, 35, 17, -7, 2, 8, 30, 12, 1], dtype=torch.int64, device="cuda")
    pk.kv_store(k, v, slots, cache)
    torch.cuda.synchronize()
    ref_k = np.zeros((P, ps, H, D), dtype=np.uint16)
    ref_v = np.zeros_like(ref_k)
    from oracle import attention as OA

    OA.kv_store(ref_k, ref_v, G.bf16_bits(k), G.bf16_bits(v), slots.cpu().numpy(), ps)
    assert np.array_equal(G.bf16_bits(kp), ref_k)
    assert np.array_equal(G.bf16_bits(vp), ref_v)
    assert torch.count_nonzero(big_k[:, 1]) == 0  # the gaps were never written


def test_kv_store_out_of_range_slot_is_reported_not_written():
    import paged_kv_attention_slot_gb300 as pk

    P, ps, H, D = 4, 2, 1, 64
    kp = torch.zeros((P, ps, H, D), dtype=torch.bfloat16, device="cuda")
    vp = torch.zeros_like(kp)
    cache = pk.KVCache(kp, vp)
    k = torch.ones((2, H, D), device="cuda").bfloat16()
    slots = torch.tensor([3, P * ps], dtype=torch.int64, device="cuda")  # the second is one past the end
    pk.kv_store(k, k, slots, cache)
    assert pk.device_error(reset=True) == 1
    assert float(kp[1, 1].float().sum()) == D  # slot 3 written
    assert float(kp.float().sum()) == D


def test_kv_store_fp8_bit_exact_including_saturation():
    import paged_kv_attention_slot_gb300 as pk

    g = torch.Generator().manual_seed(5)
    P, ps, H, D = 16, 8, 2, 128
    T = P * ps
    k = (torch.randn((T, H, D), generator=g) * torch.logspace(-6, 3, T).view(T, 1, 1)).bfloat16()
    v = (torch.randn((T, H, D), generator=g) * 3).bfloat16()
    for ks, vs in ((0.5, 0.01), (1.0 / 448.0, 2.0), (3.7e-3, 1.1)):
        kp = torch.zeros((P, ps, H, D), dtype=torch.uint8, device="cuda")
        vp = torch.zeros_like(kp)
        cache = pk.KVCache(kp, vp, ks, vs)
        perm = torch.randperm(T, generator=g)
        pk.kv_store(k.cuda(), v.cuda(), perm.cuda(), cache)
        torch.cuda.synchronize()
        from oracle import attention as OA

        rk = np.zeros((P, ps, H, D), dtype=np.uint8)
        rv = np.zeros_like(rk)
        OA.kv_store_fp8(rk, rv, k.float().numpy(), v.float().numpy(), perm.numpy(), ps, ks, vs)
        assert np.array_equal(kp.cpu().numpy(), rk)
        assert np.array_equal(vp.cpu().numpy(), rv)
        assert (kp.cpu().numpy() & 0x7F).max() == 0x7E  # saturation reached and handled


# ---------------------------------------------------------------------------------------------
# decode, every element
# ---------------------------------------------------------------------------------------------
def _decode_case(b, **plan_kw):
    g = G.GpuBatch(b)
    g.store()
    plan = g.plan(**plan_kw)
    out, lse = g.run(plan)
    kp, vp, fmt = G.oracle_pools(b)
    ro, rl = G.oracle_attention(b, kp, vp, fmt)
    tol = G.FP8_MAX_ABS if b.kv_dtype == "e4m3" else G.BF16_MAX_ABS
    return G.compare(out, lse, ro, rl, max_abs=tol), plan


def test_decode_fp8_query_beyond_the_f16_range():
    # FP8 KV runs the decode products in f16, whose largest finite value is 65504; query rows with
    # |q| up to ~1.2e5 are scaled into range by a power of two inside the kernel (exact for bf16
    # values), so the output stays within the FP8 tolerance of the oracle instead of turning NaN.
    # The heads that share a CTA with a large one (same KV head) are checked too.
    b = W.make_batch([700, 20, 5000, 129, 3000], [1] * 5, 16, 32, 8, 128, seed=91, kv_dtype="e4m3")
    q = b.q.float()
    q[0, 0:4] *= 3e4                 # one whole KV-head group of request 0: |q| up to ~1.2e5
    q[2, 5, 17] = 1.0e5              # a single element of request 2 (its KV head's other heads stay N(0,1))
    q[2, 6, 100] = -7.0e4
    q[3, :] *= 2e4                   # every head of request 3: |q| up to ~8e4
    b.q = q.bfloat16()
    assert float(b.q.float().abs().max()) > 65504
    g = G.GpuBatch(b)
    g.store()
    out, lse = g.run(g.plan())
    kp, vp, fmt = G.oracle_pools(b)
    ro, rl = G.oracle_attention(b, kp, vp, fmt)
    # an fp32 score of magnitude ~1e5 carries ~1e-2 of rounding: the LSE bound grows with |lse|
    G.compare(out, lse, ro, rl, max_abs=G.FP8_MAX_ABS, lse_rel=1e-6)
    # the same batch with the split-KV merge forced
    out, lse = g.run(g.plan(num_sms=4096))
    G.compare(out, lse, ro, rl, max_abs=G.FP8_MAX_ABS, lse_rel=1e-6)


@pytest.mark.parametrize("kv, num_sms", [("bf16", 16), ("bf16", 64), ("bf16", 600), ("e4m3", 600)])
def test_decode_split_merges_up_to_hundreds_of_partials(kv, num_sms):
    # a 100,000-key request split over 16, ~60 or ~390 CTAs (the last CTA of the unit merges them all,
    # in chunks that fit its shared memory), shorter requests with fewer or no splits; every element
    # against the oracle
    ps = 16 if kv == "bf16" else 128
    b = W.make_batch([100000, 3000, 200, 17], [1, 1, 1, 1], ps, 8, 2, 128, seed=130, kv_dtype=kv)
    stats, plan = _decode_case(b, num_sms=num_sms)
    splits = np.bincount(plan.work_items()[:, 0] * 2 + plan.work_items()[:, 1])
    assert splits.max() > 12 and plan.info()["num_merge"] > 0
    # and a second run of the same plan (the group and unit counters were returned to zero)
    g = G.GpuBatch(b)
    g.store()
    out, lse = g.run(plan)
    kp, vp, fmt = G.oracle_pools(b)
    ro, rl = G.oracle_attention(b, kp, vp, fmt)
    G.compare(out, lse, ro, rl, max_abs=G.FP8_MAX_ABS if kv == "e4m3" else G.BF16_MAX_ABS)


def test_decode_tiny_workload_all_elements():
    stats, plan = _decode_case(W.workload(1))
    assert plan.info()["num_merge"] == 0


@pytest.mark.parametrize("ps", [1, 3, 16, 64])
@pytest.mark.parametrize("D", [64, 128])
def test_decode_page_sizes_and_head_dims(ps, D):
    lens = [1, 2, 15, 16, 17, 100, 333, 1029]
    b = W.make_batch(lens, [1] * len(lens), ps, 8, 2, D, seed=100 + ps + D)
    _decode_case(b)


@pytest.mark.parametrize("hq, hkv", [(4, 4), (8, 1), (16, 2), (32, 1), (40, 2), (64, 8), (128, 1)])
def test_decode_gqa_groups(hq, hkv):
    lens = [5, 64, 250, 777]
    b = W.make_batch(lens, [1] * len(lens), 16, hq, hkv, 128, seed=hq * 7 + hkv)
    _decode_case(b)


@pytest.mark.parametrize("max_splits", [0, 1, 2, 7])
def test_decode_split_kv_merge(max_splits):
    lens = [3000, 9000, 64, 4500, 12000, 1]
    b = W.make_batch(lens, [1] * len(lens), 16, 32, 8, 128, seed=77)
    stats, plan = _decode_case(b, max_splits=max_splits, num_sms=64)  # small chunks -> many splits
    info = plan.info()
    if max_splits == 1:
        assert info["num_merge"] == 0
    else:
        assert info["num_merge"] > 0


@pytest.mark.parametrize("window", [0, 1, 100, 4096])
def test_decode_sliding_window(window):
    lens = [1, 50, 4097, 6000, 9000]
    b = W.make_batch(lens, [1] * len(lens), 32, 16, 4, 128, seed=window + 3, window_left=window)
    _decode_case(b, num_sms=64)


def test_decode_idle_requests_and_custom_scale():
    # requests with no new token (n_i = 0) produce no row; a custom softmax scale is honoured
    b = W.make_batch([40, 300, 7, 90], [1, 0, 1, 0], 16, 8, 2, 128, seed=9, sm_scale=0.3, mode="decode")
    _decode_case(b)


def test_decode_fp8_small_with_window():
    for w in (-1, 700):
        b = W.make_batch([5000, 131, 2048, 1], [1] * 4, 128, 32, 8, 128, seed=55, kv_dtype="e4m3", window_left=w)
        _decode_case(b, num_sms=64)


def test_decode_plan_reuse_across_layers_and_replan():
    """One plan serves several layers (different pools); re-planning the same object works."""
    import paged_kv_attention_slot_gb300 as pk

    b1 = W.make_batch([70, 300, 20], [1, 1, 1], 16, 8, 2, 128, seed=1)
    g1 = G.GpuBatch(b1)
    g1.store()
    plan = g1.plan()
    out_a, lse_a = g1.run(plan)
    # a second "layer": same batch (page table, slots), different pool contents and queries
    import dataclasses

    other = W.make_batch([70, 300, 20], [1, 1, 1], 16, 8, 2, 128, seed=2, num_pages=b1.num_pages)
    b2 = dataclasses.replace(b1, q=other.q, k_new=other.k_new, v_new=other.v_new, k_pool=other.k_pool,
                             v_pool=other.v_pool)
    g2 = G.GpuBatch(b2)
    g2.store()
    out_b, lse_b = plan.run(g2.q, g2.cache, return_lse=True)
    torch.cuda.synchronize()
    for b, (o, l) in ((b1, (out_a, lse_a)), (b2, (out_b, lse_b))):
        kp, vp, fmt = G.oracle_pools(b)
        ro, rl = G.oracle_attention(b, kp, vp, fmt)
        G.compare(o, l, ro, rl)
    # re-plan the same object for a different batch
    b3 = W.make_batch([5, 900], [1, 1], 16, 8, 2, 128, seed=3)
    g3 = G.GpuBatch(b3)
    g3.store()
    plan.plan(b3.qo_indptr, b3.kv_indptr, b3.kv_indices, b3.last_page_len, num_qo_heads=8, num_kv_heads=2,
              head_dim=128, page_size=16, mode="decode")
    o3, l3 = plan.run(g3.q, g3.cache, return_lse=True)
    kp, vp, fmt = G.oracle_pools(b3)
    ro, rl = G.oracle_attention(b3, kp, vp, fmt)
    G.compare(o3, l3, ro, rl)
    # the run checks the cache against the plan
    small = pk.KVCache(g3.k_pool[:1], g3.v_pool[:1])
    with pytest.raises(pk.PkvError):
        plan.run(g3.q, small)


# ---------------------------------------------------------------------------------------------
# full-size workloads: the benchmark's launch configuration, sampled requests
# ---------------------------------------------------------------------------------------------
def _sampled(b, n_req, seed):
    rng = np.random.default_rng(seed)
    req = rng.choice(b.batch_size, size=min(n_req, b.batch_size), replace=False)
    # include the longest request
    req = np.unique(np.concatenate([req, [int(np.argmax(b.kv_len))]]))
    return b.qo_indptr[req]


@pytest.mark.parametrize("n", [2, 4])
def test_decode_full_size_workload_sampled(n):
    b = W.workload(n)
    g = G.GpuBatch(b)
    g.store()
    plan = g.plan()
    out, lse = g.run(plan)
    rows = _sampled(b, 12, n)
    kp, vp, fmt = G.oracle_pools(b)
    ro, rl = G.oracle_attention(b, kp, vp, fmt, rows=rows)
    G.compare(out, lse, ro, rl, rows=rows)
    o = out.float()
    assert torch.isfinite(o).all()


def test_decode_full_size_fp8_long_context_and_window():
    b = W.workload(5)
    g = G.GpuBatch(b)
    g.store()
    torch.cuda.synchronize()
    kp, vp, fmt = G.oracle_pools(b)
    # the whole FP8 pool (history quantised on write + this step's tokens) is bit-exact
    assert np.array_equal(g.k_pool.cpu().numpy(), kp)
    assert np.array_equal(g.v_pool.cpu().numpy(), vp)
    for w in (-1, 4096):
        b.window_left = w
        plan = g.plan()
        out, lse = g.run(plan)
        ro, rl = G.oracle_attention(b, kp, vp, fmt)
        G.compare(out, lse, ro, rl, max_abs=G.FP8_MAX_ABS)
