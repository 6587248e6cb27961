"""GPU parity of the paged + merge form of prefix-cached extend ("SGLang 源码完全拆解(八)：Attention
Backend", section «extend 的两种形态»): the new tokens' queries over their own contiguous K/V (ragged,
causal), over the cached prefix through the page table (every prefix key visible), and the merge of
the two states by their LSE -- each against the CPU oracle, and the composition against the oracle's
single causal pass over prefix + new tokens."""

import numpy as np
import pytest
import torch

import workloads as W
from oracle import attention as OA
from tests import gpu_common as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import paged_kv_attention_slot_gb300 as pk

    pk._lib.lib()
    assert pk.device_error() == 0
    yield
    assert pk.device_error() == 0


def _pk():
    import paged_kv_attention_slot_gb300 as pk

    return pk


def _bf16(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16)


def _ragged_inputs(kv_lens, q_lens, hq, hkv, seed, d=128):
    T, R = sum(q_lens), sum(kv_lens)
    q = _bf16((T, hq, d), seed)
    k = _bf16((R, hkv, d), seed + 1)
    v = _bf16((R, hkv, d), seed + 2)
    qo = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    kv = np.concatenate([[0], np.cumsum(kv_lens)]).astype(np.int32)
    return q, k, v, qo, kv


def _ragged_case(kv_lens, q_lens, hq, hkv, seed, causal=True, sm_scale=0.0):
    pk = _pk()
    q, k, v, qo, kv = _ragged_inputs(kv_lens, q_lens, hq, hkv, seed)
    p = pk.Plan().plan(qo, kv, None, None, num_qo_heads=hq, num_kv_heads=hkv, head_dim=128, mode="ragged",
                       causal=causal, sm_scale=sm_scale)
    out, lse = p.run_ragged(q.cuda(), k.cuda(), v.cuda(), return_lse=True)
    torch.cuda.synchronize()
    ro, rl = OA.ragged_attention(G.bf16_bits(q), G.bf16_bits(k), G.bf16_bits(v), qo, kv,
                                 sm_scale=sm_scale if sm_scale > 0 else None, causal=causal,
                                 q_format="bf16_bits", kv_format="bf16_bits")
    return out, lse, ro, rl


def _compare_with_empty(out, lse, ro, rl):
    """Rows whose oracle state is empty must be exactly (0, -inf); the others within tolerance."""
    o = out.float().cpu().numpy()
    l = lse.float().cpu().numpy()
    empty = np.isneginf(rl)
    assert np.all(o[empty] == 0.0) and np.all(np.isneginf(l[empty]))
    rows = np.where(~np.all(empty, axis=1))[0]
    if rows.size:
        return G.compare(out, lse, ro, rl, rows=rows)
    return {}


def test_ragged_causal_fresh_segments():
    # prefill without any cached prefix: every request's K/V is its own new tokens (n == L)
    lens = [64, 1, 200, 0, 513]
    _compare_with_empty(*_ragged_case(lens, lens, 32, 8, seed=31))


@pytest.mark.parametrize("hq, hkv", [(8, 8), (16, 2), (32, 8)])
def test_ragged_causal_gqa(hq, hkv):
    lens = [130, 7, 300]
    _compare_with_empty(*_ragged_case(lens, lens, hq, hkv, seed=hq * 3 + hkv))


def test_ragged_causal_kv_longer_than_queries():
    # bottom-right alignment when the contiguous K/V holds more rows than the request has queries
    _compare_with_empty(*_ragged_case([300, 129, 64], [70, 129, 1], 8, 2, seed=33))


def test_ragged_noncausal_with_short_and_empty_segments():
    _compare_with_empty(*_ragged_case([3, 0, 700, 128], [90, 40, 65, 1], 8, 2, seed=34, causal=False))


@pytest.mark.parametrize("ps", [1, 16])
def test_paged_noncausal_prefix_segments(ps):
    # the prefix pass of an extend: every query sees all L_i keys of the pool, L_i may be < n_i or 0
    pk = _pk()
    b = W.make_batch([40, 0, 900, 257], [40, 0, 900, 257], ps, 16, 4, 128, seed=35)  # pool values only
    q_lens = [100, 33, 64, 300]
    q = _bf16((sum(q_lens), 16, 128), 36)
    qo = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    cache = pk.KVCache(b.k_pool.cuda(), b.v_pool.cuda())
    p = pk.Plan().plan(qo, b.kv_indptr, b.kv_indices, b.last_page_len, num_qo_heads=16, num_kv_heads=4,
                       head_dim=128, page_size=ps, mode="prefill", causal=False)
    out, lse = p.run(q.cuda(), cache, return_lse=True)
    torch.cuda.synchronize()
    ro, rl = OA.paged_attention(G.bf16_bits(q), G.bf16_bits(b.k_pool), G.bf16_bits(b.v_pool), qo, b.kv_indptr,
                                b.kv_indices, b.last_page_len, ps, q_format="bf16_bits", kv_format="bf16_bits",
                                causal=False)
    _compare_with_empty(out, lse, ro, rl)


def _merge_inputs(n, d, seed):
    g = np.random.default_rng(seed)
    oa = _bf16((n, d), seed, 0.7)
    ob = _bf16((n, d), seed + 1, 0.7)
    la = torch.from_numpy(g.normal(size=n) * 4).float()
    lb = torch.from_numpy(g.normal(size=n) * 4).float()
    la[::7] = -float("inf")  # one side empty
    lb[::11] = -float("inf")  # both empty where both strides meet
    return oa, la, ob, lb


@pytest.mark.parametrize("d", [64, 128])
def test_merge_state_matches_oracle(d):
    pk = _pk()
    n = 10007  # several grid-stride rounds and a ragged tail
    oa, la, ob, lb = _merge_inputs(n, d, 40 + d)
    out, lse = pk.merge_state(oa.cuda(), la.cuda(), ob.cuda(), lb.cuda())
    torch.cuda.synchronize()
    ro, rl = OA.merge_states(OA.to_f64(G.bf16_bits(oa), "bf16_bits"), la.double().numpy(),
                             OA.to_f64(G.bf16_bits(ob), "bf16_bits"), lb.double().numpy())
    o = out.float().cpu().numpy()
    l = lse.cpu().numpy()
    both_empty = np.isneginf(rl)
    assert np.all(o[both_empty] == 0.0) and np.all(np.isneginf(l[both_empty]))
    ok = ~both_empty
    # one bf16 rounding of a convex combination of bf16 values: half an ulp of |o| <= 2^-8 |o|
    assert np.max(np.abs(o[ok] - ro[ok]) - np.abs(ro[ok]) * 2.0 ** -8) <= 1e-5
    assert np.max(np.abs(l[ok] - rl[ok])) <= 1e-5 * (1 + np.max(np.abs(rl[ok])))


def test_merge_state_in_place_twice():
    # o and lse alias the first state; a second call merges a third state into the result
    pk = _pk()
    n, d = 4099, 128
    oa, la, ob, lb = _merge_inputs(n, d, 50)
    oc, lc, _, _ = _merge_inputs(n, d, 60)
    a, sa = oa.cuda(), la.cuda()
    pk.merge_state(a, sa, ob.cuda(), lb.cuda(), out=a, lse_out=sa)
    pk.merge_state(a, sa, oc.cuda(), lc.cuda(), out=a, lse_out=sa)
    torch.cuda.synchronize()
    f = lambda t: OA.to_f64(G.bf16_bits(t), "bf16_bits")
    ro, rl = OA.merge_many([f(oa), f(ob), f(oc)], [la.double().numpy(), lb.double().numpy(), lc.double().numpy()])
    o = a.float().cpu().numpy()
    l = sa.cpu().numpy()
    ok = ~np.isneginf(rl)
    # two bf16 roundings: the first (<= 2^-8 of the intermediate, which is bounded by the inputs)
    # carries into the second merge with a weight <= 1, the second is <= 2^-8 of the result
    m3 = np.maximum(np.maximum(np.abs(f(oa)), np.abs(f(ob))), np.abs(f(oc)))
    assert np.max(np.abs(o[ok] - ro[ok]) - (np.abs(ro[ok]) + m3[ok]) * 2.0 ** -8) <= 1e-5
    assert np.max(np.abs(l[ok] - rl[ok])) <= 1e-5 * (1 + np.max(np.abs(rl[ok])))
    assert np.all(np.isneginf(l[~ok]))


def prefix_csr(b):
    """CSR page table of each request's cached prefix (its first L_i - n_i keys) in the same pool."""
    ps = b.page_size
    pre = (b.kv_len - b.q_len).astype(np.int64)
    npg = (pre + ps - 1) // ps
    indptr = np.concatenate([[0], np.cumsum(npg)]).astype(np.int32)
    indices = np.concatenate([b.kv_indices[b.kv_indptr[i]:b.kv_indptr[i] + npg[i]] for i in range(len(pre))] +
                             [np.zeros(0, np.int32)]).astype(np.int32)
    last = np.where(npg > 0, pre - (npg - 1) * ps, 0).astype(np.int32)
    return indptr, indices, last


def extend_by_merge(b, g):
    """The three calls on the device: ragged (new tokens, causal), paged prefix (causal=False), merge."""
    pk = _pk()
    kw = dict(num_qo_heads=b.num_qo_heads, num_kv_heads=b.num_kv_heads, head_dim=b.head_dim,
              sm_scale=b.sm_scale)
    rag = pk.Plan().plan(b.qo_indptr, b.qo_indptr, None, None, mode="ragged", **kw)
    pi, px, pl = prefix_csr(b)
    pre = pk.Plan().plan(b.qo_indptr, pi, px, pl, page_size=b.page_size, mode="prefill", causal=False, **kw)
    o1, s1 = rag.run_ragged(g.q, g.k_new, g.v_new, return_lse=True)
    o2, s2 = pre.run(g.q, g.cache, return_lse=True)
    out, lse = pk.merge_state(o1, s1, o2, s2, out=o1, lse_out=s1)
    torch.cuda.synchronize()
    return out, lse, (rag, pre)


@pytest.mark.parametrize("ps", [1, 16])
def test_extend_by_merge_equals_single_causal_pass(ps):
    b = W.make_batch([700, 129, 64, 1000, 90], [300, 129, 1, 37, 0], ps, 32, 8, 128, seed=70 + ps)
    g = G.GpuBatch(b)
    g.store()
    out, lse, _ = extend_by_merge(b, g)
    kp, vp, fmt = G.oracle_pools(b)
    ro, rl = G.oracle_attention(b, kp, vp, fmt)
    G.compare(out, lse, ro, rl)


def test_extend_by_merge_full_size_prefix_extend_sampled():
    # the prefix-cached extend workload (batch 8, new U[128, 2048], prefix U[0, 4096], page size 1)
    b = W.workload(3)
    g = G.GpuBatch(b)
    g.store()
    out, lse, (rag, pre) = extend_by_merge(b, g)
    rng = np.random.default_rng(3)
    rows = []
    for i in range(b.batch_size):
        q0, q1 = int(b.qo_indptr[i]), int(b.qo_indptr[i + 1])
        rows += [q0, q1 - 1] + rng.integers(q0, q1, size=3).tolist()
    rows = sorted(set(rows))
    kp, vp, fmt = G.oracle_pools(b)
    ro, rl = G.oracle_attention(b, kp, vp, fmt, rows=rows)
    G.compare(out, lse, ro, rl, rows=rows)
    assert rag.info()["num_work"] > 500 and pre.info()["num_work"] > 500


def test_split_noncausal_prefix_and_ragged_segments():
    # a long cached prefix attended by few queries (split), merged with the new tokens' ragged pass
    b = W.make_batch([9000, 40], [48, 40], 16, 32, 8, 128, seed=90)
    g = G.GpuBatch(b)
    g.store()
    out, lse, (rag, pre) = extend_by_merge(b, g)
    assert pre.info()["num_prefill_partials"] > 0
    kp, vp, fmt = G.oracle_pools(b)
    ro, rl = G.oracle_attention(b, kp, vp, fmt)
    G.compare(out, lse, ro, rl)


def test_split_ragged_long_kv():
    # contiguous K/V much longer than the queries: a split ragged pass
    out, lse, ro, rl = _ragged_case([12000, 64], [32, 64], 16, 4, seed=91)
    _compare_with_empty(out, lse, ro, rl)


def extend_by_fused_merge(b, g, **prefix_kw):
    """Two calls: ragged (new tokens, causal) into (o, lse), then the paged prefix pass merged into them."""
    pk = _pk()
    kw = dict(num_qo_heads=b.num_qo_heads, num_kv_heads=b.num_kv_heads, head_dim=b.head_dim,
              sm_scale=b.sm_scale)
    rag = pk.Plan().plan(b.qo_indptr, b.qo_indptr, None, None, mode="ragged", **kw)
    pi, px, pl = prefix_csr(b)
    pre = pk.Plan().plan(b.qo_indptr, pi, px, pl, page_size=b.page_size, mode="prefill", causal=False, **kw,
                         **prefix_kw)
    out, lse = rag.run_ragged(g.q, g.k_new, g.v_new, return_lse=True)
    pre.run(g.q, g.cache, out=out, lse=lse, merge_into=True)
    torch.cuda.synchronize()
    return out, lse, pre


@pytest.mark.parametrize("ps, split", [(1, False), (16, False), (16, True)])
def test_extend_by_fused_merge_equals_single_causal_pass(ps, split):
    # includes a request without a cached prefix (its rows keep the ragged state) and, with split,
    # a prefix pass cut into chunks whose merge kernel merges into the held state
    b = W.make_batch([700, 129, 64, 1000, 90], [300, 129, 1, 37, 0], ps, 32, 8, 128, seed=80 + ps)
    g = G.GpuBatch(b)
    g.store()
    out, lse, pre = extend_by_fused_merge(b, g, **({"num_sms": 4096} if split else {"max_splits": 1}))
    assert (pre.info()["num_prefill_partials"] > 0) == split
    kp, vp, fmt = G.oracle_pools(b)
    ro, rl = G.oracle_attention(b, kp, vp, fmt)
    G.compare(out, lse, ro, rl)


def test_extend_by_fused_merge_full_size_sampled():
    b = W.workload(3)
    g = G.GpuBatch(b)
    g.store()
    out, lse, _ = extend_by_fused_merge(b, g)
    rng = np.random.default_rng(4)
    rows = []
    for i in range(b.batch_size):
        q0, q1 = int(b.qo_indptr[i]), int(b.qo_indptr[i + 1])
        rows += [q0, q1 - 1] + rng.integers(q0, q1, size=3).tolist()
    rows = sorted(set(rows))
    kp, vp, fmt = G.oracle_pools(b)
    ro, rl = G.oracle_attention(b, kp, vp, fmt, rows=rows)
    G.compare(out, lse, ro, rl, rows=rows)


# ---- the same extend in ONE pass over two sources (PKV_MODE_PAGED_RAGGED) -------------------------
def paged_ragged(b, g, **extra):
    """One launch: each request's cached prefix through the prefix page table, its new tokens' K/V
    from the contiguous k_new / v_new rows, one online softmax over both."""
    pk = _pk()
    pi, px, pl = prefix_csr(b)
    p = pk.Plan().plan(b.qo_indptr, pi, px, pl, num_qo_heads=b.num_qo_heads, num_kv_heads=b.num_kv_heads,
                       head_dim=b.head_dim, page_size=b.page_size, mode="paged_ragged", sm_scale=b.sm_scale,
                       window_left=b.window_left, **extra)
    out, lse = p.run_paged_ragged(g.q, g.cache, g.k_new, g.v_new, return_lse=True)
    torch.cuda.synchronize()
    return out, lse, p


def _new_rows_differ_from_pool(b):
    """The pool's slots for the new tokens hold other values than k_new (so a kernel reading them from
    the pool instead of k_new would fail the comparison)."""
    P, ps, H, D = b.k_pool.shape
    k = b.k_pool.view(P * ps, H, D)[torch.from_numpy(b.slot_mapping)]
    return not torch.equal(k, b.k_new)


@pytest.mark.parametrize("ps", [1, 16, 64])
def test_paged_ragged_one_pass_reads_new_rows_from_the_contiguous_tensors(ps):
    # the pool is NOT written with this step's K/V first: the new keys can only come from k_new / v_new;
    # the result is the oracle's causal pass over prefix + new tokens (the oracle's pool is written)
    b = W.make_batch([700, 129, 64, 1000, 90, 33], [300, 129, 1, 37, 0, 33], ps, 32, 8, 128, seed=100 + ps)
    assert _new_rows_differ_from_pool(b)
    g = G.GpuBatch(b)
    out, lse, p = paged_ragged(b, g)
    kp, vp, fmt = G.oracle_pools(b)
    ro, rl = G.oracle_attention(b, kp, vp, fmt)
    G.compare(out, lse, ro, rl)


@pytest.mark.parametrize("hq, hkv, window", [(8, 8, -1), (16, 2, -1), (128, 1, -1), (32, 8, 0), (32, 8, 100)])
def test_paged_ragged_gqa_and_windows(hq, hkv, window):
    b = W.make_batch([500, 40, 1300], [200, 40, 129], 16, hq, hkv, 128, seed=110 + hq + window, window_left=window)
    g = G.GpuBatch(b)
    out, lse, p = paged_ragged(b, g)
    kp, vp, fmt = G.oracle_pools(b)
    ro, rl = G.oracle_attention(b, kp, vp, fmt)
    G.compare(out, lse, ro, rl)


def test_paged_ragged_noncausal_and_split():
    # causal=False: every new token sees the whole prefix and every new token of its request; and a
    # long prefix with few queries, split into key chunks (the chunks may straddle the two sources)
    pk = _pk()
    b = W.make_batch([300, 9000, 45], [60, 48, 45], 16, 32, 8, 128, seed=120)
    g = G.GpuBatch(b)
    kp, vp, fmt = G.oracle_pools(b)
    out, lse, p = paged_ragged(b, g, causal=False)
    ro, rl = OA.paged_attention(G.bf16_bits(b.q), kp, vp, b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len,
                                b.page_size, q_format="bf16_bits", kv_format=fmt, causal=False)
    G.compare(out, lse, ro, rl)
    out, lse, p = paged_ragged(b, g, num_sms=4096)
    assert p.info()["num_prefill_partials"] > 0
    ro, rl = G.oracle_attention(b, kp, vp, fmt)
    G.compare(out, lse, ro, rl)


def test_paged_ragged_full_size_prefix_extend():
    # the prefix-cached extend workload in the benchmark's launch: every row of the longest and the
    # shortest request, sampled rows of the others
    b = W.workload(3)
    g = G.GpuBatch(b)
    out, lse, p = paged_ragged(b, g)
    rng = np.random.default_rng(5)
    n = np.diff(b.qo_indptr)
    whole = {int(np.argmax(n)), int(np.argmin(n))}
    rows = []
    for i in range(b.batch_size):
        q0, q1 = int(b.qo_indptr[i]), int(b.qo_indptr[i + 1])
        rows += list(range(q0, q1)) if i in whole else [q0, q1 - 1] + rng.integers(q0, q1, size=3).tolist()
    rows = sorted(set(rows))
    kp, vp, fmt = G.oracle_pools(b)
    ro, rl = G.oracle_attention(b, kp, vp, fmt, rows=rows)
    G.compare(out, lse, ro, rl, rows=rows)
    assert p.info()["num_work"] > 1000
