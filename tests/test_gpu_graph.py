"""CUDA-graph capture and replay of the runs, and a re-plan in place under a captured graph.

"vLLM Attention 后端与 FlashInfer 元数据", section «CUDA Graph 约束的是控制路径，不只是 Tensor 形状»: replay needs
stable device addresses and an unchanged launch sequence, so a backend must not allocate, re-size
its workspace or change its launches per batch; dynamic content goes into stable buffers.  Here the
runs allocate nothing and launch a fixed number of kernels, so `plan.run` is captured once; a new
batch with the same lengths (new page table, new values) is planned in place into the same
workspace and the same graph replays it."""

import dataclasses

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


def _capture(fn):
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(2):
            fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fn()
    return graph


def _load_batch_into(g, b):
    """Overwrite g's device tensors (same shapes) with batch b's pools, queries and new tokens."""
    g.k_pool.copy_(b.k_pool.to(g.k_pool.device))
    g.v_pool.copy_(b.v_pool.to(g.v_pool.device))
    g.q.copy_(b.q.to(g.q.device))
    g.k_new.copy_(b.k_new.to(g.q.device))
    g.v_new.copy_(b.v_new.to(g.q.device))
    g.slots.copy_(torch.from_numpy(b.slot_mapping).to(g.q.device))
    g.b = b


def _plan_args(b):
    return dict(num_qo_heads=b.num_qo_heads, num_kv_heads=b.num_kv_heads, head_dim=b.head_dim,
                page_size=b.page_size, mode=b.mode, window_left=b.window_left, sm_scale=b.sm_scale,
                kv_dtype=b.kv_dtype)


@pytest.mark.parametrize("kind", ["decode_split", "extend", "mixed"])
def test_graph_replay_and_replan_in_place(kind):
    rng = np.random.default_rng(5)
    if kind == "decode_split":
        L = rng.integers(1, 6000, 12).tolist()
        n = [1] * 12
        mode, extra = "decode", dict(num_sms=24)
    elif kind == "extend":
        n = rng.integers(1, 400, 5).tolist()
        L = [q + int(rng.integers(0, 900)) for q in n]
        mode, extra = "extend", {}
    else:
        n = [1, 37, 1, 1, 200, 1]
        L = [2500, 90, 17, 4100, 650, 1]
        mode, extra = "mixed", dict(num_sms=24)
    b1 = W.make_batch(L, n, 16, 32, 8, 128, seed=51, mode=mode)
    b2 = W.make_batch(L, n, 16, 32, 8, 128, seed=52, mode=mode)  # same lengths: new pages and values
    assert b1.num_pages == b2.num_pages

    g = G.GpuBatch(b1)
    g.store()
    plan = g.plan(**extra)
    out = torch.empty_like(g.q)
    lse = torch.empty(g.q.shape[:2], dtype=torch.float32, device=g.q.device)
    graph = _capture(lambda: plan.run(g.q, g.cache, out=out, lse=lse))

    # replay on batch 1
    out.fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    kp, vp, fmt = G.oracle_pools(b1)
    ro, rl = G.oracle_attention(b1, kp, vp, fmt)
    G.compare(out, lse, ro, rl)

    # batch 2: new data in the same buffers, re-planned in place (same workspace), same graph
    ws = plan.workspace.data_ptr()
    _load_batch_into(g, b2)
    g.store()
    plan.plan(b2.qo_indptr, b2.kv_indptr, b2.kv_indices, b2.last_page_len, **_plan_args(b2), **extra)
    assert plan.workspace.data_ptr() == ws
    out.fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    kp, vp, fmt = G.oracle_pools(b2)
    ro, rl = G.oracle_attention(b2, kp, vp, fmt)
    G.compare(out, lse, ro, rl)

    # and replaying again (the kernels leave the split counters at zero) gives the same answer
    first = out.clone()
    graph.replay()
    torch.cuda.synchronize()
    G.compare(out, lse, ro, rl)
    assert float((out.float() - first.float()).abs().max()) <= 2e-2
