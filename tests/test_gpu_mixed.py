"""GPU parity of mixed decode + extend batches (one plan, decode kernel + prefill kernel, one output)
against the CPU oracle.

The decode/extend split follows "vLLM Attention 后端与 FlashInfer 元数据", sections «为什么先把 Decode 移到前面»
and «FlashInfer Builder 的结果»: one-token requests go to the decode path, the others to the
prefill/extend path, and both write their rows of the same output tensor."""

import json
import os

import numpy as np
import pytest
import torch

import workloads as W
from tests import gpu_common as G

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import paged_kv_attention_slot_gb300 as pk

    pk._lib.lib()
    assert pk.device_error() == 0
    yield
    assert pk.device_error() == 0


def _case(b, **plan_kw):
    g = G.GpuBatch(b)
    g.store()
    plan = g.plan(**plan_kw)
    out, lse = g.run(plan)
    kp, vp, fmt = G.oracle_pools(b)
    ro, rl = G.oracle_attention(b, kp, vp, fmt)
    G.compare(out, lse, ro, rl)
    return plan, g, out, lse


def test_mixed_worked_example_shapes():
    """The printed batch: A decodes 1 token over 128 keys, B prefills 4 tokens, C extends 3 tokens over
    35 keys (page size 16), random values."""
    ex = json.load(open(os.path.join(GOLDEN, "vllm_worked_example.json")))
    q_lens = np.diff(ex["query_start_loc"]).tolist()
    b = W.make_batch(ex["seq_lens"], q_lens, ex["page_size"], 32, 8, 128, seed=31, mode="mixed")
    plan, *_ = _case(b)
    info = plan.info()
    assert (info["num_decodes"], info["num_prefill_tokens"]) == (1, 7)


@pytest.mark.parametrize("num_sms", [152, 16])
def test_mixed_interleaved_decode_and_extend(num_sms):
    """Decode requests interleaved with extends (not decode-first); num_sms=16 forces split-KV decode."""
    rng = np.random.default_rng(7)
    L, n = [], []
    for i in range(24):
        if i % 5 == 2:
            q = int(rng.integers(2, 300))
            L.append(q + int(rng.integers(0, 1500)))
            n.append(q)
        elif i % 7 == 3:  # a few long decodes, split across CTAs when SMs are few
            L.append(int(rng.integers(20000, 24000)))
            n.append(1)
        else:
            L.append(int(rng.integers(1, 3000)))
            n.append(1)
    b = W.make_batch(L, n, 16, 32, 8, 128, seed=32, mode="mixed")
    plan, *_ = _case(b, num_sms=num_sms)
    info = plan.info()
    assert info["num_decodes"] == sum(1 for q in n if q == 1)
    if num_sms == 16:
        assert info["num_merge"] > 0


def test_mixed_with_idle_requests_window_and_page_size_1():
    b = W.make_batch([40, 0, 700, 1, 260, 33], [1, 0, 129, 1, 1, 33], 1, 16, 4, 128, seed=33, mode="mixed",
                     window_left=100)
    _case(b)


def test_mixed_runs_write_disjoint_rows():
    """decode_run and prefill_run of a mixed plan each write only their own rows."""
    import paged_kv_attention_slot_gb300 as pk

    b = W.make_batch([500, 90, 1200, 64], [1, 90, 1, 17], 16, 16, 4, 128, seed=34, mode="mixed")
    g = G.GpuBatch(b)
    g.store()
    plan = g.plan()
    sentinel = torch.full_like(g.q, 7.0)
    out = sentinel.clone()
    lse = torch.full(g.q.shape[:2], float("nan"), dtype=torch.float32, device=g.q.device)
    st = pk._lib.lib().pkv_attn_decode_run(plan._h, g.q.data_ptr(), pk._lib.C.byref(g.cache.struct),
                                           out.data_ptr(), lse.data_ptr(), torch.cuda.current_stream().cuda_stream)
    pk._lib.check(st)
    torch.cuda.synchronize()
    dec_rows = [int(b.qo_indptr[i]) for i in range(b.batch_size) if b.q_len[i] == 1]
    ext_rows = [r for r in range(b.num_tokens) if r not in dec_rows]
    assert torch.equal(out[ext_rows], sentinel[ext_rows])
    assert not torch.equal(out[dec_rows], sentinel[dec_rows])
    st = pk._lib.lib().pkv_attn_prefill_run(plan._h, g.q.data_ptr(), pk._lib.C.byref(g.cache.struct),
                                            out.data_ptr(), lse.data_ptr(), torch.cuda.current_stream().cuda_stream)
    pk._lib.check(st)
    torch.cuda.synchronize()
    kp, vp, fmt = G.oracle_pools(b)
    ro, rl = G.oracle_attention(b, kp, vp, fmt)
    G.compare(out, lse, ro, rl)
