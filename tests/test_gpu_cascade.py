"""GPU parity of cascade (shared-prefix) attention ("vLLM 源码完全拆解（六）：Attention Backend", section
«Cascade Attention 把共享前缀只算一次»): the shared prefix computed once for every query of the batch
(non-causal, split-KV), each request's own suffix (causal), merged by LSE -- against the oracle's flat
causal pass over prefix + suffix."""

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


def suffix_csr(b):
    """Each request's own pages (after the shared ones) as a CSR page table."""
    ns = len(b.meta["shared_pages"])
    ps = b.page_size
    rows = [r[ns:] for r in b.block_rows]
    suf = (b.kv_len - b.meta["shared_prefix"]).astype(np.int64)
    indptr = np.concatenate([[0], np.cumsum([len(r) for r in rows])]).astype(np.int32)
    indices = np.concatenate(rows + [np.zeros(0, np.int64)]).astype(np.int32)
    last = np.array([x - (len(r) - 1) * ps if len(r) else 0 for x, r in zip(suf, rows)], dtype=np.int32)
    return indptr, indices, last


def cascade_plan(b, **kw):
    import paged_kv_attention_slot_gb300 as pk

    si, sx, sl = suffix_csr(b)
    return pk.CascadePlan().plan(b.qo_indptr, b.meta["shared_pages"], b.page_size, si, sx, sl,
                                 num_qo_heads=b.num_qo_heads, num_kv_heads=b.num_kv_heads, head_dim=b.head_dim,
                                 page_size=b.page_size, sm_scale=b.sm_scale, **kw)


def _run(b):
    g = G.GpuBatch(b)
    g.store()
    cp = cascade_plan(b)
    out, lse = cp.run(g.q, g.cache, return_lse=True)
    torch.cuda.synchronize()
    kp, vp, fmt = G.oracle_pools(b)
    ro, rl = G.oracle_attention(b, kp, vp, fmt)
    return G.compare(out, lse, ro, rl), cp, g


def test_cascade_decode_shared_system_prompt():
    # batch 64 decode, shared prefix 4096 tokens on common pages, suffixes U[1, 512]
    b = W.shared_prefix_workload()
    stats, cp, _ = _run(b)
    assert cp.shared.info()["num_prefill_partials"] > 0  # the shared pass is split over the SMs
    assert cp.suffix.info()["mode"] == 0


@pytest.mark.parametrize("ps", [1, 16])
def test_cascade_extend_and_mixed(ps):
    # several new tokens per request (and one request with a single token: a mixed suffix plan)
    shared = 48 * ps if ps > 1 else 700
    b = W.make_batch([shared + 300, shared + 1, shared + 90, shared + 65], [200, 1, 90, 64], ps, 16, 4, 128,
                     seed=100 + ps, shared_prefix=shared)
    stats, cp, _ = _run(b)
    assert cp.suffix.info()["mode"] == 2


def test_cascade_matches_flat_decode_and_replans_in_place():
    # the same batch by the flat decode plan and by cascade agree within the oracle tolerance, and a
    # second cascade plan on the same object (new shared length) still matches the oracle
    b = W.shared_prefix_workload(batch=16, shared_prefix=1024, suffix_max=200)
    stats, cp, g = _run(b)
    flat = g.plan()
    fo, fl = g.run(flat)
    co, cl = cp.run(g.q, g.cache, return_lse=True)
    torch.cuda.synchronize()
    assert (fo.float() - co.float()).abs().max().item() <= 2 * G.BF16_MAX_ABS
    b2 = W.shared_prefix_workload(seed_offset=1, batch=16, shared_prefix=2048, suffix_max=64)
    g2 = G.GpuBatch(b2)
    g2.store()
    si, sx, sl = suffix_csr(b2)
    cp.plan(b2.qo_indptr, b2.meta["shared_pages"], b2.page_size, si, sx, sl, num_qo_heads=32, num_kv_heads=8,
            head_dim=128, page_size=16)
    out, lse = cp.run(g2.q, g2.cache, return_lse=True)
    torch.cuda.synchronize()
    kp, vp, fmt = G.oracle_pools(b2)
    ro, rl = G.oracle_attention(b2, kp, vp, fmt)
    G.compare(out, lse, ro, rl)
