"""pkv_attn_decode_run_noalloc: decode for callers that cannot allocate device memory.

Such callers (a host framework whose memory pool forbids raw cudaMalloc, because an allocation
behind the pool's back breaks its accounting; an embedded runtime with a fixed device-memory budget)
cannot provide the plan workspace; this entry point keeps the plan metadata and the split-KV partials in the
library's own static device array instead.  The test calls it through the C ABI, twice in a row on
different batches (and once more on the first), and checks each result against the ordinary
workspace-based pkv_attn_decode_run on the same plan arguments.

The file name makes pytest collect it last, so a stop-at-first-failure run has already run every
other test before it.  It must pass alone in a fresh process as well as after the other tests.
"""

import ctypes as C

import numpy as np
import pytest
import torch

import workloads as W
from tests import gpu_common as G

pytestmark = pytest.mark.gpu


def _plan_kw(b, **extra):
    kw = dict(num_qo_heads=b.num_qo_heads, num_kv_heads=b.num_kv_heads, head_dim=b.head_dim, page_size=b.page_size,
              mode="decode", window_left=b.window_left, sm_scale=b.sm_scale, kv_dtype=b.kv_dtype)
    kw.update(extra)
    return kw


def _noalloc(pk, plan, g, out, lse):
    st = pk._lib.lib().pkv_attn_decode_run_noalloc(plan._h, g.q.data_ptr(), C.byref(g.cache.struct),
                                                   out.data_ptr(), lse.data_ptr(),
                                                   torch.cuda.current_stream().cuda_stream)
    pk._lib.check(st)


def test_noalloc_decode_matches_workspace_decode_on_consecutive_calls():
    import paged_kv_attention_slot_gb300 as pk

    batches = [
        # long requests on few SMs: split-KV with merges, so the static scratch holds partials
        W.make_batch([3000, 9000, 64, 4500, 12000, 1], [1] * 6, 16, 32, 8, 128, seed=77),
        # a different batch straight after: FP8 cache, sliding window, other page size
        W.make_batch([700, 20, 5000, 129], [1] * 4, 128, 32, 8, 128, seed=78, kv_dtype="e4m3", window_left=900),
    ]
    gpu = [G.GpuBatch(b) for b in batches]
    refs = []
    for b, g in zip(batches, gpu):
        g.store()
        ref_plan = pk.Plan().plan(b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, **_plan_kw(b, num_sms=64))
        refs.append(g.run(ref_plan))
    host_plans = [pk.Plan().plan(b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len,
                                 **_plan_kw(b, num_sms=64), host_only=True) for b in batches]
    assert host_plans[0].info()["num_merge"] > 0

    tol = {"bf16": G.BF16_MAX_ABS, "e4m3": G.FP8_MAX_ABS}
    for k in (0, 1, 0):  # consecutive calls: batch A, batch B, batch A again
        b, g = batches[k], gpu[k]
        out = torch.full_like(g.q, float("nan"))
        lse = torch.full(g.q.shape[:2], float("nan"), dtype=torch.float32, device=g.q.device)
        _noalloc(pk, host_plans[k], g, out, lse)
        torch.cuda.synchronize()
        ref_o, ref_lse = refs[k]
        d = (out.float() - ref_o.float()).abs()
        assert torch.isfinite(out.float()).all()
        assert float(d.max()) <= tol[b.kv_dtype]
        assert float(d.mean()) <= G.BF16_MEAN_ABS
        assert float((lse - ref_lse).abs().max()) <= G.LSE_MAX_ABS
    assert pk.device_error() == 0

    # and the result is the attention the oracle defines
    kp, vp, fmt = G.oracle_pools(batches[0])
    ro, rl = G.oracle_attention(batches[0], kp, vp, fmt)
    G.compare(out, lse, ro, rl)


def test_noalloc_rejects_plans_beyond_the_static_scratch():
    import paged_kv_attention_slot_gb300 as pk

    b = W.make_batch([4], [1], 16, 32, 8, 128, seed=5)
    g = G.GpuBatch(b)
    # a plan for 512 requests of 65536 keys on a large (pretend) SM count needs far more than 32 MiB
    # of split-KV partials; the call must refuse it before touching the GPU
    kv_indptr = np.arange(0, 512 * 4096 + 1, 4096, dtype=np.int32)
    kv_indices = np.zeros(512 * 4096, dtype=np.int32)
    plan = pk.Plan().plan(np.arange(513, dtype=np.int32), kv_indptr, kv_indices, np.full(512, 16, np.int32),
                          num_qo_heads=32, num_kv_heads=8, head_dim=128, page_size=16, mode="decode",
                          num_sms=4096, host_only=True)
    assert plan.info()["workspace_bytes"] > 32 << 20
    q = torch.zeros((512, 32, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty((512, 32), dtype=torch.float32, device="cuda")
    st = pk._lib.lib().pkv_attn_decode_run_noalloc(plan._h, q.data_ptr(), C.byref(g.cache.struct), out.data_ptr(),
                                                   lse.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == pk._lib.PKV_EWORKSPACE
    assert "no-allocation path" in pk._lib.lib().pkv_last_error().decode()
