"""GPU parity over a seeded random sweep of configurations that combine the axes the other GPU tests
vary one at a time: mode (decode, extend, mixed), page size, GQA ratio, head dim, sliding window, KV
dtype, softmax scale, split cap, SM count the plan is made for, and request lengths (idle requests,
extends without a prefix, one-token extends next to decodes).  Every case compares every output
element and LSE with the fp64 oracle on the same seeded inputs."""

import numpy as np
import pytest

import workloads as W
from tests import gpu_common as G

CASES = 40


@pytest.fixture(scope="module")
def _lib():
    import paged_kv_attention_slot_gb300 as pk

    pk._lib.lib()
    assert pk.device_error() == 0
    yield
    assert pk.device_error() == 0


def _draw(case: int):
    """One configuration, a pure function of the case number."""
    r = np.random.default_rng(5000 + case)
    mode = ["decode", "extend", "mixed"][case % 3]
    kv_dtype = "e4m3" if mode == "decode" and r.random() < 0.35 else "bf16"
    # the extend path (and FP8 KV) needs head_dim 128; decode also takes 64
    D = 128 if (mode != "decode" or kv_dtype == "e4m3") else int(r.choice([64, 128]))
    hkv = int(r.choice([1, 2, 4, 8]))
    group = int(r.choice([1, 2, 4, 8, 16]))
    ps = int(r.choice([1, 2, 8, 16, 64, 128]))
    B = int(r.integers(1, 7))
    window = -1 if r.random() < 0.6 else int(r.integers(0, 400))
    sm_scale = 0.0 if r.random() < 0.7 else float(r.uniform(0.02, 0.2))
    q_lens, kv_lens = [], []
    for _ in range(B):
        u = r.random()
        if u < 0.1:  # idle: cached keys, no new token
            q, pre = 0, int(r.integers(0, 500))
        elif mode == "decode" or (mode == "mixed" and u < 0.5):
            q, pre = 1, int(r.integers(0, 1500))
        else:
            q = int(r.integers(1, 200))
            pre = 0 if r.random() < 0.25 else int(r.integers(0, 700))
        q_lens.append(q)
        kv_lens.append(q + pre)
    plan_kw = {"max_splits": int(r.choice([0, 0, 1, 3])), "num_sms": int(r.choice([152, 152, 40]))}
    b = W.make_batch(kv_lens, q_lens, ps, hkv * group, hkv, D, seed=6000 + case, kv_dtype=kv_dtype,
                     window_left=window, sm_scale=sm_scale, mode=mode)
    return b, plan_kw


@pytest.mark.gpu
@pytest.mark.parametrize("case", range(CASES))
def test_random_configuration(_lib, case):
    b, plan_kw = _draw(case)
    g = G.GpuBatch(b)
    g.store()
    plan = g.plan(**plan_kw)
    out, lse = g.run(plan)
    kp, vp, fmt = G.oracle_pools(b)
    ro, rl = G.oracle_attention(b, kp, vp, fmt)
    tol = G.FP8_MAX_ABS if b.kv_dtype == "e4m3" else G.BF16_MAX_ABS
    G.compare(out, lse, ro, rl, max_abs=tol)


def test_sweep_spans_every_axis():
    """The drawn configurations cover each value of each axis at least once (host only)."""
    seen = {k: set() for k in ("mode", "dtype", "D", "ps", "window", "splits", "idle", "scale")}
    for case in range(CASES):
        b, kw = _draw(case)
        q = np.diff(b.qo_indptr)
        seen["mode"].add(b.mode)
        seen["dtype"].add(b.kv_dtype)
        seen["D"].add(b.head_dim)
        seen["ps"].add(b.page_size)
        seen["window"].add(b.window_left >= 0)
        seen["splits"].add(kw["max_splits"])
        seen["idle"].add(bool(np.any(q == 0)))
        seen["scale"].add(b.sm_scale > 0)
    assert seen["mode"] == {"decode", "extend", "mixed"}
    assert seen["dtype"] == {"bf16", "e4m3"}
    assert seen["D"] == {64, 128}
    assert len(seen["ps"]) >= 5
    assert seen["window"] == {True, False}
    assert seen["splits"] == {0, 1, 3}
    assert seen["idle"] == {True, False}
    assert seen["scale"] == {True, False}
