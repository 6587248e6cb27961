"""The prefill kernel's bounded waits: a wait that runs out records PKV_DEVERR_TIMEOUT, the CTA
drains what it issued, frees its tensor memory and exits, and the device stays usable.

The failure is made the allowed way: with the wait limit shortened to ~20,000 clock cycles, every
prefill CTA first waits on a barrier that nothing arrives at (pkv_test_hold_wait), so that wait runs
out; nothing faults, traps or hangs.  The next ordinary run on the same device must match the oracle.
"""

import pytest
import torch

import workloads as W
from tests import gpu_common as G

pytestmark = pytest.mark.gpu

PKV_DEVERR_TIMEOUT = 3


def _held_run(pk, g, plan):
    L = pk._lib.lib()
    pk.set_wait_limit(20000)
    pk._lib.check(L.pkv_test_hold_wait(1))
    try:
        plan.run(g.q, g.cache, return_lse=True)
        torch.cuda.synchronize()
    finally:
        pk._lib.check(L.pkv_test_hold_wait(0))
        pk.set_wait_limit(0)
    return pk.device_error()


@pytest.mark.parametrize("case", ["two_tiles", "split"])
def test_prefill_wait_timeout_is_reported_and_the_device_stays_usable(case):
    import paged_kv_attention_slot_gb300 as pk

    pk._lib.lib()
    assert pk.device_error() == 0
    if case == "two_tiles":  # many CTAs, two query tiles each, several key tiles
        b = W.make_batch([3000, 700, 129], [600, 300, 129], 1, 16, 4, 128, seed=95)
    else:  # split-KV items followed by the merge kernel (which then merges unwritten partials)
        b = W.make_batch([20000], [64], 16, 32, 8, 128, seed=96)
    g = G.GpuBatch(b)
    g.store()
    plan = g.plan()
    assert _held_run(pk, g, plan) == PKV_DEVERR_TIMEOUT
    assert pk.device_error() == 0  # read and cleared above
    # the same plan on the same device, limit restored: every element against the oracle
    out, lse = g.run(plan)
    assert pk.device_error() == 0
    kp, vp, fmt = G.oracle_pools(b)
    ro, rl = G.oracle_attention(b, kp, vp, fmt)
    G.compare(out, lse, ro, rl)
