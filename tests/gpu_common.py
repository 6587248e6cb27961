"""Shared helpers for the GPU parity tests: put a seeded batch on the device through the library's
own calls, and compute the oracle's answer on the CPU from the same host arrays (never from the
device)."""

from __future__ import annotations

import numpy as np
import torch

from oracle import attention as OA
from oracle import fp8 as OF

# tolerances for bf16 inputs with fp32 accumulation, and for FP8 KV (vs the fp64 oracle on the
# dequantised stored codes)
BF16_MAX_ABS = 2e-2
BF16_MEAN_ABS = 2e-3
FP8_MAX_ABS = 6e-2
LSE_MAX_ABS = 2e-3


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def quantize_chunked(x_bf16: torch.Tensor, scale: float, chunk: int = 1 << 24) -> np.ndarray:
    """Oracle E4M3 codes of a bf16 tensor (chunked to bound host memory)."""
    flat = x_bf16.reshape(-1)
    out = np.empty(flat.numel(), dtype=np.uint8)
    for s in range(0, flat.numel(), chunk):
        out[s:s + chunk] = OF.quantize(flat[s:s + chunk].float().numpy(), scale)
    return out.reshape(tuple(x_bf16.shape))


class GpuBatch:
    """Device copy of a workloads.Batch; FP8 pools are filled by the library's own kv_store."""

    def __init__(self, b, device="cuda"):
        import paged_kv_attention_slot_gb300 as pk

        self.pk = pk
        self.b = b
        P, ps, H, D = b.k_pool.shape
        if b.kv_dtype == "bf16":
            self.k_pool = b.k_pool.to(device)
            self.v_pool = b.v_pool.to(device)
            self.cache = pk.KVCache(self.k_pool, self.v_pool)
        else:
            self.k_pool = torch.zeros((P, ps, H, D), dtype=torch.uint8, device=device)
            self.v_pool = torch.zeros((P, ps, H, D), dtype=torch.uint8, device=device)
            self.cache = pk.KVCache(self.k_pool, self.v_pool, b.k_scale, b.v_scale)
            slots = torch.arange(P * ps, dtype=torch.int64, device=device)
            kh = b.k_pool.to(device).view(P * ps, H, D)
            vh = b.v_pool.to(device).view(P * ps, H, D)
            pk.kv_store(kh, vh, slots, self.cache)
            del kh, vh
        self.q = b.q.to(device)
        self.k_new = b.k_new.to(device)
        self.v_new = b.v_new.to(device)
        self.slots = torch.from_numpy(b.slot_mapping).to(device)

    def store(self):
        self.pk.kv_store(self.k_new, self.v_new, self.slots, self.cache)

    def plan(self, **kw):
        b = self.b
        p = self.pk.Plan()
        args = dict(num_qo_heads=b.num_qo_heads, num_kv_heads=b.num_kv_heads, head_dim=b.head_dim,
                    page_size=b.page_size, mode=b.mode, window_left=b.window_left, sm_scale=b.sm_scale,
                    kv_dtype=b.kv_dtype)
        args.update(kw)
        p.plan(b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, **args)
        return p

    def run(self, plan):
        out, lse = plan.run(self.q, self.cache, return_lse=True)
        torch.cuda.synchronize()
        return out, lse


def oracle_pools(b):
    """The oracle's own pools after this step's KV write (numpy; format tag for oracle.attention)."""
    ps = b.page_size
    if b.kv_dtype == "bf16":
        kp = bf16_bits(b.k_pool).copy()
        vp = bf16_bits(b.v_pool).copy()
        OA.kv_store(kp, vp, bf16_bits(b.k_new), bf16_bits(b.v_new), b.slot_mapping, ps)
        return kp, vp, "bf16_bits"
    kp = quantize_chunked(b.k_pool, b.k_scale)
    vp = quantize_chunked(b.v_pool, b.v_scale)
    OA.kv_store_fp8(kp, vp, b.k_new.float().numpy(), b.v_new.float().numpy(), b.slot_mapping, ps, b.k_scale,
                    b.v_scale)
    return kp, vp, "e4m3"


def oracle_attention(b, kp, vp, fmt, rows=None):
    return OA.paged_attention(
        bf16_bits(b.q), kp, vp, b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, b.page_size,
        sm_scale=b.sm_scale if b.sm_scale > 0 else None, window_left=b.window_left, q_format="bf16_bits",
        kv_format=fmt, k_scale=b.k_scale, v_scale=b.v_scale, rows=rows)


def compare(out, lse, ref_o, ref_lse, rows=None, max_abs=BF16_MAX_ABS, mean_abs=BF16_MEAN_ABS, lse_rel=0.0):
    """Element-by-element comparison on the given token rows (all rows by default).

    lse_rel > 0 widens the LSE bound to LSE_MAX_ABS + lse_rel * |lse| for scores so large that an
    fp32 LSE cannot hold LSE_MAX_ABS absolute (its unit in the last place exceeds it above 2^14)."""
    o = out.float().cpu().numpy().astype(np.float64)
    l = lse.float().cpu().numpy().astype(np.float64)
    if rows is None:
        rows = np.arange(o.shape[0])
    rows = np.asarray(rows)
    d = np.abs(o[rows] - ref_o[rows])
    dl = np.abs(l[rows] - ref_lse[rows])
    assert np.all(np.isfinite(o[rows])), "non-finite output"
    stats = dict(max_abs=float(d.max(initial=0)), mean_abs=float(d.mean()) if d.size else 0.0,
                 lse_max_abs=float(dl.max(initial=0)))
    assert stats["max_abs"] <= max_abs, stats
    assert stats["mean_abs"] <= mean_abs, stats
    if lse_rel > 0:
        assert np.all(dl <= LSE_MAX_ABS + lse_rel * np.abs(ref_lse[rows])), stats
    else:
        assert stats["lse_max_abs"] <= LSE_MAX_ABS, stats
    return stats
