"""Seeded synthetic batches for batched attention over a paged KV cache.

This module is the ONLY code shared by the CUDA path's tests/benchmark and the
CPU oracle.  It draws random numbers and lays out inputs; it holds none of the
method's arithmetic (no attention, no planning, no quantisation).

A batch is described the way the pages' runners hand it to an attention
backend: per-request KV lengths L_i (including this step's tokens), per-request
new-token counts n_i, each request's physical pages in logical order (a row of
the block table), the CSR page table built from them (``kv_indptr`` = running
total of page counts, ``kv_indices`` = the concatenated rows, ``last_page_len``
= fill of the final page), the new tokens' write slots, and random values:

* Q, the new tokens' K/V and the pool's history are N(0, 1) drawn in float32 by
  ``torch.Generator('cpu').manual_seed(seed)`` and rounded to bfloat16;
* physical pages are a random permutation of the pool: the first pages of the
  permutation go to request 0, the next to request 1, and so on, so every
  request's pages are distinct and out of order;
* for FP8-KV batches the pool history holds the pre-quantisation values, and
  the per-tensor scale is amax(|K|) / 448 (resp. V) over the layer's pool and
  new tokens, in float32.

The five named workloads are the shapes the attention backends on the pages
serve (tiny decode; Llama-3-8B-shaped decode; prefix-cached extend with a
token-granular pool; Llama-3-70B-shaped ragged decode; long-context FP8-KV
decode with an optional 4096-token sliding window).
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

E4M3_MAX = 448.0


@dataclass
class Batch:
    name: str
    mode: str  # "decode" (one new token per request) or "extend"
    page_size: int
    num_pages: int
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    kv_len: np.ndarray  # [B] L_i, including this step's tokens
    q_len: np.ndarray  # [B] n_i
    block_rows: list  # per request: physical page ids in logical order
    qo_indptr: np.ndarray  # [B+1] int32
    kv_indptr: np.ndarray  # [B+1] int32
    kv_indices: np.ndarray  # [nnz] int32
    last_page_len: np.ndarray  # [B] int32
    slot_mapping: np.ndarray  # [T] int64, write slot of each new token
    q: torch.Tensor  # [T, Hq, D] bf16
    k_new: torch.Tensor  # [T, Hkv, D] bf16
    v_new: torch.Tensor  # [T, Hkv, D] bf16
    k_pool: torch.Tensor  # [P, ps, Hkv, D] bf16 (FP8 batches: values before quantisation)
    v_pool: torch.Tensor
    kv_dtype: str = "bf16"  # "bf16" or "e4m3"
    k_scale: float = 1.0
    v_scale: float = 1.0
    window_left: int = -1
    sm_scale: float = 0.0  # <= 0 means 1/sqrt(D)
    meta: dict = field(default_factory=dict)

    @property
    def batch_size(self) -> int:
        return len(self.kv_len)

    @property
    def num_tokens(self) -> int:
        return int(self.qo_indptr[-1])

    def kv_bytes_read(self) -> int:
        """Bytes of K and V a decode pass must read: every visible key row, K and V, all KV heads."""
        elem = 1 if self.kv_dtype == "e4m3" else 2
        if self.window_left >= 0:
            vis = np.minimum(self.kv_len, self.window_left + 1)
        else:
            vis = self.kv_len
        return int(vis.sum()) * self.num_kv_heads * self.head_dim * elem * 2


def _randn_bf16(g: torch.Generator, shape, chunk_rows: int = 1 << 14) -> torch.Tensor:
    """N(0,1) float32 rounded to bf16, drawn in row chunks to bound peak host memory."""
    out = torch.empty(shape, dtype=torch.bfloat16)
    flat = out.view(shape[0], -1)
    for r0 in range(0, shape[0], chunk_rows):
        r1 = min(shape[0], r0 + chunk_rows)
        flat[r0:r1] = torch.randn((r1 - r0, flat.shape[1]), generator=g, dtype=torch.float32).to(torch.bfloat16)
    return out


def make_batch(
    kv_lens,
    q_lens,
    page_size: int,
    num_qo_heads: int,
    num_kv_heads: int,
    head_dim: int,
    seed: int,
    num_pages: int | None = None,
    pool_factor: float = 1.25,
    kv_dtype: str = "bf16",
    window_left: int = -1,
    sm_scale: float = 0.0,
    name: str = "custom",
    mode: str | None = None,
    shared_prefix: int = 0,
) -> Batch:
    """Build one seeded batch.  kv_lens[i] >= q_lens[i] >= 0; a request with kv_len 0 owns no page.

    ``shared_prefix`` > 0 (a multiple of page_size): the first shared_prefix tokens of every request
    live on the SAME physical pages (a common system prompt); each request's remaining kv_len -
    shared_prefix tokens, which hold its q_len new tokens, are on pages of its own.
    """
    kv_len = np.asarray(kv_lens, dtype=np.int64)
    q_len = np.asarray(q_lens, dtype=np.int64)
    if kv_len.shape != q_len.shape or np.any(q_len < 0) or np.any(kv_len < q_len):
        raise ValueError("need kv_len >= q_len >= 0 per request")
    if shared_prefix % page_size or np.any(kv_len - shared_prefix < q_len):
        raise ValueError("the shared prefix must be whole pages and precede every request's new tokens")
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    n_shared = shared_prefix // page_size
    own = [(int(L) - shared_prefix + page_size - 1) // page_size for L in kv_len]
    counts = [n_shared + c for c in own]
    need = n_shared + sum(own)
    P = int(num_pages) if num_pages is not None else max(1, math.ceil(pool_factor * need))
    if P < need:
        raise ValueError(f"pool of {P} pages cannot hold {need}")
    perm = torch.randperm(P, generator=g).numpy().astype(np.int64)
    shared_rows = perm[:n_shared].copy()
    rows, at = [], n_shared
    for c in own:
        rows.append(np.concatenate([shared_rows, perm[at : at + c]]))
        at += c
    k_pool = _randn_bf16(g, (P, page_size, num_kv_heads, head_dim))
    v_pool = _randn_bf16(g, (P, page_size, num_kv_heads, head_dim))
    T = int(q_len.sum())
    q = _randn_bf16(g, (T, num_qo_heads, head_dim)) if T else torch.empty((0, num_qo_heads, head_dim), dtype=torch.bfloat16)
    k_new = _randn_bf16(g, (T, num_kv_heads, head_dim)) if T else torch.empty((0, num_kv_heads, head_dim), dtype=torch.bfloat16)
    v_new = _randn_bf16(g, (T, num_kv_heads, head_dim)) if T else torch.empty((0, num_kv_heads, head_dim), dtype=torch.bfloat16)

    # the runner's per-token write addresses: the new tokens are each request's last positions
    slots = []
    for i, (L, n) in enumerate(zip(kv_len, q_len)):
        for pos in range(int(L - n), int(L)):
            slots.append(int(rows[i][pos // page_size]) * page_size + pos % page_size)
    qo_indptr = np.concatenate([[0], np.cumsum(q_len)]).astype(np.int32)
    kv_indptr = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    kv_indices = (np.concatenate(rows) if rows and need else np.zeros(0, dtype=np.int64)).astype(np.int32)
    last = np.array([(int(L) - (c - 1) * page_size) if c else 0 for L, c in zip(kv_len, counts)], dtype=np.int32)

    k_scale = v_scale = 1.0
    if kv_dtype == "e4m3":
        k_amax = max(float(k_pool.float().abs().max()), float(k_new.float().abs().max()) if T else 0.0)
        v_amax = max(float(v_pool.float().abs().max()), float(v_new.float().abs().max()) if T else 0.0)
        k_scale = float(np.float32(k_amax) / np.float32(E4M3_MAX))
        v_scale = float(np.float32(v_amax) / np.float32(E4M3_MAX))
    elif kv_dtype != "bf16":
        raise ValueError("kv_dtype must be 'bf16' or 'e4m3'")
    if mode is None:
        mode = "decode" if np.all(q_len == 1) else "extend"
    return Batch(
        name=name, mode=mode, page_size=page_size, num_pages=P, num_qo_heads=num_qo_heads,
        num_kv_heads=num_kv_heads, head_dim=head_dim, kv_len=kv_len, q_len=q_len, block_rows=rows,
        qo_indptr=qo_indptr, kv_indptr=kv_indptr, kv_indices=kv_indices, last_page_len=last,
        slot_mapping=np.asarray(slots, dtype=np.int64), q=q, k_new=k_new, v_new=v_new,
        k_pool=k_pool, v_pool=v_pool, kv_dtype=kv_dtype, k_scale=k_scale, v_scale=v_scale,
        window_left=window_left, sm_scale=sm_scale,
        meta={"shared_prefix": int(shared_prefix), "shared_pages": shared_rows} if shared_prefix else {},
    )


# ------------------------------------------------------------------------------------------------
# the named workloads
# ------------------------------------------------------------------------------------------------
WORKLOADS = {
    1: "tiny paged decode: 4 requests, KV lengths {7,16,33,64}, page 16, 32-page pool, 4q/2kv heads, D 64",
    2: "Llama-3-8B-shaped paged decode: batch 64, 32q/8kv heads, D 128, KV length U[512,4096], page 16",
    3: "prefix-cached causal extend: batch 8, new U[128,2048], prefix U[0,4096], page 1, 32q/8kv, D 128",
    4: "Llama-3-70B-shaped ragged decode: batch 256, 64q/8kv, D 128, KV length log-normal median 1024, page 64",
    5: "long-context FP8-KV decode: batch 2, KV length 131072, 32q/8kv, D 128, e4m3 K/V, page 128",
}


def shared_prefix_workload(seed_offset: int = 0, batch: int = 64, shared_prefix: int = 4096,
                           suffix_max: int = 512) -> Batch:
    """Decode batch whose requests share a system prompt (the case cascade attention serves).

    Llama-3-8B-shaped heads (32 q / 8 kv, head_dim 128), page size 16, a shared prefix of
    ``shared_prefix`` tokens on common pages, and per-request suffixes of U[1, suffix_max] tokens
    (the last of which is the new token), bf16 N(0, 1) values, seed 1006 (+ 100000 * seed_offset).
    """
    seed = 1006 + 100000 * int(seed_offset)
    g = torch.Generator(device="cpu").manual_seed(seed + 7919)
    suf = torch.randint(1, suffix_max + 1, (batch,), generator=g).tolist()
    L = [shared_prefix + x for x in suf]
    return make_batch(L, [1] * batch, 16, 32, 8, 128, seed, name="shared_prefix_decode", mode="decode",
                      shared_prefix=shared_prefix)


def workload(n: int, window_left: int = -1, scale_batch: float = 1.0, seed_offset: int = 0) -> Batch:
    """Named workload n (1..5), seed 1000 + n (+ 100000 * seed_offset, e.g. one batch per rank).

    ``window_left`` applies to workload 5 only; ``scale_batch`` scales the batch size (bounded samples).
    """
    seed = 1000 + n + 100000 * int(seed_offset)
    g = torch.Generator(device="cpu").manual_seed(seed + 7919)  # lengths use their own stream
    if n == 1:
        L = [7, 16, 33, 64]
        return make_batch(L, [1] * 4, 16, 4, 2, 64, seed, num_pages=32, sm_scale=1.0 / 8.0,
                          name="tiny_decode", mode="decode")
    if n == 2:
        B = max(1, int(round(64 * scale_batch)))
        L = torch.randint(512, 4097, (B,), generator=g).tolist()
        return make_batch(L, [1] * B, 16, 32, 8, 128, seed, name="llama8b_decode", mode="decode")
    if n == 3:
        B = max(1, int(round(8 * scale_batch)))
        nq = torch.randint(128, 2049, (B,), generator=g).tolist()
        pre = torch.randint(0, 4097, (B,), generator=g).tolist()
        L = [a + b for a, b in zip(nq, pre)]
        return make_batch(L, nq, 1, 32, 8, 128, seed, name="prefix_extend", mode="extend")
    if n == 4:
        B = max(1, int(round(256 * scale_batch)))
        z = torch.randn((B,), generator=g, dtype=torch.float64).numpy()
        L = np.clip(np.rint(np.exp(math.log(1024.0) + 1.0 * z)), 16, 32768).astype(np.int64).tolist()
        return make_batch(L, [1] * B, 64, 64, 8, 128, seed, name="llama70b_ragged_decode", mode="decode")
    if n == 5:
        B = max(1, int(round(2 * scale_batch)))
        L = [131072] * B
        return make_batch(L, [1] * B, 128, 32, 8, 128, seed, num_pages=(131072 // 128) * B, kv_dtype="e4m3",
                          window_left=window_left, name="fp8_long_decode" + ("_window" if window_left >= 0 else ""),
                          mode="decode")
    raise ValueError("workloads are numbered 1..5")
