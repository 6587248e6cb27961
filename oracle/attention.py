"""KV write, paged attention and state merge, restated in float64 (oracle; test infrastructure only).

Definition followed (plain, unblocked, unfused):

* "手写 mini-sglang 阶段四 · GPU 注意力后端", section «在 CPU 上验证» (the CPU
  reference ``paged_attention``): for each request, gather its pages in logical
  order, keep the first ``kv_len`` tokens, treat the request's queries as the
  LAST n positions of the sequence (causal mask aligned bottom-right), and take
  softmax(q k^T * scale) v with the query heads grouped onto KV heads.
* "vLLM 源码完全拆解（六）：Attention Backend", sections «为什么 KV 写入在 Attention
  之前» (the KV write happens first, so a query sees the keys of its own step)
  and «九条必须成立的不变量» (items 3-6: query_start_loc starts at 0 and is
  non-decreasing; seq_len - query_len is the context readable before the step;
  slot_mapping entries point into pages the request owns).
* "SGLang 源码完全拆解(八)：Attention Backend", sections «统一元数据的编译» (CSR
  page table), «mask 从哪里来» (sliding window keeps keys k >= q - w) and «extend
  的两种形态» (the merge of two attention states by their log-sum-exp).

Readings taken where the pages are silent (each is listed with its reason in
the design notes of this repository):

* GQA: query head h reads KV head h // (Hq / Hkv) (contiguous groups; the same
  grouping as the ``enable_gqa`` flag of the library routine the reference uses).
* A window ``w >= 0`` keeps keys j with P - w <= j <= P (w + 1 keys including
  the query's own position P).
* A negative slot in slot_mapping marks a padding token: nothing is written.
* Exported log-sum-exp values are natural logarithms of the softmax
  denominator of the scaled scores.
"""

from __future__ import annotations

import math

import numpy as np

from . import fp8 as _fp8


# ----------------------------------------------------------------------------------------------
# element formats
# ----------------------------------------------------------------------------------------------
def bf16_bits_to_f64(bits) -> np.ndarray:
    """bfloat16 bit patterns -> exact float64: a bf16 value is the upper half of a binary32."""
    u = np.asarray(bits).view(np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def to_f64(x, fmt: str = "float", scale: float = 1.0) -> np.ndarray:
    """Widen stored elements to float64 exactly.

    fmt: "float" (any numpy float array), "bf16_bits" (uint16/int16 bit patterns)
    or "e4m3" (uint8 codes; multiplied by ``scale``).
    """
    if fmt == "float":
        return np.asarray(x, dtype=np.float64)
    if fmt == "bf16_bits":
        return bf16_bits_to_f64(x)
    if fmt == "e4m3":
        return _fp8.dequantize(x, scale)
    raise ValueError(f"unknown element format {fmt!r}")


# ----------------------------------------------------------------------------------------------
# the KV write
# ----------------------------------------------------------------------------------------------
def page_and_offset(slot: int, page_size: int):
    """Slot -> (physical page, offset in page)."""
    return slot // page_size, slot % page_size


def kv_store(k_pool, v_pool, k, v, slot_mapping, page_size: int) -> None:
    """Scatter this step's K/V rows into the pools, in place.

    Pools are [num_pages, page_size, Hkv, D]; k, v are [T, Hkv, D] in the same
    element type as the pools.  Token t goes to pool[slot // ps, slot % ps];
    a negative slot is padding and writes nothing.
    """
    for t, slot in enumerate(np.asarray(slot_mapping, dtype=np.int64)):
        if slot < 0:
            continue
        page, off = page_and_offset(int(slot), page_size)
        k_pool[page, off] = k[t]
        v_pool[page, off] = v[t]


def kv_store_fp8(k_codes, v_codes, k_fp32, v_fp32, slot_mapping, page_size: int, k_scale: float, v_scale: float):
    """FP8 KV write: quantise each row with the layer's scale, then scatter the codes."""
    kq = _fp8.quantize(k_fp32, k_scale)
    vq = _fp8.quantize(v_fp32, v_scale)
    kv_store(k_codes, v_codes, kq, vq, slot_mapping, page_size)


# ----------------------------------------------------------------------------------------------
# paged attention
# ----------------------------------------------------------------------------------------------
def kv_len_of(pages_i: int, last_page_len_i: int, page_size: int) -> int:
    """L_i = (pages - 1) * page_size + last_page_len (0 when the request owns no page)."""
    return 0 if pages_i == 0 else (pages_i - 1) * page_size + last_page_len_i


def kv_head_of(h: int, group: int) -> int:
    """KV head read by query head h when ``group`` query heads share one KV head."""
    return h // group


def query_position(kv_len: int, q_len: int, t: int) -> int:
    """Absolute position of new token t: the queries are the last q_len positions."""
    return kv_len - q_len + t


def visible_range(position: int, window_left: int):
    """Inclusive key range [lo, hi] seen by a query at ``position`` (causal, optional window)."""
    lo = 0 if window_left < 0 else max(0, position - window_left)
    return lo, position


def full_range(kv_len: int):
    """Inclusive key range [0, kv_len - 1] seen by every query of a non-causal call.

    "SGLang 源码完全拆解(八)：Attention Backend", section «extend 的两种形态：ragged 直算与 paged + merge»:
    the cached-prefix segment is attended with causal=False, because every prefix key lies before
    every new query, so the whole segment is visible.
    """
    return 0, kv_len - 1


def gather_logical(pool, pages, kv_len: int, page_size: int):
    """Logical token j of a request lives at pool[pages[j // ps], j % ps]; returns [kv_len, ...]."""
    j = np.arange(kv_len)
    return pool[np.asarray(pages, dtype=np.int64)[j // page_size], j % page_size]


def attend(q, K, V, lo: int, hi: int, scale: float):
    """softmax over keys lo..hi of (q . K_j) * scale, applied to V; returns (o, natural-log lse)."""
    s = (K[lo : hi + 1] @ q) * scale
    m = s.max()
    e = np.exp(s - m)
    den = e.sum()
    return (e @ V[lo : hi + 1]) / den, m + math.log(den)


def paged_attention(
    q,
    k_pool,
    v_pool,
    qo_indptr,
    kv_indptr,
    kv_indices,
    last_page_len,
    page_size: int,
    sm_scale: float | None = None,
    window_left: int = -1,
    q_format: str = "float",
    kv_format: str = "float",
    k_scale: float = 1.0,
    v_scale: float = 1.0,
    rows=None,
    causal: bool = True,
):
    """Batched attention over a paged KV cache, float64.

    q: [T, Hq, D]; pools: [num_pages, page_size, Hkv, D].  Element formats as in
    ``to_f64``.  ``rows``: optional iterable of token rows of q to compute (the
    others are left NaN), for sampling large batches.  ``causal=False``: every
    query sees all kv_len keys of its request (``full_range``); a window is then
    not allowed and kv_len may be smaller than the number of queries.  A
    non-causal request with kv_len 0 yields the empty state (o = 0, lse = -inf),
    which ``merge_states`` treats as the identity: in the paged + merge form of
    extend ("SGLang 源码完全拆解(八)：Attention Backend", section «extend 的两种
    形态»), a request without a cached prefix has an empty paged segment.

    Returns (o [T, Hq, D] float64, lse [T, Hq] float64).
    """
    qo_indptr = np.asarray(qo_indptr, dtype=np.int64)
    kv_indptr = np.asarray(kv_indptr, dtype=np.int64)
    kv_indices = np.asarray(kv_indices, dtype=np.int64)
    last_page_len = np.asarray(last_page_len, dtype=np.int64)
    T, Hq, D = q.shape
    Hkv = k_pool.shape[2]
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    group = Hq // Hkv
    scale = (1.0 / math.sqrt(D)) if (sm_scale is None or sm_scale <= 0) else float(sm_scale)
    if qo_indptr[0] != 0 or np.any(np.diff(qo_indptr) < 0):
        raise ValueError("qo_indptr must start at 0 and be non-decreasing")
    if not causal and window_left >= 0:
        raise ValueError("a window needs causal attention")
    wanted = None if rows is None else set(int(r) for r in rows)

    o = np.full((T, Hq, D), np.nan)
    lse = np.full((T, Hq), np.nan)
    for i in range(len(qo_indptr) - 1):
        q0, q1 = int(qo_indptr[i]), int(qo_indptr[i + 1])
        n = q1 - q0
        if n == 0:
            continue
        todo = [t for t in range(n) if wanted is None or (q0 + t) in wanted]
        if not todo:
            continue
        pages = kv_indices[kv_indptr[i] : kv_indptr[i + 1]]
        L = kv_len_of(len(pages), int(last_page_len[i]), page_size)
        if causal and L < n:
            raise ValueError(f"request {i}: kv_len {L} too short for {n} queries")
        if L == 0:  # non-causal segment with no keys: the empty state
            for t in todo:
                o[q0 + t], lse[q0 + t] = 0.0, -np.inf
            continue
        K = to_f64(gather_logical(k_pool, pages, L, page_size), kv_format, k_scale)  # [L, Hkv, D]
        V = to_f64(gather_logical(v_pool, pages, L, page_size), kv_format, v_scale)
        Q = to_f64(q[q0:q1], q_format)
        for t in todo:
            lo, hi = visible_range(query_position(L, n, t), window_left) if causal else full_range(L)
            for h in range(Hq):
                kvh = kv_head_of(h, group)
                o[q0 + t, h], lse[q0 + t, h] = attend(Q[t, h], K[:, kvh], V[:, kvh], lo, hi, scale)
    return o, lse


def kv_rows_of(kv_indptr, i: int):
    """Rows [begin, end) of the contiguous K/V tensors that request i owns."""
    return int(kv_indptr[i]), int(kv_indptr[i + 1])


def ragged_attention(q, k, v, qo_indptr, kv_indptr, sm_scale: float | None = None, causal: bool = True,
                     window_left: int = -1, q_format: str = "float", kv_format: str = "float"):
    """Batched attention over contiguous ("ragged") K/V, float64.

    "SGLang 源码完全拆解(八)：Attention Backend", section «extend 的两种形态»: the
    ragged form takes this step's K/V as plain tensors, not through the page
    table.  Request i owns K/V rows kv_indptr[i] .. kv_indptr[i+1]-1 of k / v
    ([rows, Hkv, D]) in logical order and query rows qo_indptr[i] ..
    qo_indptr[i+1]-1 of q ([T, Hq, D]).  The visibility rule is the paged one:
    with causal=True the queries are the last n positions of the request's
    kv_len keys (bottom-right aligned, optional window); with causal=False every
    query sees all kv_len keys (kv_len 0 gives the empty state).

    Returns (o [T, Hq, D] float64, lse [T, Hq] float64).
    """
    qo_indptr = np.asarray(qo_indptr, dtype=np.int64)
    kv_indptr = np.asarray(kv_indptr, dtype=np.int64)
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    if len(kv_indptr) != len(qo_indptr):
        raise ValueError("qo_indptr and kv_indptr must have the same length")
    if qo_indptr[0] != 0 or np.any(np.diff(qo_indptr) < 0) or kv_indptr[0] != 0 or np.any(np.diff(kv_indptr) < 0):
        raise ValueError("indptr arrays must start at 0 and be non-decreasing")
    if not causal and window_left >= 0:
        raise ValueError("a window needs causal attention")
    group = Hq // Hkv
    scale = (1.0 / math.sqrt(D)) if (sm_scale is None or sm_scale <= 0) else float(sm_scale)
    o = np.full((T, Hq, D), np.nan)
    lse = np.full((T, Hq), np.nan)
    for i in range(len(qo_indptr) - 1):
        q0, q1 = int(qo_indptr[i]), int(qo_indptr[i + 1])
        k0, k1 = kv_rows_of(kv_indptr, i)
        n, L = q1 - q0, k1 - k0
        if n == 0:
            continue
        if causal and L < n:
            raise ValueError(f"request {i}: kv_len {L} too short for {n} queries")
        if L == 0:
            o[q0:q1], lse[q0:q1] = 0.0, -np.inf
            continue
        K = to_f64(k[k0:k1], kv_format)
        V = to_f64(v[k0:k1], kv_format)
        Q = to_f64(q[q0:q1], q_format)
        for t in range(n):
            lo, hi = visible_range(query_position(L, n, t), window_left) if causal else full_range(L)
            for h in range(Hq):
                kvh = kv_head_of(h, group)
                o[q0 + t, h], lse[q0 + t, h] = attend(Q[t, h], K[:, kvh], V[:, kvh], lo, hi, scale)
    return o, lse


# ----------------------------------------------------------------------------------------------
# merging attention states
# ----------------------------------------------------------------------------------------------
def merge_states(o1, s1, o2, s2):
    """Merge two normalised attention outputs with their log-sum-exps.

    o = (o1 e^(s1-m) + o2 e^(s2-m)) / (e^(s1-m) + e^(s2-m)), m = max(s1, s2);
    the merged lse is m + ln(e^(s1-m) + e^(s2-m)).  An empty state has lse = -inf.
    """
    o1, o2 = np.asarray(o1, dtype=np.float64), np.asarray(o2, dtype=np.float64)
    s1, s2 = np.asarray(s1, dtype=np.float64), np.asarray(s2, dtype=np.float64)
    m = np.maximum(s1, s2)
    finite = np.isfinite(m)
    mm = np.where(finite, m, 0.0)
    w1 = np.where(finite, np.exp(s1 - mm), 0.0)
    w2 = np.where(finite, np.exp(s2 - mm), 0.0)
    den = w1 + w2
    safe = np.where(den > 0, den, 1.0)
    o = (o1 * w1[..., None] + o2 * w2[..., None]) / safe[..., None]
    return np.where((den > 0)[..., None], o, 0.0), np.where(den > 0, mm + np.log(safe), -np.inf)


def merge_many(os, lses):
    """Split-KV reduction of any number of states.

    m = max_s lse_s, w_s = e^(lse_s - m), o = sum_s w_s o_s / sum_s w_s,
    lse = m + ln(sum_s w_s).  Inputs are stacked along a new leading axis.
    """
    o = np.stack([np.asarray(x, dtype=np.float64) for x in os])
    s = np.stack([np.asarray(x, dtype=np.float64) for x in lses])
    m = s.max(axis=0)
    finite = np.isfinite(m)
    mm = np.where(finite, m, 0.0)
    w = np.where(finite[None], np.exp(s - mm[None]), 0.0)
    den = w.sum(axis=0)
    safe = np.where(den > 0, den, 1.0)
    out = (o * w[..., None]).sum(axis=0) / safe[..., None]
    return np.where((den > 0)[..., None], out, 0.0), np.where(den > 0, mm + np.log(safe), -np.inf)
